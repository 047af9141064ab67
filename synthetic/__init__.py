"""Seeded synthetic inputs for the MoE expert layer.

This module is the ONE piece of code shared by the CPU oracle's tests and the CUDA
path's tests/benchmark.  It only draws random numbers and rounds them to the storage
dtype; it holds none of the layer's arithmetic (no routing, no permutation, no GEMM,
no activation, no quantisation).

Recipe (every tensor has its own counter-keyed stream so that any subset of experts can
be regenerated without drawing the others):

* ``np.random.default_rng([seed, TAG, global_expert_id])`` per weight tensor and expert,
  ``np.random.default_rng([seed, TAG])`` for x, logits and bias.
* x ~ N(0, 1), shape [T, d].
* W_gate, W_up ~ N(0, 1/d) with shape [E_loc, d, f]; W_down ~ N(0, 1/f) with shape
  [E_loc, f, d] (N(mu, sigma^2) notation, fan_in = the contracted size).
* router logits ~ N(0, 1), shape [T, E], fp32, plus an optional per-expert bias that is
  folded into the logits: ``normal`` -> bias_e ~ N(0, var) ; ``zipf`` -> popularity
  p_r ~ r^-s over ranks r = 1..E, ranks assigned to expert ids by a seeded permutation,
  bias_e = ln p_rank(e).
* Everything is drawn in fp32; bf16 workloads round x and the weights to bf16 with
  round-to-nearest-even, and those rounded values are the exact inputs of both sides.
  bf16 arrays are carried as uint16 bit patterns (numpy has no bf16 type).

The workload table mirrors the layer shapes of the source pages: DeepSeek-R1-style 256
experts with top-8 routing, and the local expert slices one GPU holds under EP8 (32
experts) and EP64 (4 experts) (NVIDIA NVL72 Wide-EP explainer, "Wide-EP" section).
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

TAG_X = 1
TAG_LOGITS = 2
TAG_BIAS = 3
TAG_ZIPF_PERM = 4
TAG_DY = 5
TAG_W_GATE = 10
TAG_W_UP = 11
TAG_W_DOWN = 12


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    e0: int
    E_loc: int
    dtype: str  # "f32" | "bf16" | "mxfp8" | "fp8"  (mxfp8 / fp8: inputs drawn as bf16, quantised by the layer)
    bias: tuple = ()  # () | ("normal", var) | ("zipf", s)
    seed: int = 0

    @property
    def act_dtype(self) -> str:
        """Storage dtype of x and of the unquantised weights."""
        return "f32" if self.dtype == "f32" else "bf16"

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Tiny fp32 layer: T=64, d=128, f=256, E=8, top-2, all experts local.
    "tiny_fp32": Workload("tiny_fp32", 64, 128, 256, 8, 2, 0, 8, "f32"),
    # BF16 layer, all 64 experts local, mild skew from a N(0, 0.5) per-expert bias.
    "bf16_e64": Workload("bf16_e64", 4096, 2048, 1024, 64, 8, 0, 64, "bf16", ("normal", 0.5)),
    # EP8-shaped slice of a 256-expert top-8 layer, decode-like batch, Zipf(1.1) hot experts.
    "ep8_zipf_T512": Workload("ep8_zipf_T512", 512, 7168, 2048, 256, 8, 0, 32, "bf16", ("zipf", 1.1)),
    # EP64-shaped slice (4 local experts), uniform logits, T sweep.
    "ep64_T2048": Workload("ep64_T2048", 2048, 7168, 2048, 256, 8, 0, 4, "bf16"),
    "ep64_T8192": Workload("ep64_T8192", 8192, 7168, 2048, 256, 8, 0, 4, "bf16"),
    "ep64_T32768": Workload("ep64_T32768", 32768, 7168, 2048, 256, 8, 0, 4, "bf16"),
    # MXFP8 variant of the EP8 Zipf slice at T=8192.
    "mxfp8_ep8_zipf_T8192": Workload("mxfp8_ep8_zipf_T8192", 8192, 7168, 2048, 256, 8, 0, 32, "mxfp8", ("zipf", 1.1)),
    # MXFP8 variant of the EP64 slice at T=8192.
    "mxfp8_ep64_T8192": Workload("mxfp8_ep64_T8192", 8192, 7168, 2048, 256, 8, 0, 4, "mxfp8"),
    # the same slice with per-tensor FP8 (one power-of-two scale per tensor)
    "fp8_ep64_T8192": Workload("fp8_ep64_T8192", 8192, 7168, 2048, 256, 8, 0, 4, "fp8"),
    # One expert holding every token (E = 1, top-1) at the slices' d and f: the grouped GEMMs
    # without ragged segments, i.e. the dense tensor-core rate of the same kernels.
    "dense_bf16_T16384": Workload("dense_bf16_T16384", 16384, 7168, 2048, 1, 1, 0, 1, "bf16"),
    "dense_mxfp8_T16384": Workload("dense_mxfp8_T16384", 16384, 7168, 2048, 1, 1, 0, 1, "mxfp8"),
}


# ----------------------------------------------------------------------------- storage
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (inputs carry no NaN)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_storage(a32: np.ndarray, act_dtype: str) -> np.ndarray:
    return a32.astype(np.float32) if act_dtype == "f32" else bf16_bits(a32)


def to_f64(a: np.ndarray, act_dtype: str) -> np.ndarray:
    """Exact widening of a storage array to fp64."""
    return (a if act_dtype == "f32" else bf16_to_f32(a)).astype(np.float64)


# ----------------------------------------------------------------------------- draws
def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([seed, *key])


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def gen_x(w: Workload, T: int | None = None) -> np.ndarray:
    """x [T, d] in storage dtype (fp32 or bf16 bits)."""
    T = w.T if T is None else T
    return as_storage(_normal(_rng(w.seed, TAG_X), (T, w.d), 1.0), w.act_dtype)


def gen_dy(w: Workload, T: int | None = None) -> np.ndarray:
    """Output gradient dy [T, d] for the backward, N(0, 1), in storage dtype."""
    T = w.T if T is None else T
    return as_storage(_normal(_rng(w.seed, TAG_DY), (T, w.d), 1.0), w.act_dtype)


def gen_bias(w: Workload) -> np.ndarray:
    """Per-expert router bias [E] fp32 (zeros when the workload has none)."""
    if not w.bias:
        return np.zeros(w.E, np.float32)
    kind, par = w.bias
    if kind == "normal":
        return _normal(_rng(w.seed, TAG_BIAS), (w.E,), float(np.sqrt(par)))
    if kind == "zipf":
        rank = _rng(w.seed, TAG_ZIPF_PERM).permutation(w.E) + 1  # rank of expert e
        pop = rank.astype(np.float64) ** (-float(par))
        pop /= pop.sum()
        return np.log(pop).astype(np.float32)
    raise ValueError(kind)


def gen_logits(w: Workload, T: int | None = None) -> np.ndarray:
    """Router logits [T, E] fp32 = N(0,1) draws + per-expert bias (folded in)."""
    T = w.T if T is None else T
    lg = _normal(_rng(w.seed, TAG_LOGITS), (T, w.E), 1.0)
    lg += gen_bias(w)[None, :]
    return lg


def gen_expert_weights(w: Workload, e_global: int):
    """(W_gate [d,f], W_up [d,f], W_down [f,d]) of one expert, storage dtype."""
    wg = _normal(_rng(w.seed, TAG_W_GATE, e_global), (w.d, w.f), w.d ** -0.5)
    wu = _normal(_rng(w.seed, TAG_W_UP, e_global), (w.d, w.f), w.d ** -0.5)
    wd = _normal(_rng(w.seed, TAG_W_DOWN, e_global), (w.f, w.d), w.f ** -0.5)
    return tuple(as_storage(a, w.act_dtype) for a in (wg, wu, wd))


def gen_weights(w: Workload, experts=None, threads: int = 8):
    """Stacked user-layout weights of the local experts (or of the listed global ids).

    Returns W_gate [n, d, f], W_up [n, d, f], W_down [n, f, d] in storage dtype.
    """
    ids = list(range(w.e0, w.e0 + w.E_loc)) if experts is None else list(experts)
    dt = np.float32 if w.act_dtype == "f32" else np.uint16
    n = len(ids)
    wg = np.empty((n, w.d, w.f), dt)
    wu = np.empty((n, w.d, w.f), dt)
    wd = np.empty((n, w.f, w.d), dt)

    def one(i):
        wg[i], wu[i], wd[i] = gen_expert_weights(w, ids[i])

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(one, range(n)))
    return wg, wu, wd


def sample_tokens(w: Workload, n: int, salt: int = 99) -> np.ndarray:
    """A seeded, sorted sample of n distinct token indices (for sampled parity checks)."""
    n = min(n, w.T)
    return np.sort(_rng(w.seed, salt).choice(w.T, size=n, replace=False)).astype(np.int64)
