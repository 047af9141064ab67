"""B300 (sm_103a) MoE expert layer: Python binding of libmoe.so.

Thin ctypes marshalling over the C ABI declared in ``include/moe.h``: every function
here has the same name as the C entry point it calls, passes raw device pointers and the
current torch CUDA stream, and raises :class:`MoeError` on a non-zero status.  torch is
used only to allocate device memory and to name the stream; every step of the layer runs
in the library's CUDA kernels.  There is no fallback: importing this package builds ``libmoe.so``
if it is missing or stale and fails if it cannot be built or loaded.

The layer (sources: "Wide-EP ... NVIDIA" explainer, section "MoE basics"; "Efficient MoE
training for biological foundation models", sections "GroupedLinear Optimizes Expert
Computation" and "MXFP8 Precision Reduces Memory Footprint"): route each token to its
top-k experts, permute token rows into expert-contiguous order, grouped GEMM1 with the
scaled SwiGLU fused into its epilogue, grouped GEMM2, and combine back to token order.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_F32, MOE_BF16, MOE_MXFP8, MOE_FP8 = 0, 1, 2, 3
DTYPES = {"f32": MOE_F32, "bf16": MOE_BF16, "mxfp8": MOE_MXFP8, "fp8": MOE_FP8}
FP8_CODES = (MOE_MXFP8, MOE_FP8)  # E4M3 codes with scales in the SF tile layouts
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


from . import build as _build  # noqa: E402  (build.py does not import this package)

try:
    # compiles libmoe.so when it is missing or older than its sources (nvcc, sm_103a)
    LIB_PATH = _build.build()
except Exception as exc:  # no CUDA library, no layer: fail loudly
    raise ImportError(f"cannot build or find {LIB_PATH}: {exc}") from exc
_lib = ctypes.CDLL(LIB_PATH)

_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "moe_gu_block": (_I, [_I]),
    "moe_route_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_permute_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_mx_act_scale_bytes": (_SZ, [_I64, _I, _I]),
    "moe_expert_gemm1_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_pack_weights_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_pack_weights": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_mx_weight_scale_bytes": (_SZ, [_I, _I, _I]),
    "moe_grouped_mlp": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_rows_hint": (_I, [_I, _I, _I]),
    "moe_layer_gemm1_pairs": (_I, [_I, _I, _I, _I, _I, _I]),
    "moe_layer_fused_combine": (_I, [_I, _I, _I, _I]),
    "moe_layer_gemm_kernel": (_I, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "moe_grouped_mlp_workspace_size": (_SZ, [_I64, _I, _I, _I, _I]),
    "moe_expert_gemm1_swiglu": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_expert_gemm1_swiglu_gather": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _SZ,
                                            _P]),
    "moe_quantize_mx_rows": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "moe_eplb_plan": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_layer_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                _P, _SZ, _P]),
    "moe_layer_forward_train": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_layer_backward_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_pack_weights_backward": (_I, [_P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_pack_weights_backward_mx": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_pack_weights_backward_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_layer_backward_mx": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _SZ, _P]),
    "moe_layer_backward_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _SZ, _P]),
    "moe_layer_backward_mx_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_layer_backward_fp8_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_expert_gemm2": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_expert_gemm_workspace_size": (_SZ, []),
    "moe_unpermute_combine": (_I, [_P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_expert_gemm2_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I64, _I, _I, _I, _I, _P, _P, _P, _I, _P, _SZ,
                                      _P]),
    "moe_expert_gemm2_combine_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_layer_forward": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_layer_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_get_device_error": (_I, [_P, _P, _P]),
    "moe_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_selftest_wait_timeout": (_I, [ctypes.c_uint64, _P, _SZ, _P]),
    "moe_supported": (_I, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def lib():
    return _lib


def _check(fn: str, st: int):
    if st != 0:
        raise MoeError(fn, st)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def torch_dtype(dtype) -> torch.dtype:
    """Storage dtype of activations/outputs for a layer dtype."""
    return torch.float32 if _dt(dtype) == MOE_F32 else torch.bfloat16


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned device workspace (torch allocations are 256-byte aligned), its error
    word initialised by moe_workspace_init on the current stream."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _check("moe_workspace_init", _lib.moe_workspace_init(_ptr(ws), ws.numel(), _stream()))
    return ws


def n_cap(T: int, k: int, E_loc: int) -> int:
    return T * min(k, E_loc)


# ----------------------------------------------------------------------------- entry points
def moe_supported() -> bool:
    return bool(_lib.moe_supported())


def moe_route_topk(logits: torch.Tensor, k: int, topk_ids=None, topk_probs=None):
    T, E = logits.shape
    ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=logits.device)
    probs = topk_probs if topk_probs is not None else torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check("moe_route_topk", _lib.moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(probs), _stream()))
    return ids, probs


def alloc_permute(T: int, d: int, k: int, E_loc: int, x_dtype: torch.dtype, perm_dtype="bf16", device="cuda",
                  maps_only=False) -> dict:
    """Output buffers of moe_permute (maps_only: no permuted copy of x)."""
    cap = n_cap(T, k, E_loc)
    if maps_only:
        perm_x = perm_sf = None
    elif _dt(perm_dtype) in FP8_CODES:
        perm_x = torch.empty(cap, d, dtype=torch.uint8, device=device)
        perm_sf = torch.empty(max(1, _lib.moe_mx_act_scale_bytes(cap, d, E_loc)), dtype=torch.uint8, device=device)
    else:
        perm_x = torch.empty(cap, d, dtype=x_dtype, device=device)
        perm_sf = None
    return dict(perm_x=perm_x, perm_x_scale=perm_sf,
                counts=torch.empty(E_loc, dtype=torch.int32, device=device),
                offsets=torch.empty(E_loc + 1, dtype=torch.int32, device=device),
                row_src_token=torch.empty(cap, dtype=torch.int32, device=device),
                row_prob=torch.empty(cap, dtype=torch.float32, device=device),
                pair_to_row=torch.empty(T, k, dtype=torch.int32, device=device))


def moe_permute(x: torch.Tensor, topk_ids: torch.Tensor, topk_probs: torch.Tensor, e0: int, E_loc: int,
                perm_dtype="bf16", ws=None, out=None, maps_only=False) -> dict:
    T, d = x.shape
    k = topk_ids.shape[1]
    x_dt = MOE_F32 if x.dtype == torch.float32 else MOE_BF16
    out = out if out is not None else alloc_permute(T, d, k, E_loc, x.dtype, perm_dtype, x.device, maps_only)
    nb = _lib.moe_permute_workspace_size(T, k, E_loc)
    ws = ws if ws is not None else workspace(nb, x.device)
    _check("moe_permute", _lib.moe_permute(
        _ptr(x), x_dt, _dt(perm_dtype), T, d, _ptr(topk_ids), _ptr(topk_probs), k, e0, E_loc, _ptr(out["perm_x"]),
        _ptr(out["perm_x_scale"]), _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["row_src_token"]),
        _ptr(out["row_prob"]), _ptr(out["pair_to_row"]), _ptr(ws), ws.numel(), _stream()))
    return out


def moe_permute_noalloc(x: torch.Tensor, topk_ids: torch.Tensor, topk_probs: torch.Tensor, e0: int, E_loc: int,
                        perm_dtype="bf16", out=None) -> dict:
    """moe_permute with the library's static scratch (no workspace; the library allocates nothing)."""
    T, d = x.shape
    k = topk_ids.shape[1]
    x_dt = MOE_F32 if x.dtype == torch.float32 else MOE_BF16
    out = out if out is not None else alloc_permute(T, d, k, E_loc, x.dtype, perm_dtype, x.device)
    _check("moe_permute_noalloc", _lib.moe_permute_noalloc(
        _ptr(x), x_dt, _dt(perm_dtype), T, d, _ptr(topk_ids), _ptr(topk_probs), k, e0, E_loc, _ptr(out["perm_x"]),
        _ptr(out["perm_x_scale"]), _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["row_src_token"]),
        _ptr(out["row_prob"]), _ptr(out["pair_to_row"]), _stream()))
    return out


def moe_permute_workspace_size(T: int, k: int, E_loc: int) -> int:
    return int(_lib.moe_permute_workspace_size(T, k, E_loc))


@dataclasses.dataclass
class PackedWeights:
    dtype: int
    E_loc: int
    d: int
    f: int
    Wgu: torch.Tensor
    Wd: torch.Tensor
    Wgu_scale: torch.Tensor | None = None
    Wd_scale: torch.Tensor | None = None
    w_exp: torch.Tensor | None = None  # per-tensor FP8: exponents [3, E_loc] of W_gate, W_up, W_down


def moe_pack_weights(W_gate: torch.Tensor, W_up: torch.Tensor, W_down: torch.Tensor, dtype="bf16") -> PackedWeights:
    E_loc, d, f = W_gate.shape
    dev = W_gate.device
    src = MOE_F32 if W_gate.dtype == torch.float32 else MOE_BF16
    dst = _dt(dtype)
    if dst in FP8_CODES:
        Wgu = torch.empty(E_loc, 2 * f, d, dtype=torch.uint8, device=dev)
        Wd = torch.empty(E_loc, d, f, dtype=torch.uint8, device=dev)
        sg = torch.empty(_lib.moe_mx_weight_scale_bytes(E_loc, 2 * f, d), dtype=torch.uint8, device=dev)
        sd = torch.empty(_lib.moe_mx_weight_scale_bytes(E_loc, d, f), dtype=torch.uint8, device=dev)
    else:
        tdt = torch.float32 if dst == MOE_F32 else torch.bfloat16
        Wgu = torch.empty(E_loc, 2 * f, d, dtype=tdt, device=dev)
        Wd = torch.empty(E_loc, d, f, dtype=tdt, device=dev)
        sg = sd = None
    if dst == MOE_FP8:
        w_exp = torch.empty(3, E_loc, dtype=torch.int32, device=dev)
        _check("moe_pack_weights_fp8", _lib.moe_pack_weights_fp8(
            _ptr(W_gate), _ptr(W_up), _ptr(W_down), src, E_loc, d, f, _ptr(Wgu), _ptr(Wd), _ptr(sg), _ptr(sd),
            _ptr(w_exp), _stream()))
        return PackedWeights(dst, E_loc, d, f, Wgu, Wd, sg, sd, w_exp)
    _check("moe_pack_weights", _lib.moe_pack_weights(
        _ptr(W_gate), _ptr(W_up), _ptr(W_down), src, dst, E_loc, d, f, _ptr(Wgu), _ptr(Wd), _ptr(sg), _ptr(sd),
        _stream()))
    return PackedWeights(dst, E_loc, d, f, Wgu, Wd, sg, sd)


def moe_rows_hint(T: int, k: int, E: int) -> int:
    return int(_lib.moe_rows_hint(T, k, E))


def moe_layer_gemm1_pairs(T: int, d: int, k: int, E: int, E_loc: int, dtype: str) -> bool:
    """True if moe_layer_forward runs GEMM1 on CTA pairs (A from a permuted copy of x)."""
    r = int(_lib.moe_layer_gemm1_pairs(T, d, k, E, E_loc, _dt(dtype)))
    if r < 0:
        raise ValueError("invalid sizes")
    return bool(r)


# rows_hint values that force a grouped-GEMM kernel (moe.h MOE_KERNEL_*)
KERNEL_CTA, KERNEL_PAIR, KERNEL_SWAP = -1, -2, -3
_KERNEL_NAMES = {KERNEL_CTA: "cta", KERNEL_PAIR: "pair", KERNEL_SWAP: "swap"}


def moe_layer_gemm_kernel(T: int, d: int, f: int, k: int, E: int, E_loc: int, dtype: str, gemm: int) -> str:
    """The kernel moe_layer_forward runs for GEMM 1 or 2: "cta", "pair" or "swap"."""
    r = int(_lib.moe_layer_gemm_kernel(T, d, f, k, E, E_loc, _dt(dtype), gemm))
    if r not in _KERNEL_NAMES:
        raise ValueError("invalid sizes")
    return _KERNEL_NAMES[r]


def moe_layer_fused_combine(k: int, E: int, E_loc: int, dtype: str) -> bool:
    """True if moe_layer_forward folds the combine into GEMM2 for this routing shape."""
    r = int(_lib.moe_layer_fused_combine(k, E, E_loc, _dt(dtype)))
    if r < 0:
        raise ValueError("invalid sizes")
    return bool(r)


def moe_grouped_mlp(perm_x, perm_x_scale, offsets, row_prob, pw: PackedWeights, Y2=None, ws=None, rows_hint=0):
    cap = perm_x.shape[0]
    dev = perm_x.device
    Y2 = Y2 if Y2 is not None else torch.empty(cap, pw.d, dtype=torch_dtype(pw.dtype), device=dev)
    nb = _lib.moe_grouped_mlp_workspace_size(cap, pw.E_loc, pw.d, pw.f, pw.dtype)
    ws = ws if ws is not None else workspace(nb, dev)
    _check("moe_grouped_mlp", _lib.moe_grouped_mlp(
        _ptr(perm_x), _ptr(perm_x_scale), _ptr(offsets), _ptr(row_prob), cap, pw.E_loc, pw.d, pw.f, pw.dtype,
        _ptr(pw.Wgu), _ptr(pw.Wgu_scale), _ptr(pw.Wd), _ptr(pw.Wd_scale), _ptr(Y2), int(rows_hint), _ptr(ws), ws.numel(),
        _stream()))
    return Y2, ws


def alloc_h(N_cap: int, pw: PackedWeights, device="cuda"):
    """h buffer (+ its MXFP8 scales) for moe_expert_gemm1_swiglu."""
    if pw.dtype in FP8_CODES:
        return (torch.empty(N_cap, pw.f, dtype=torch.uint8, device=device),
                torch.empty(max(1, _lib.moe_mx_act_scale_bytes(N_cap, pw.f, pw.E_loc)), dtype=torch.uint8,
                            device=device))
    return torch.empty(N_cap, pw.f, dtype=torch_dtype(pw.dtype), device=device), None


def moe_expert_gemm1_swiglu(perm_x, perm_x_scale, offsets, row_prob, pw: PackedWeights, h=None, h_scale=None,
                            ws=None, rows_hint=0):
    cap = perm_x.shape[0]
    if h is None:
        h, h_scale = alloc_h(cap, pw, perm_x.device)
    ws = ws if ws is not None else workspace(_lib.moe_expert_gemm1_workspace_size(cap, pw.f, pw.dtype), perm_x.device)
    _check("moe_expert_gemm1_swiglu", _lib.moe_expert_gemm1_swiglu(
        _ptr(perm_x), _ptr(perm_x_scale), _ptr(offsets), _ptr(row_prob), cap, pw.E_loc, pw.d, pw.f, pw.dtype,
        _ptr(pw.Wgu), _ptr(pw.Wgu_scale), _ptr(h), _ptr(h_scale), int(rows_hint), _ptr(ws), ws.numel(), _stream()))
    return h, h_scale, ws


def moe_expert_gemm1_swiglu_gather(x, x_scale, row_src_token, offsets, row_prob, pw: PackedWeights, h=None,
                                   h_scale=None, ws=None, rows_hint=KERNEL_CTA):
    """GEMM1 + scaled SwiGLU reading the token rows x (bf16, or E4M3 + row scales from
    moe_quantize_mx_rows) through row_src_token.  rows_hint picks the kernel shape as for
    moe_expert_gemm1_swiglu (the default keeps the 1-CTA kernel)."""
    cap = row_src_token.shape[0]
    if h is None:
        h, h_scale = alloc_h(cap, pw, x.device)
    ws = ws if ws is not None else workspace(_lib.moe_expert_gemm_workspace_size(), x.device)
    _check("moe_expert_gemm1_swiglu_gather", _lib.moe_expert_gemm1_swiglu_gather(
        _ptr(x), _ptr(x_scale), _ptr(row_src_token), _ptr(offsets), _ptr(row_prob), cap, pw.E_loc, pw.d, pw.f,
        pw.dtype, _ptr(pw.Wgu), _ptr(pw.Wgu_scale), _ptr(h), _ptr(h_scale), int(rows_hint), _ptr(ws), ws.numel(),
        _stream()))
    return h, h_scale, ws


def moe_quantize_mx_rows(x: torch.Tensor, xq=None, x_scale=None, pair_to_row=None):
    """E4M3 codes [T, d] and row-major E8M0 scales [T, d / 32] of the rows of x (with
    pair_to_row: only the rows of tokens that have a local expert)."""
    T, d = x.shape
    x_dt = MOE_F32 if x.dtype == torch.float32 else MOE_BF16
    xq = xq if xq is not None else torch.empty(T, d, dtype=torch.uint8, device=x.device)
    x_scale = x_scale if x_scale is not None else torch.empty(T, d // 32, dtype=torch.uint8, device=x.device)
    k = pair_to_row.shape[1] if pair_to_row is not None else 0
    _check("moe_quantize_mx_rows", _lib.moe_quantize_mx_rows(_ptr(x), x_dt, T, d, _ptr(pair_to_row), k, _ptr(xq),
                                                             _ptr(x_scale), _stream()))
    return xq, x_scale


def moe_expert_gemm2(h, h_scale, offsets, pw: PackedWeights, Y2=None, ws=None, rows_hint=0):
    cap = h.shape[0]
    Y2 = Y2 if Y2 is not None else torch.empty(cap, pw.d, dtype=torch_dtype(pw.dtype), device=h.device)
    ws = ws if ws is not None else workspace(_lib.moe_expert_gemm_workspace_size(), h.device)
    _check("moe_expert_gemm2", _lib.moe_expert_gemm2(
        _ptr(h), _ptr(h_scale), _ptr(offsets), cap, pw.E_loc, pw.d, pw.f, pw.dtype, _ptr(pw.Wd), _ptr(pw.Wd_scale),
        _ptr(Y2), int(rows_hint), _ptr(ws), ws.numel(), _stream()))
    return Y2, ws


def moe_unpermute_combine(Y2, pair_to_row, dtype, y=None):
    T, k = pair_to_row.shape
    d = Y2.shape[1]
    y = y if y is not None else torch.empty(T, d, dtype=torch_dtype(dtype), device=Y2.device)
    _check("moe_unpermute_combine", _lib.moe_unpermute_combine(_ptr(Y2), _ptr(pair_to_row), T, k, d, _dt(dtype),
                                                               _ptr(y), _stream()))
    return y


def moe_expert_gemm2_combine(h, h_scale, offsets, row_src_token, pair_to_row, pw: PackedWeights, y=None, ws=None,
                             rows_hint=0):
    """GEMM2 with the unpermute + combine in its epilogue: y [T, d] bf16 straight from h."""
    cap = h.shape[0]
    T, k = pair_to_row.shape
    y = y if y is not None else torch.empty(T, pw.d, dtype=torch.bfloat16, device=h.device)
    ws = ws if ws is not None else workspace(_lib.moe_expert_gemm2_combine_workspace_size(cap, T, pw.d), h.device)
    _check("moe_expert_gemm2_combine", _lib.moe_expert_gemm2_combine(
        _ptr(h), _ptr(h_scale), _ptr(offsets), _ptr(row_src_token), _ptr(pair_to_row), T, k, cap, pw.E_loc, pw.d,
        pw.f, pw.dtype, _ptr(pw.Wd), _ptr(pw.Wd_scale), _ptr(y), int(rows_hint), _ptr(ws), ws.numel(), _stream()))
    return y, ws


def moe_layer_workspace_size(T, d, f, E, k, E_loc, dtype) -> int:
    return int(_lib.moe_layer_workspace_size(T, d, f, E, k, E_loc, _dt(dtype)))


def moe_layer_forward(x, logits, E: int, k: int, e0: int, pw: PackedWeights, y=None, ws=None):
    T, d = x.shape
    y = y if y is not None else torch.empty(T, d, dtype=torch_dtype(pw.dtype), device=x.device)
    nb = moe_layer_workspace_size(T, d, pw.f, E, k, pw.E_loc, pw.dtype)
    ws = ws if ws is not None else workspace(nb, x.device)
    _check("moe_layer_forward", _lib.moe_layer_forward(
        _ptr(x), _ptr(logits), T, d, pw.f, E, k, e0, pw.E_loc, pw.dtype, _ptr(pw.Wgu), _ptr(pw.Wgu_scale),
        _ptr(pw.Wd), _ptr(pw.Wd_scale), _ptr(y), _ptr(ws), ws.numel(), _stream()))
    return y, ws


def moe_pack_weights_backward(W_gate: torch.Tensor, W_up: torch.Tensor) -> torch.Tensor:
    """WguT [E_loc, d, 2f] bf16 for moe_layer_backward."""
    E_loc, d, f = W_gate.shape
    src = MOE_F32 if W_gate.dtype == torch.float32 else MOE_BF16
    out = torch.empty(E_loc, d, 2 * f, dtype=torch.bfloat16, device=W_gate.device)
    _check("moe_pack_weights_backward", _lib.moe_pack_weights_backward(_ptr(W_gate), _ptr(W_up), src, E_loc, d, f,
                                                                       _ptr(out), _stream()))
    return out


def moe_layer_forward_train(x, logits, E: int, k: int, e0: int, pw: PackedWeights, y=None, ws=None):
    """bf16 forward that also returns the routing and the gate/up pre-activations for the
    backward: (y, topk_ids, topk_probs, gu_saved, ws)."""
    T, d = x.shape
    dev = x.device
    y = y if y is not None else torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    probs = torch.empty(T, k, dtype=torch.float32, device=dev)
    gu = torch.empty(n_cap(T, k, pw.E_loc), 2 * pw.f, dtype=torch.bfloat16, device=dev)
    nb = moe_layer_workspace_size(T, d, pw.f, E, k, pw.E_loc, "bf16")
    ws = ws if ws is not None else workspace(nb, dev)
    _check("moe_layer_forward_train", _lib.moe_layer_forward_train(
        _ptr(x), _ptr(logits), T, d, pw.f, E, k, e0, pw.E_loc, _ptr(pw.Wgu), _ptr(pw.Wd), _ptr(y), _ptr(ids),
        _ptr(probs), _ptr(gu), _ptr(ws), ws.numel(), _stream()))
    return y, ids, probs, gu, ws


def moe_layer_backward(x, dy, topk_ids, topk_probs, E: int, e0: int, pw: PackedWeights, W_down: torch.Tensor,
                       WguT: torch.Tensor, ws=None, out=None, gu_saved=None):
    """Gradients of sum(dy * y) of the bf16 layer: dict(dx, dlogits, dW_gate, dW_up, dW_down).
    gu_saved: the pre-activations from moe_layer_forward_train (else recomputed)."""
    T, d = x.shape
    k = topk_ids.shape[1]
    f, E_loc = pw.f, pw.E_loc
    dev = x.device
    if out is None:
        out = dict(dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
                   dlogits=torch.empty(T, E, dtype=torch.float32, device=dev),
                   dW_gate=torch.empty(E_loc, d, f, dtype=torch.float32, device=dev),
                   dW_up=torch.empty(E_loc, d, f, dtype=torch.float32, device=dev),
                   dW_down=torch.empty(E_loc, f, d, dtype=torch.float32, device=dev))
    nb = _lib.moe_layer_backward_workspace_size(T, d, f, k, E_loc)
    ws = ws if ws is not None else workspace(nb, dev)
    _check("moe_layer_backward", _lib.moe_layer_backward(
        _ptr(x), _ptr(dy), _ptr(topk_ids), _ptr(topk_probs), T, d, f, E, k, e0, E_loc, _ptr(pw.Wgu), _ptr(W_down),
        _ptr(WguT), _ptr(gu_saved), _ptr(out["dx"]), _ptr(out["dlogits"]), _ptr(out["dW_gate"]), _ptr(out["dW_up"]),
        _ptr(out["dW_down"]), _ptr(ws), ws.numel(), _stream()))
    return out, ws


@dataclasses.dataclass
class BackwardWeightsMx:
    """MXFP8 operands of the backward's row-wise GEMMs (moe_pack_weights_backward_mx)."""
    Wd_q: torch.Tensor
    Wd_scale: torch.Tensor
    WguT_q: torch.Tensor
    WguT_scale: torch.Tensor


def moe_pack_weights_backward_mx(W_gate: torch.Tensor, W_up: torch.Tensor, W_down: torch.Tensor,
                                 w_exp: torch.Tensor | None = None) -> BackwardWeightsMx:
    """Backward weight layouts; with w_exp (PackedWeights.w_exp of a per-tensor FP8 pack)
    the per-tensor FP8 ones (moe_pack_weights_backward_fp8)."""
    E_loc, d, f = W_gate.shape
    dev = W_gate.device
    src = MOE_F32 if W_gate.dtype == torch.float32 else MOE_BF16
    bw = BackwardWeightsMx(
        Wd_q=torch.empty(E_loc, f, d, dtype=torch.uint8, device=dev),
        Wd_scale=torch.empty(_lib.moe_mx_weight_scale_bytes(E_loc, f, d), dtype=torch.uint8, device=dev),
        WguT_q=torch.empty(E_loc, d, 2 * f, dtype=torch.uint8, device=dev),
        WguT_scale=torch.empty(_lib.moe_mx_weight_scale_bytes(E_loc, d, 2 * f), dtype=torch.uint8, device=dev))
    if w_exp is not None:
        _check("moe_pack_weights_backward_fp8", _lib.moe_pack_weights_backward_fp8(
            _ptr(W_gate), _ptr(W_up), _ptr(W_down), src, E_loc, d, f, _ptr(w_exp), _ptr(bw.WguT_q),
            _ptr(bw.WguT_scale), _ptr(bw.Wd_q), _ptr(bw.Wd_scale), _stream()))
        return bw
    _check("moe_pack_weights_backward_mx", _lib.moe_pack_weights_backward_mx(
        _ptr(W_gate), _ptr(W_up), _ptr(W_down), src, E_loc, d, f, _ptr(bw.WguT_q), _ptr(bw.WguT_scale), _ptr(bw.Wd_q),
        _ptr(bw.Wd_scale), _stream()))
    return bw


def moe_layer_backward_mx(x, dy, topk_ids, topk_probs, E: int, e0: int, pw: PackedWeights, bw: BackwardWeightsMx,
                          ws=None, out=None):
    """Gradients of sum(dy * y) of the MXFP8 layer, or of the per-tensor FP8 layer when pw
    is a per-tensor FP8 pack: dict(dx, dlogits, dW_gate, dW_up, dW_down)."""
    T, d = x.shape
    k = topk_ids.shape[1]
    f, E_loc = pw.f, pw.E_loc
    dev = x.device
    if out is None:
        out = dict(dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
                   dlogits=torch.empty(T, E, dtype=torch.float32, device=dev),
                   dW_gate=torch.empty(E_loc, d, f, dtype=torch.float32, device=dev),
                   dW_up=torch.empty(E_loc, d, f, dtype=torch.float32, device=dev),
                   dW_down=torch.empty(E_loc, f, d, dtype=torch.float32, device=dev))
    nb = _lib.moe_layer_backward_mx_workspace_size(T, d, f, k, E_loc)
    ws = ws if ws is not None else workspace(nb, dev)
    fn = "moe_layer_backward_fp8" if pw.dtype == MOE_FP8 else "moe_layer_backward_mx"
    _check(fn, getattr(_lib, fn)(
        _ptr(x), _ptr(dy), _ptr(topk_ids), _ptr(topk_probs), T, d, f, E, k, e0, E_loc, _ptr(pw.Wgu), _ptr(pw.Wgu_scale),
        _ptr(bw.Wd_q), _ptr(bw.Wd_scale), _ptr(bw.WguT_q), _ptr(bw.WguT_scale), _ptr(out["dx"]), _ptr(out["dlogits"]),
        _ptr(out["dW_gate"]), _ptr(out["dW_up"]), _ptr(out["dW_down"]), _ptr(ws), ws.numel(), _stream()))
    return out, ws


def moe_eplb_plan(load, G: int, S: int):
    """Placement of E experts (load[e] tokens each) on G GPUs with S slots each, with
    copies of the most loaded experts: (slot_expert [G, S], replicas [E], gpu_load [G])."""
    ld = np.ascontiguousarray(np.asarray(load, dtype=np.int64))
    E = ld.size
    slot = np.empty((G, S), np.int32)
    rep = np.empty(E, np.int32)
    gl = np.empty(G, np.float64)
    _check("moe_eplb_plan", _lib.moe_eplb_plan(ld.ctypes.data_as(ctypes.c_void_p), E, G, S,
                                               slot.ctypes.data_as(ctypes.c_void_p),
                                               rep.ctypes.data_as(ctypes.c_void_p),
                                               gl.ctypes.data_as(ctypes.c_void_p)))
    return slot, rep, gl


def moe_get_device_error(ws: torch.Tensor) -> int:
    code = ctypes.c_int32(0)
    _check("moe_get_device_error", _lib.moe_get_device_error(_ptr(ws), _stream(), ctypes.byref(code)))
    return code.value


def moe_selftest_wait_timeout(timeout_ns: int, ws=None):
    """Run the bounded-wait self-test; returns the device error code it recorded."""
    ws = ws if ws is not None else workspace(256)
    _check("moe_selftest_wait_timeout", _lib.moe_selftest_wait_timeout(int(timeout_ns), _ptr(ws), ws.numel(),
                                                                       _stream()))
    return moe_get_device_error(ws)


class MoELayer:
    """The expert layer on one GPU's experts [e0, e0 + E_loc): packed weights + workspace."""

    def __init__(self, W_gate, W_up, W_down, E: int, k: int, e0: int = 0, dtype="bf16"):
        self.E, self.k, self.e0 = E, k, e0
        self.weights = moe_pack_weights(W_gate, W_up, W_down, dtype)
        self._ws = None

    def __call__(self, x, logits, y=None):
        T, d = x.shape
        nb = moe_layer_workspace_size(T, d, self.weights.f, self.E, self.k, self.weights.E_loc, self.weights.dtype)
        if self._ws is None or self._ws.numel() < nb:
            self._ws = workspace(nb, x.device)
        y, _ = moe_layer_forward(x, logits, self.E, self.k, self.e0, self.weights, y=y, ws=self._ws)
        return y

    def device_error(self) -> int:
        return 0 if self._ws is None else moe_get_device_error(self._ws)
