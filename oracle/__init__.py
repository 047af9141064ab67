"""CPU oracle for the MoE expert layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The CUDA library never imports, links or calls it, and it never
imports the CUDA library.

* ``moe_oracle.cpp`` (built into ``liboracle.so``): the fp64 reference of the layer
  (routing, permutation, scaled-SwiGLU expert FFN, combine, MXFP8 codec).
* ``brute.py``: a second, independent numpy brute force (all experts evaluated densely,
  top-k by a full stable sort, quantiser by nearest-code search) used to pin the C++
  oracle on tiny inputs, and the MXFP8 backward token by token.
* ``moe_backward_mx`` (numpy over the C++ codec): the MXFP8 layer backward, every backward
  GEMM operand quantised along that GEMM's contraction axis.
* ``moe_forward_fp8``, ``moe_backward_fp8`` (numpy over the C++ codec): the per-tensor FP8
  layer and its backward (one power-of-two scale per tensor).

Functions of this module are thin ctypes marshalling around the C++ oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

DT = {"f32": 0, "bf16": 1, "e4m3": 2, "f64": 3}


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.oracle_version.restype = i32
        lib.oracle_e4m3_decode.argtypes = [P, i64, P]
        lib.oracle_e4m3_encode.argtypes = [P, i64, P]
        lib.oracle_mx_quantize.argtypes = [P, i32, i64, i64, i64, P, P, i32]
        lib.oracle_mx_quantize.restype = i32
        lib.oracle_route_topk.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_route_topk.restype = i32
        lib.oracle_permute.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P]
        lib.oracle_permute.restype = i32
        lib.oracle_moe_forward.argtypes = [P, i32, P, i64, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                           P, P, P, i32, P, i64, P, i32]
        lib.oracle_moe_forward.restype = i32
        lib.oracle_down_proj_mx.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, P, P, i32]
        lib.oracle_down_proj_mx.restype = i32
        lib.oracle_moe_backward.argtypes = [P, i32, P, i64, i32, i32, i32, i32, i32, i32, i32, P, P, P, P, i32,
                                            P, i64, P, P, P, i32, P, P, P, i32]
        lib.oracle_moe_backward.restype = i32
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    return len(os.sched_getaffinity(0))


# ----------------------------------------------------------------------------- codec
def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode(_p(c), c.size, _p(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().oracle_e4m3_encode(_p(a), a.size, _p(out))
    return out


def mx_quantize(a, dtype: str, shape3) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8-quantise ``a`` viewed as [n_outer, K, n_inner] in 32-blocks along K.

    Returns (codes with a's shape, scales [n_outer, K/32, n_inner]) as uint8.
    """
    n_outer, K, n_inner = shape3
    src = _c(a, {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype])
    assert src.size == n_outer * K * n_inner
    codes = np.empty(src.shape, np.uint8)
    scales = np.empty((n_outer, K // 32, n_inner), np.uint8)
    st = _load().oracle_mx_quantize(_p(src), DT[dtype], n_outer, K, n_inner, _p(codes), _p(scales), threads())
    if st != 0:
        raise ValueError("oracle_mx_quantize: K must be a multiple of 32")
    return codes, scales


# ----------------------------------------------------------------------------- layer
def route_topk(logits, k: int):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    probs = np.empty((T, k), np.float64)
    st = _load().oracle_route_topk(_p(lg), T, E, k, _p(ids), _p(probs))
    if st != 0:
        raise ValueError(f"oracle_route_topk status {st}")
    return ids, probs


def permute(ids, e0: int, E_loc: int) -> dict:
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E_loc, np.int32)
    offsets = np.empty(E_loc + 1, np.int32)
    cap = T * k
    row_src = np.full(cap, -1, np.int32)
    row_slot = np.full(cap, -1, np.int32)
    p2r = np.empty((T, k), np.int32)
    _load().oracle_permute(_p(ids), T, k, e0, E_loc, _p(counts), _p(offsets), _p(row_src), _p(row_slot), _p(p2r))
    N = int(offsets[-1])
    return dict(counts=counts, offsets=offsets, row_src_token=row_src[:N], row_slot=row_slot[:N], pair_to_row=p2r, N=N)


def moe_forward(x, x_dtype: str, logits, d: int, f: int, E: int, k: int, e0: int, E_loc: int,
                W_gate, W_up, W_down, w_dtype: str, w_scales=(None, None, None), mx_act: bool = False,
                tokens=None, nthreads: int | None = None) -> np.ndarray:
    """fp64 layer output for ``tokens`` (default: all) -> [n_tokens, d].

    x: [T, d] f32 or bf16 bits; logits [T, E] fp32; weights in user layout
    (W_gate/W_up [E_loc, d, f], W_down [E_loc, f, d]) as f32, bf16 bits, or E4M3 codes
    with E8M0 scales ``w_scales`` ([E_loc, d/32, f], [E_loc, d/32, f], [E_loc, f/32, d]).
    """
    npdt = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8, "f64": np.float64}
    x = _c(x, npdt[x_dtype])
    lg = _c(logits, np.float32)
    T = x.shape[0]
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    wg, wu, wd = (_c(w, npdt[w_dtype]) for w in (W_gate, W_up, W_down))
    sg, su, sd = ((None if s is None else _c(s, np.uint8)) for s in w_scales)
    y = np.empty((tok.size, d), np.float64)
    st = _load().oracle_moe_forward(_p(x), DT[x_dtype], _p(lg), T, d, f, E, k, e0, E_loc, DT[w_dtype],
                                    _p(wg), _p(wu), _p(wd), _p(sg), _p(su), _p(sd), int(mx_act),
                                    _p(tok), tok.size, _p(y), nthreads or threads())
    if st != 0:
        raise ValueError(f"oracle_moe_forward status {st}")
    return y


def down_proj_mx(h_codes, h_scales, row_expert, d: int, f: int, E_loc: int, W_down, w_dtype: str,
                 Wd_scale=None) -> np.ndarray:
    """fp64 h W_down for given MXFP8 h rows (diagnostic)."""
    npdt = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
    hc = _c(h_codes, np.uint8)
    hs = _c(h_scales, np.uint8)
    re = _c(row_expert, np.int32)
    wd = _c(W_down, npdt[w_dtype])
    sd = None if Wd_scale is None else _c(Wd_scale, np.uint8)
    out = np.empty((re.size, d), np.float64)
    st = _load().oracle_down_proj_mx(_p(hc), _p(hs), _p(re), re.size, d, f, E_loc, DT[w_dtype], _p(wd), _p(sd),
                                     _p(out), threads())
    if st != 0:
        raise ValueError(f"oracle_down_proj_mx status {st}")
    return out


def moe_backward(x, x_dtype: str, logits, dy, dy_dtype: str, k: int, e0: int, E_loc: int, w_dtype: str,
                 W_gate, W_up, W_down, tokens=None, experts=None, want_dx=True, want_dlogits=True,
                 want_dw=True) -> dict:
    """fp64 gradients of L = sum(dy * y): dx [n_tokens, d], dlogits [n_tokens, E] for
    ``tokens`` (default all), dW_gate/dW_up [n_experts, d, f] and dW_down [n_experts, f, d]
    for the local ``experts`` (default all)."""
    sd = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}
    xa, dya = _c(x, sd[x_dtype]), _c(dy, sd[dy_dtype])
    lg = _c(logits, np.float32)
    T, E = lg.shape
    d = xa.shape[1]
    f = W_gate.shape[2]
    wg, wu, wd = (_c(w, sd[w_dtype]) for w in (W_gate, W_up, W_down))
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    exps = np.arange(E_loc, dtype=np.int32) if experts is None else _c(experts, np.int32)
    out = {}
    dx = np.empty((tok.size, d)) if want_dx else None
    dl = np.empty((tok.size, E)) if want_dlogits else None
    dwg = np.empty((exps.size, d, f)) if want_dw else None
    dwu = np.empty((exps.size, d, f)) if want_dw else None
    dwd = np.empty((exps.size, f, d)) if want_dw else None
    st = _load().oracle_moe_backward(_p(xa), DT[x_dtype], _p(lg), T, d, f, E, k, e0, E_loc, DT[w_dtype], _p(wg),
                                     _p(wu), _p(wd), _p(dya), DT[dy_dtype], _p(tok), tok.size, _p(dx), _p(dl),
                                     _p(exps), exps.size, _p(dwg), _p(dwu), _p(dwd), threads())
    if st != 0:
        raise ValueError(f"oracle_moe_backward status {st}")
    out.update(dx=dx, dlogits=dl, dW_gate=dwg, dW_up=dwu, dW_down=dwd)
    return out


# ----------------------------------------------------------------------------- MXFP8 backward
def mx_dequantized(a, axis: int) -> np.ndarray:
    """Values of ``a`` (fp64) after MXFP8 quantisation in 32-blocks along ``axis`` (the
    rule of ``mx_quantize``); a length that is not a multiple of 32 is padded with zeros
    (zeros never raise a block's amax) and the padding is dropped again."""
    a = np.moveaxis(np.asarray(a, np.float64), axis, -1)
    n = a.shape[-1]
    pad = (-n) % 32
    if pad:
        a = np.concatenate([a, np.zeros(a.shape[:-1] + (pad,))], axis=-1)
    K = a.shape[-1]
    lead = int(np.prod(a.shape[:-1])) if a.ndim > 1 else 1
    if lead == 0 or K == 0:
        return np.moveaxis(a[..., :n], -1, axis)
    codes, scales = mx_quantize(np.ascontiguousarray(a.reshape(lead, K)), "f64", (lead, K, 1))
    vals = e4m3_decode(codes).reshape(lead, K // 32, 32) * np.exp2(scales.astype(np.float64) - 127.0)
    return np.moveaxis(vals.reshape(a.shape)[..., :n], -1, axis)


def _bf16_values(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def moe_backward_mx(x, logits, dy, k: int, e0: int, E_loc: int, W_gate, W_up, W_down) -> dict:
    """fp64 gradients of L = sum(dy * y) for the MXFP8 layer (bf16 bits in: x, dy [T, d];
    W_gate, W_up [E_loc, d, f]; W_down [E_loc, f, d]; logits [T, E] fp32).

    The forward is the MXFP8 layer's (x rows and the gate/up weights quantised along d).
    Every backward GEMM reads its two operands MXFP8-quantised in 32-blocks along that
    GEMM's own contraction axis ("Efficient MoE training for biological foundation
    models", section "MXFP8 Precision Reduces Memory Footprint": 8-bit values with one
    scale per 32 consecutive values, on Blackwell's MXFP8 GEMMs):
      dh = dy W_down^T              dy rows and W_down along d
      dx_row = dg W_gate^T + du W_up^T   dg, du rows and W_gate, W_up along f
      dW_down = h^T dy_rows         h and the expert's dy rows along the expert's rows
      dW_gate, dW_up = x_rows^T dg, du   x rows and dg / du along the expert's rows
    (the weight gradients contract over tokens, so their operands are quantised
    column-wise, each expert segment padded with zero rows to a multiple of 32).  The
    ScaledSwiGLU backward and the router gradient are exact fp64 arithmetic:
      du = p dh silu(g), dg = p dh u s (1 + g (1 - s)), dp = sum dh silu(g) u,
      dlogit_j = p_j (dp_j - sum_i p_i dp_i) over the token's k slots (dp = 0 off-slice).
    Returns dict(dx [T, d], dlogits [T, E], dW_gate, dW_up [E_loc, d, f], dW_down [E_loc, f, d]).
    """
    xv, dyv = _bf16_values(x), _bf16_values(dy)
    Wg, Wu, Wd = (_bf16_values(w) for w in (W_gate, W_up, W_down))
    lg = np.asarray(logits, np.float32)
    T, d = xv.shape
    E = lg.shape[1]
    f = Wg.shape[2]
    ids, probs = route_topk(lg, k)
    P = permute(ids, e0, E_loc)
    off, rst, slot = P["offsets"], P["row_src_token"], P["row_slot"]
    # forward operands (GEMM1 contracts over d) and backward operands of the row-wise GEMMs
    xq, Wgq, Wuq = mx_dequantized(xv, 1), mx_dequantized(Wg, 1), mx_dequantized(Wu, 1)
    dyq, Wd_d = mx_dequantized(dyv, 1), mx_dequantized(Wd, 2)
    Wg_f, Wu_f = mx_dequantized(Wg, 2), mx_dequantized(Wu, 2)
    dx = np.zeros((T, d))
    dp = np.zeros((T, k))
    dWg, dWu, dWd = np.zeros((E_loc, d, f)), np.zeros((E_loc, d, f)), np.zeros((E_loc, f, d))
    for e in range(E_loc):
        rows = slice(int(off[e]), int(off[e + 1]))
        t, j = rst[rows].astype(np.int64), slot[rows].astype(np.int64)
        if t.size == 0:
            continue
        p = probs[t, j][:, None]
        g, u = xq[t] @ Wgq[e], xq[t] @ Wuq[e]
        s = 1.0 / (1.0 + np.exp(-g))
        a = g * s
        h = p * a * u
        dh = dyq[t] @ Wd_d[e].T
        du = p * dh * a
        dg = p * dh * u * s * (1.0 + g * (1.0 - s))
        dp[t, j] = (dh * a * u).sum(axis=1)
        np.add.at(dx, t, mx_dequantized(dg, 1) @ Wg_f[e].T + mx_dequantized(du, 1) @ Wu_f[e].T)
        dWd[e] = mx_dequantized(h, 0).T @ mx_dequantized(dyv[t], 0)
        xr = mx_dequantized(xv[t], 0)
        dWg[e] = xr.T @ mx_dequantized(dg, 0)
        dWu[e] = xr.T @ mx_dequantized(du, 0)
    dl = np.zeros((T, E))
    mix = (probs * dp).sum(axis=1, keepdims=True)
    np.add.at(dl, (np.arange(T)[:, None].repeat(k, 1), ids), probs * (dp - mix))
    return dict(dx=dx, dlogits=dl, dW_gate=dWg, dW_up=dWu, dW_down=dWd)


# ----------------------------------------------------------------------------- per-tensor FP8
def fp8_tensor_exponent(amax: float) -> int:
    """Scale exponent X of a per-tensor FP8 (E4M3) tensor whose largest magnitude is
    ``amax``: the smallest integer with amax <= 448 * 2^X, so every value divided by 2^X
    lies within E4M3's finite range (448 = 0.875 * 2^9; with amax = m * 2^e, m in
    [0.5, 1): X = e - 9, or e - 8 when m > 0.875), clamped to [-127, 127]; 0 for an
    all-zero tensor."""
    a = float(amax)
    if a == 0.0:
        return 0
    m, e = np.frexp(a)
    X = int(e) - 9 + (1 if m > 0.875 else 0)
    return max(-127, min(127, X))


def fp8_tensor_quantize(a) -> tuple[np.ndarray, int]:
    """Per-tensor FP8: E4M3 codes of a / 2^X (round to nearest even) and X for the whole of
    ``a`` (fp64 values)."""
    v = np.asarray(a, np.float64)
    X = fp8_tensor_exponent(np.abs(v).max() if v.size else 0.0)
    return e4m3_encode(v * np.exp2(-X)), X


def fp8_tensor_dequantized(a) -> np.ndarray:
    codes, X = fp8_tensor_quantize(a)
    return e4m3_decode(codes) * np.exp2(X)


def moe_forward_fp8(x, logits, k: int, e0: int, E_loc: int, W_gate, W_up, W_down, tokens=None) -> np.ndarray:
    """fp64 layer output [n_tokens, d] of the per-tensor FP8 layer (bf16 bits in: x [T, d];
    W_gate, W_up [E_loc, d, f]; W_down [E_loc, f, d]; logits [T, E] fp32).

    "Efficient MoE training for biological foundation models", section "MXFP8 Precision
    Reduces Memory Footprint" (the layer runs in FP8 as well as MXFP8): here every GEMM
    operand is an E4M3 tensor with one power-of-two scale for the whole tensor
    (``fp8_tensor_quantize``): x [T, d] as one tensor; each expert's W_gate, W_up and
    W_down as one tensor each; h (all local routed rows, after the probability scaling)
    as one tensor.  Accumulation, SwiGLU and the slot-ordered combine are exact fp64.
    """
    xv = _bf16_values(x)
    Wg, Wu, Wd = (_bf16_values(w) for w in (W_gate, W_up, W_down))
    lg = np.asarray(logits, np.float32)
    T, d = xv.shape
    f = Wg.shape[2]
    ids, probs = route_topk(lg, k)
    P = permute(ids, e0, E_loc)
    off, rst, slot = P["offsets"], P["row_src_token"], P["row_slot"]
    xq = fp8_tensor_dequantized(xv)
    N = int(off[-1])
    h = np.zeros((N, f))
    for e in range(E_loc):
        rows = slice(int(off[e]), int(off[e + 1]))
        t, j = rst[rows].astype(np.int64), slot[rows].astype(np.int64)
        if t.size == 0:
            continue
        g = xq[t] @ fp8_tensor_dequantized(Wg[e])
        u = xq[t] @ fp8_tensor_dequantized(Wu[e])
        h[rows] = probs[t, j][:, None] * (g / (1.0 + np.exp(-g))) * u
    hq = fp8_tensor_dequantized(h)
    Y2 = np.zeros((N, d))
    for e in range(E_loc):
        rows = slice(int(off[e]), int(off[e + 1]))
        if off[e + 1] > off[e]:
            Y2[rows] = hq[rows] @ fp8_tensor_dequantized(Wd[e])
    y = np.zeros((T, d))
    p2r = P["pair_to_row"]
    for j in range(k):  # slot order
        r = p2r[:, j]
        m = r >= 0
        y[m] += Y2[r[m]]
    return y if tokens is None else y[np.asarray(tokens, np.int64)]


def moe_backward_fp8(x, logits, dy, k: int, e0: int, E_loc: int, W_gate, W_up, W_down) -> dict:
    """fp64 gradients of L = sum(dy * y) for the per-tensor FP8 layer (bf16 bits in: x, dy
    [T, d]; W_gate, W_up [E_loc, d, f]; W_down [E_loc, f, d]; logits [T, E] fp32).

    Every GEMM operand is one per-tensor FP8 tensor (``fp8_tensor_quantize``), the same
    whichever axis a GEMM contracts: x and dy as wholes; each expert's W_gate, W_up and
    W_down; h over all local routed rows; and the gradient of the gate/up pre-activation
    [dg du] over all local routed rows (one tensor, the input gradient of the first grouped
    linear).  The forward g, u, h are recomputed from the quantised x and weights.  Then,
    with Q the per-tensor quantisation:
      dh = Q(dy) Q(W_down)^T,  du = p dh silu(g),  dg = p dh u s (1 + g (1 - s)),
      dp = sum dh silu(g) u,   dx_row = Q(dg) Q(W_gate)^T + Q(du) Q(W_up)^T,
      dW_down = Q(h)^T Q(dy),  dW_gate = Q(x)^T Q(dg),  dW_up = Q(x)^T Q(du)  (per expert)
    and the router gradient as for the MXFP8 backward.
    Returns dict(dx [T, d], dlogits [T, E], dW_gate, dW_up [E_loc, d, f], dW_down [E_loc, f, d]).
    """
    xv, dyv = _bf16_values(x), _bf16_values(dy)
    Wg, Wu, Wd = (_bf16_values(w) for w in (W_gate, W_up, W_down))
    lg = np.asarray(logits, np.float32)
    T, d = xv.shape
    E = lg.shape[1]
    f = Wg.shape[2]
    ids, probs = route_topk(lg, k)
    P = permute(ids, e0, E_loc)
    off, rst, slot = P["offsets"], P["row_src_token"], P["row_slot"]
    N = int(off[-1])
    xq, dyq = fp8_tensor_dequantized(xv), fp8_tensor_dequantized(dyv)
    Wgq = [fp8_tensor_dequantized(Wg[e]) for e in range(E_loc)]
    Wuq = [fp8_tensor_dequantized(Wu[e]) for e in range(E_loc)]
    Wdq = [fp8_tensor_dequantized(Wd[e]) for e in range(E_loc)]
    h, dg, du = np.zeros((N, f)), np.zeros((N, f)), np.zeros((N, f))
    dp = np.zeros((T, k))
    for e in range(E_loc):
        rows = slice(int(off[e]), int(off[e + 1]))
        t, j = rst[rows].astype(np.int64), slot[rows].astype(np.int64)
        if t.size == 0:
            continue
        p = probs[t, j][:, None]
        g, u = xq[t] @ Wgq[e], xq[t] @ Wuq[e]
        s = 1.0 / (1.0 + np.exp(-g))
        a = g * s
        h[rows] = p * a * u
        dh = dyq[t] @ Wdq[e].T
        du[rows] = p * dh * a
        dg[rows] = p * dh * u * s * (1.0 + g * (1.0 - s))
        dp[t, j] = (dh * a * u).sum(axis=1)
    hq = fp8_tensor_dequantized(h)
    dgu = fp8_tensor_dequantized(np.concatenate([dg, du], axis=1)) if N else np.zeros((0, 2 * f))
    dgq, duq = dgu[:, :f], dgu[:, f:]
    dx = np.zeros((T, d))
    dWg, dWu, dWd = np.zeros((E_loc, d, f)), np.zeros((E_loc, d, f)), np.zeros((E_loc, f, d))
    for e in range(E_loc):
        rows = slice(int(off[e]), int(off[e + 1]))
        t = rst[rows].astype(np.int64)
        if t.size == 0:
            continue
        np.add.at(dx, t, dgq[rows] @ Wgq[e].T + duq[rows] @ Wuq[e].T)
        dWd[e] = hq[rows].T @ dyq[t]
        dWg[e] = xq[t].T @ dgq[rows]
        dWu[e] = xq[t].T @ duq[rows]
    dl = np.zeros((T, E))
    mix = (probs * dp).sum(axis=1, keepdims=True)
    np.add.at(dl, (np.arange(T)[:, None].repeat(k, 1), ids), probs * (dp - mix))
    return dict(dx=dx, dlogits=dl, dW_gate=dWg, dW_up=dWu, dW_down=dWd)
