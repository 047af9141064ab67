"""Independent numpy brute force of the MoE expert layer (test infrastructure only).

It pins the C++ oracle on tiny inputs.  It shares no code with it and takes different
routes to the same definitions:

* top-k by a full stable sort on the key (-logit, id) with ``np.lexsort`` (the C++ side
  uses a partial sort with a comparator);
* every local expert's FFN is evaluated densely for every token with matrix products, and
  the routing probability multiplies the expert output after the down projection (the
  C++ side applies it to h; the two agree in exact arithmetic, and in fp64 to ~1e-15);
* the E4M3 quantiser is a nearest-code search over a table decoded from the format's
  bit fields, ties going to the code with an even mantissa (the C++ side rounds the
  scaled value arithmetically).  In MXFP8 mode the probability is applied before h is
  quantised, as the layer's fused epilogue does.

Sources: "Wide-EP ... (NVIDIA)" explainer, section "MoE basics" (router picks experts per
token, chosen experts' results are summed); "Efficient MoE training for biological
foundation models", sections "GroupedLinear Optimizes Expert Computation" (ScaledSwiGLU)
and "MXFP8 Precision Reduces Memory Footprint" (one scale per 32 consecutive values).
"""
from __future__ import annotations

import numpy as np


def _e4m3_table() -> np.ndarray:
    """Values of the 126 non-negative finite codes 0x00..0x7E from the bit fields."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append((m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, np.float64)


_TABLE = _e4m3_table()


def e4m3_nearest(v: np.ndarray) -> np.ndarray:
    """Codes of v by nearest search; ties to the even-mantissa code; |v| >= 448 -> 448."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 448.0).reshape(-1)
    dist = np.abs(a[:, None] - _TABLE[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among the (at most two) nearest codes prefer the one with an even code (even mantissa)
    even = cand & ((np.arange(0x7F) % 2) == 0)[None, :]
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    codes = pick.astype(np.uint8)
    codes = np.where(np.signbit(v.reshape(-1)), codes | np.uint8(0x80), codes)
    return codes.reshape(v.shape).astype(np.uint8)


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    mag = _TABLE[np.minimum(c & 0x7F, 0x7E)]
    return np.where(c & 0x80, -mag, mag)


def mx_quantize_rows(v: np.ndarray):
    """Quantise the last axis of v in blocks of 32; returns (codes, scale codes, dequantised)."""
    v = np.asarray(v, np.float64)
    *lead, K = v.shape
    b = v.reshape(*lead, K // 32, 32)
    amax = np.abs(b).max(axis=-1)
    _, ex = np.frexp(amax)  # amax = m 2^ex, m in [0.5, 1)
    X = np.where(amax == 0, 0, np.clip(ex - 1 - 8, -127, 127)).astype(np.int64)
    scaled = b * np.exp2(-X.astype(np.float64))[..., None]
    codes = e4m3_nearest(scaled)
    deq = e4m3_value(codes) * np.exp2(X.astype(np.float64))[..., None]
    return codes.reshape(v.shape), (X + 127).astype(np.uint8), deq.reshape(v.shape)


def topk(logits_row: np.ndarray, k: int):
    lg = np.asarray(logits_row, np.float64)
    order = np.lexsort((np.arange(lg.size), -lg))
    ids = order[:k]
    sel = lg[ids]
    w = np.exp(sel - sel.max())
    return ids, w / w.sum()


def silu(a):
    return a / (1.0 + np.exp(-a))


def forward(x, logits, Wg, Wu, Wd, k: int, e0: int, mx: bool = False) -> np.ndarray:
    """y [T, d] (fp64).  x [T,d], logits [T,E], Wg/Wu [E_loc,d,f], Wd [E_loc,f,d] (fp64 values).

    In ``mx`` mode the weights must already be the dequantised MXFP8 values; x rows and h
    rows are quantised here.
    """
    x = np.asarray(x, np.float64)
    T, d = x.shape
    E_loc = Wg.shape[0]
    if mx:
        x = mx_quantize_rows(x)[2]
    y = np.zeros((T, d))
    for t in range(T):
        ids, p = topk(logits[t], k)
        g = np.einsum("c,ecn->en", x[t], Wg)       # all local experts, densely
        u = np.einsum("c,ecn->en", x[t], Wu)
        act = silu(g) * u                           # [E_loc, f]
        if not mx:
            out = np.einsum("en,enm->em", act, Wd)  # every expert's FFN output
            for j in range(k):
                e = ids[j] - e0
                if 0 <= e < E_loc:
                    y[t] += p[j] * out[e]
        else:
            for j in range(k):
                e = ids[j] - e0
                if 0 <= e < E_loc:
                    h = mx_quantize_rows(p[j] * act[e])[2]
                    y[t] += h @ Wd[e]
    return y


def fp8_tensor_exponent(amax: float) -> int:
    """The smallest integer X with amax <= 448 * 2^X, by search (0 for amax == 0)."""
    if amax == 0:
        return 0
    X = -160
    while not amax <= 448.0 * 2.0 ** X:
        X += 1
    return int(min(max(X, -127), 127))


def fp8_tensor_quantize(v: np.ndarray):
    """Per-tensor FP8 of the whole of v: (codes, X, dequantised values)."""
    v = np.asarray(v, np.float64)
    X = fp8_tensor_exponent(float(np.abs(v).max()) if v.size else 0.0)
    codes = e4m3_nearest(v * 2.0 ** -X)
    return codes, X, e4m3_value(codes) * 2.0 ** X


def forward_fp8(x, logits, Wg, Wu, Wd, k: int, e0: int) -> np.ndarray:
    """y [T, d] (fp64) of the per-tensor FP8 layer, token by token: x, each expert's three
    matrices and h (every local routed row of the batch) are each one FP8 tensor."""
    xq = fp8_tensor_quantize(x)[2]
    E_loc = Wg.shape[0]
    Wgq = np.stack([fp8_tensor_quantize(Wg[e])[2] for e in range(E_loc)])
    Wuq = np.stack([fp8_tensor_quantize(Wu[e])[2] for e in range(E_loc)])
    Wdq = np.stack([fp8_tensor_quantize(Wd[e])[2] for e in range(E_loc)])
    T, d = xq.shape
    pairs = []  # (token, expert, h row) of every local slot
    for t in range(T):
        ids, p = topk(logits[t], k)
        for j in range(k):
            e = ids[j] - e0
            if 0 <= e < E_loc:
                pairs.append((t, e, p[j] * silu(xq[t] @ Wgq[e]) * (xq[t] @ Wuq[e])))
    y = np.zeros((T, d))
    if not pairs:
        return y
    hq = fp8_tensor_quantize(np.stack([h for _, _, h in pairs]))[2]
    for (t, e, _), h in zip(pairs, hq):
        y[t] += h @ Wdq[e]
    return y


def _q(v: np.ndarray, axis: int) -> np.ndarray:
    """Dequantised MXFP8 values of v in 32-blocks along ``axis`` (zero-padded to 32)."""
    v = np.moveaxis(np.asarray(v, np.float64), axis, -1)
    n = v.shape[-1]
    pad = (-n) % 32
    if pad:
        v = np.concatenate([v, np.zeros(v.shape[:-1] + (pad,))], axis=-1)
    return np.moveaxis(mx_quantize_rows(v)[2][..., :n], -1, axis)


def backward_mx(x, logits, dy, Wg, Wu, Wd, k: int, e0: int):
    """Gradients of sum(dy * y) for the MXFP8 layer, token by token (fp64 values in).

    Same definition as the oracle's MXFP8 backward, reached another way: experts are
    visited in id order and their tokens collected by a scan in ascending token order (no
    permutation tables), the per-row backward is evaluated one token at a time, and the
    weight gradients are accumulated as sums of per-token outer products of the
    column-wise quantised operands.
    """
    x, dy = np.asarray(x, np.float64), np.asarray(dy, np.float64)
    T, d = x.shape
    E_loc, _, f = Wg.shape
    E = logits.shape[1]
    sel = [topk(logits[t], k) for t in range(T)]
    xq, dyq = _q(x, 1), _q(dy, 1)
    Wgq, Wuq, Wd_d, Wg_f, Wu_f = _q(Wg, 1), _q(Wu, 1), _q(Wd, 2), _q(Wg, 2), _q(Wu, 2)
    dx, dlog = np.zeros((T, d)), np.zeros((T, E))
    dp = np.zeros((T, k))
    dWg, dWu, dWd = np.zeros((E_loc, d, f)), np.zeros((E_loc, d, f)), np.zeros((E_loc, f, d))
    for e in range(E_loc):
        members = [(t, list(sel[t][0]).index(e0 + e)) for t in range(T) if e0 + e in sel[t][0]]
        if not members:
            continue
        H, DG, DU = [], [], []
        for t, j in members:
            p = sel[t][1][j]
            g = np.array([xq[t] @ Wgq[e][:, n] for n in range(f)])
            u = np.array([xq[t] @ Wuq[e][:, n] for n in range(f)])
            s = 1.0 / (1.0 + np.exp(-g))
            dh = np.array([dyq[t] @ Wd_d[e][n, :] for n in range(f)])
            dg = p * dh * u * s * (1.0 + g * (1.0 - s))
            du = p * dh * g * s
            dp[t, j] = float(np.sum(dh * g * s * u))
            dx[t] += _q(dg[None, :], 1)[0] @ Wg_f[e].T + _q(du[None, :], 1)[0] @ Wu_f[e].T
            H.append(p * g * s * u)
            DG.append(dg)
            DU.append(du)
        ts = [t for t, _ in members]
        Hq, DYq = _q(np.array(H), 0), _q(dy[ts], 0)
        Xq, DGq, DUq = _q(x[ts], 0), _q(np.array(DG), 0), _q(np.array(DU), 0)
        for r in range(len(ts)):
            dWd[e] += np.outer(Hq[r], DYq[r])
            dWg[e] += np.outer(Xq[r], DGq[r])
            dWu[e] += np.outer(Xq[r], DUq[r])
    for t in range(T):
        ids, p = sel[t]
        mix = float(np.sum(p * dp[t]))
        for j in range(k):
            dlog[t, ids[j]] += p[j] * (dp[t, j] - mix)
    return dict(dx=dx, dlogits=dlog, dW_gate=dWg, dW_up=dWu, dW_down=dWd)


def backward_fp8(x, logits, dy, Wg, Wu, Wd, k: int, e0: int):
    """Gradients of sum(dy * y) for the per-tensor FP8 layer, token by token (fp64 values
    in): x, dy, each expert matrix, h and [dg du] (every local routed row of the batch) are
    one FP8 tensor each; experts visited by a scan over tokens, no permutation tables."""
    x, dy = np.asarray(x, np.float64), np.asarray(dy, np.float64)
    T, d = x.shape
    E_loc, _, f = Wg.shape
    E = logits.shape[1]
    xq, dyq = fp8_tensor_quantize(x)[2], fp8_tensor_quantize(dy)[2]
    Wgq = [fp8_tensor_quantize(Wg[e])[2] for e in range(E_loc)]
    Wuq = [fp8_tensor_quantize(Wu[e])[2] for e in range(E_loc)]
    Wdq = [fp8_tensor_quantize(Wd[e])[2] for e in range(E_loc)]
    route = [topk(logits[t], k) for t in range(T)]
    rows = []  # (token, slot, expert, h, dg, du) in expert order, ascending tokens
    dp = np.zeros((T, k))
    for e in range(E_loc):
        for t in range(T):
            ids, p = route[t]
            for j in range(k):
                if ids[j] - e0 != e:
                    continue
                g, u = xq[t] @ Wgq[e], xq[t] @ Wuq[e]
                s = 1.0 / (1.0 + np.exp(-g))
                dh = Wdq[e] @ dyq[t]
                dp[t, j] = np.sum(dh * g * s * u)
                rows.append((t, j, e, p[j] * g * s * u, p[j] * dh * u * s * (1.0 + g * (1.0 - s)), p[j] * dh * g * s))
    dx = np.zeros((T, d))
    dWg, dWu, dWd = np.zeros((E_loc, d, f)), np.zeros((E_loc, d, f)), np.zeros((E_loc, f, d))
    if rows:
        hq = fp8_tensor_quantize(np.stack([r[3] for r in rows]))[2]
        dgu = fp8_tensor_quantize(np.stack([np.concatenate([r[4], r[5]]) for r in rows]))[2]
        for (t, j, e, _, _, _), hr, gr in zip(rows, hq, dgu):
            dgq, duq = gr[:f], gr[f:]
            dx[t] += Wgq[e] @ dgq + Wuq[e] @ duq
            dWd[e] += np.outer(hr, dyq[t])
            dWg[e] += np.outer(xq[t], dgq)
            dWu[e] += np.outer(xq[t], duq)
    dl = np.zeros((T, E))
    for t in range(T):
        ids, p = route[t]
        mix = np.sum(p * dp[t])
        for j in range(k):
            dl[t, ids[j]] += p[j] * (dp[t, j] - mix)
    return dict(dx=dx, dlogits=dl, dW_gate=dWg, dW_up=dWu, dW_down=dWd)

