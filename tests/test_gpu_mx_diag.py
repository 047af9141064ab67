"""Tight MXFP8 diagnostics of the two grouped GEMMs on a B300 (through the C ABI).

The layer test compares the MXFP8 output with the oracle only through y, at 5e-2.  These
two checks look inside the path, each against the oracle on the GPU's own operands:

* GEMM1 + ScaledSwiGLU + requantisation: the GPU's h codes and E8M0 scale bytes against
  the oracle's quantiser applied to the fp64 h of the same rows (h = p silu(g) u with g, u
  from the MXFP8 x rows and gate/up weights).  The GPU computes h in fp32, so a block's
  scale may differ by one binade where amax sits at a power of two, and a code may differ
  by one step where h sits at a rounding midpoint; both are counted and must be rare, and
  no other difference is allowed.
* GEMM2: the GPU's Y2 rows against oracle.down_proj_mx run on the GPU's own h codes and
  scales.  Only the bf16 rounding of Y2 separates the two: every element must lie within
  one bf16 ulp of the fp64 value (plus 1e-4 of the row's rms for elements near zero), and
  each row within 3e-3 relative L2 (bf16 rounding alone gives 1-2e-3).  A wrong scale byte in one 32-block of h, or a
  mis-indexed scale atom of W_down, moves a row by far more than that.

"Efficient MoE training for biological foundation models", section "MXFP8 Precision
Reduces Memory Footprint" (8-bit values with one scale per 32 consecutive values), and
section "GroupedLinear Optimizes Expert Computation" (ScaledSwiGLU fused after GEMM1).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, Workload, gen_logits, gen_weights, gen_x
from moe_testlib import to_dev, unpack_act_sf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported(), "needs compute capability 10.3 (B300)"
    return m


def _deq(codes, scales, axis):
    """Values of MXFP8 codes with scales [.., K/32, ..] (blocks of 32 along ``axis``)."""
    s = np.repeat(np.exp2(scales.astype(np.float64) - 127.0), 32, axis=axis)
    return oracle.e4m3_decode(codes) * s


def _ulp_bf16(v):
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def _run(moe, w: Workload, rows_wanted: int | None, hint=None):
    """MXFP8 permute -> GEMM1 -> GEMM2 through the separate entry points (rows_hint: the
    layer's own, or a forced kernel shape); returns the device results and the oracle-side
    operands for a set of permuted rows."""
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "mxfp8")
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    P = moe.moe_permute(to_dev(x), ids, probs, w.e0, w.E_loc, "mxfp8")
    hint = moe.moe_rows_hint(w.T, w.k, w.E) if hint is None else hint
    h, hs, ws1 = moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw,
                                             rows_hint=hint)
    Y2, ws2 = moe.moe_expert_gemm2(h, hs, P["offsets"], pw, rows_hint=hint)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws1) == 0 and moe.moe_get_device_error(ws2) == 0
    offs = P["offsets"].cpu().numpy().astype(np.int64)
    N = int(offs[-1])
    assert N > 0
    if rows_wanted is None or rows_wanted >= N:
        rows = np.arange(N)
    else:  # rows spread over every non-empty expert, first and last rows of segments included
        rng = np.random.default_rng(7)
        pick = [rng.choice(N, size=rows_wanted, replace=False)]
        for e in range(w.E_loc):
            if offs[e + 1] > offs[e]:
                pick.append([offs[e], offs[e + 1] - 1])
        rows = np.unique(np.concatenate(pick)).astype(np.int64)
    row_expert = (np.searchsorted(offs, rows, side="right") - 1).astype(np.int32)
    rst = P["row_src_token"].cpu().numpy()[rows].astype(np.int64)
    # the oracle's routing gives the slot of each (token, expert) and its fp64 probability
    oids, oprobs = oracle.route_topk(lg, w.k)
    slot = np.array([int(np.where(oids[t] == w.e0 + e)[0][0]) for t, e in zip(rst, row_expert)])
    p = oprobs[rst, slot]
    return dict(x=x, Wg=Wg, Wu=Wu, Wd=Wd, rows=rows, row_expert=row_expert, tok=rst, p=p, N=N, offs=offs,
                h=h.cpu().numpy(), hs=unpack_act_sf(hs.cpu().numpy(), offs, w.f, N),
                Y2=Y2[:N].float().cpu().numpy().astype(np.float64))  # rows >= N are never written


CASES = [
    Workload("mx_a", 256, 256, 256, 8, 2, 0, 8, "mxfp8"),
    Workload("mx_ragged", 300, 384, 384, 16, 4, 4, 8, "mxfp8"),
    Workload("mx_zipf", 1024, 512, 256, 256, 8, 0, 32, "mxfp8", ("zipf", 1.1)),
]
FULL = [("mxfp8_ep64_T8192", 96), ("mxfp8_ep8_zipf_T8192", 96)]
MX_PAIR_HINT = 1 << 16  # expected rows per expert from which MXFP8 GEMMs run on CTA pairs


K_CTA, K_SWAP = -1, -3  # rows_hint values that force a kernel (moe.h MOE_KERNEL_*)


def _cases():
    # hint 65536: both GEMMs on token-major CTA pairs (block-scaled cta_group::2 MMAs);
    # K_CTA: the 1-CTA kernel; K_SWAP: the swapped-operand pair kernel; None: the layer's
    # choice (the swapped kernel at both full-size slices)
    out = [(w, None, h) for w in CASES for h in (K_CTA, MX_PAIR_HINT, K_SWAP)]
    return out + [(WORKLOADS[n], r, h) for n, r in FULL for h in (None, K_CTA, MX_PAIR_HINT)]


@pytest.mark.parametrize("w,rows_wanted,hint", _cases(),
                         ids=[f"{w.name}-{'auto' if h is None else h}" for w, _, h in _cases()])
def test_mx_h_quantisation_and_gemm2(moe, w, rows_wanted, hint):
    R = _run(moe, w, rows_wanted, hint)
    rows, re_, tok = R["rows"], R["row_expert"], R["tok"]
    d, f, E_loc = w.d, w.f, w.E_loc
    # ---- GEMM1 + ScaledSwiGLU: fp64 h of these rows from the MXFP8 operands
    xc, xs = oracle.mx_quantize(R["x"][tok], "bf16", (rows.size, d, 1))
    xq = _deq(xc, xs[:, :, 0], axis=1)
    h_ref = np.empty((rows.size, f))
    for e in np.unique(re_):
        sel = np.where(re_ == e)[0]
        cg, sg = oracle.mx_quantize(R["Wg"][e], "bf16", (1, d, f))
        cu, su = oracle.mx_quantize(R["Wu"][e], "bf16", (1, d, f))
        Wgq = _deq(cg.reshape(1, d, f), sg, axis=1)[0]
        Wuq = _deq(cu.reshape(1, d, f), su, axis=1)[0]
        g, u = xq[sel] @ Wgq, xq[sel] @ Wuq
        h_ref[sel] = R["p"][sel, None] * (g / (1.0 + np.exp(-g))) * u
    hc_ref, hs_ref = oracle.mx_quantize(h_ref, "f64", (rows.size, f, 1))
    hs_ref = hs_ref[:, :, 0]
    hc_gpu, hs_gpu = R["h"][rows], R["hs"][rows]
    scale_diff = hs_gpu.astype(np.int64) - hs_ref.astype(np.int64)
    assert np.abs(scale_diff).max() <= 1, "a block scale off by more than one binade"
    n_scale = int((scale_diff != 0).sum())
    assert n_scale <= max(2, hs_ref.size // 1000), f"{n_scale} of {hs_ref.size} block scales differ"
    same_scale = np.repeat(scale_diff == 0, 32, axis=1)
    step = np.abs(hc_gpu.astype(np.int64) - hc_ref.astype(np.int64))
    # where the scales agree, a code may differ only by one step (a rounding midpoint)
    # and only where fp32 and fp64 h straddle it
    diff_codes = same_scale & (hc_gpu != hc_ref)
    both_zero = ((hc_gpu & 0x7F) == 0) & ((hc_ref & 0x7F) == 0)
    assert ((step == 1) | both_zero)[diff_codes].all(), "an h code more than one step from the oracle's"
    n_code = int(diff_codes.sum())
    assert n_code <= max(4, same_scale.sum() // 500), f"{n_code} of {int(same_scale.sum())} h codes differ"
    # ---- GEMM2 on the GPU's own h
    cd, sd = oracle.mx_quantize(R["Wd"], "bf16", (E_loc, f, d))
    o = oracle.down_proj_mx(hc_gpu, hs_gpu, re_, d, f, E_loc, cd, "e4m3", sd)
    y = R["Y2"][rows]
    rms = np.sqrt((o ** 2).mean(axis=1, keepdims=True))
    bad = np.abs(y - o) > _ulp_bf16(o) + 1e-4 * rms
    assert not bad.any(), f"{int(bad.sum())} Y2 elements beyond one bf16 ulp, e.g. row {np.argwhere(bad)[0]}"
    row_err = np.linalg.norm(y - o, axis=1) / np.maximum(np.linalg.norm(o, axis=1), 1e-300)
    assert row_err.max() <= 3e-3, f"row rel L2 {row_err.max():.2e}"
    print(f"{w.name}: {rows.size} rows; h scales differing {n_scale}/{hs_ref.size}, "
          f"codes differing {n_code}/{int(same_scale.sum())}; GEMM2 worst row rel L2 {row_err.max():.2e}")

