"""Per-tensor FP8 on a B300, through the C ABI, against the oracle's per-tensor FP8 layer
(oracle.moe_forward_fp8: x, each expert weight matrix and h each one E4M3 tensor with one
power-of-two scale):

* packing: the exponents of every expert's W_gate, W_up, W_down and the codes, bit for
  bit; every scale byte of a matrix equal to its exponent + 127;
* the permute's quantise-on-copy of x: codes bit for bit, one exponent for all of x (an
  all-zero x row and a large outlier included);
* the layer on small and ragged workloads, with the combine folded into GEMM2 (expert
  slices) and separate, within the FP8 tolerance (the MXFP8 one, 5e-2);
* deterministic results and the entry points that do not take FP8.

"Efficient MoE training for biological foundation models", section "MXFP8 Precision
Reduces Memory Footprint" (the layer runs in FP8 as well as MXFP8).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import Workload, bf16_bits, bf16_to_f32, gen_logits, gen_weights, gen_x
from moe_testlib import TOL, gate_up_rows, rel_l2, to_dev, to_np, unpack_act_sf, unpack_w_sf
from test_gpu_parity import gpu_layer, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported()
    return m


def _bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("E_loc,d,f", [(3, 256, 384), (2, 384, 128)])
def test_fp8_pack_matches_oracle(moe, E_loc, d, f):
    w = Workload("pack8", 1, d, f, E_loc, 1, 0, E_loc, "bf16")
    Wg, Wu, Wd = gen_weights(w)
    Wg[1] = bf16_bits(bf16_to_f32(Wg[1]) * 300.0)   # experts of very different magnitude
    Wu[0] = bf16_bits(bf16_to_f32(Wu[0]) * 1e-3)
    Wd[E_loc - 1] = 0  # an all-zero matrix: exponent 0, zero codes
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "fp8")
    torch.cuda.synchronize()
    w_exp = pw.w_exp.cpu().numpy()
    gr, ur = gate_up_rows(f)
    Wgu, Wdp = pw.Wgu.cpu().numpy(), pw.Wd.cpu().numpy()
    Sg = unpack_w_sf(pw.Wgu_scale.cpu().numpy(), E_loc, 2 * f, d)
    Sd = unpack_w_sf(pw.Wd_scale.cpu().numpy(), E_loc, d, f)
    for e in range(E_loc):
        for m, (W, rows) in enumerate(((Wg, gr), (Wu, ur))):
            codes, X = oracle.fp8_tensor_quantize(_bf16_values(W[e]))
            assert w_exp[m, e] == X, (m, e)
            np.testing.assert_array_equal(Wgu[e][rows, :], codes.T)
            assert (Sg[e][rows, :] == X + 127).all()
        codes, X = oracle.fp8_tensor_quantize(_bf16_values(Wd[e]))
        assert w_exp[2, e] == X
        np.testing.assert_array_equal(Wdp[e], codes.T)
        assert (Sd[e] == X + 127).all()
    assert w_exp[2, E_loc - 1] == 0


@pytest.mark.parametrize("T,E,k,e0,E_loc,d", [(300, 16, 4, 4, 8, 256), (64, 8, 2, 0, 8, 512)])
def test_fp8_permute_quantises_x_as_one_tensor(moe, T, E, k, e0, E_loc, d):
    w = Workload("perm8", T, d, 32, E, k, e0, E_loc, "bf16")
    x = gen_x(w)
    x[5] = 0
    x[7, 3] = np.uint16(0x4700)  # 32768.0: an outlier sets the tensor's exponent
    lg = gen_logits(w)
    ids, probs = moe.moe_route_topk(to_dev(lg), k)
    P = moe.moe_permute(to_dev(x), ids, probs, e0, E_loc, "fp8")
    torch.cuda.synchronize()
    O = oracle.permute(ids.cpu().numpy(), e0, E_loc)
    N = O["N"]
    codes, X = oracle.fp8_tensor_quantize(_bf16_values(x))
    assert X == 7  # 32768 <= 448 * 2^7 = 57344, > 448 * 2^6
    np.testing.assert_array_equal(P["perm_x"][:N].cpu().numpy(), codes[O["row_src_token"]])
    sf = unpack_act_sf(P["perm_x_scale"].cpu().numpy(), O["offsets"], d, N)
    assert (sf == X + 127).all()


SMALL = [
    Workload("fp8_a", 256, 256, 256, 8, 2, 0, 8, "fp8"),
    Workload("fp8_ragged", 300, 384, 384, 16, 4, 4, 8, "fp8"),
    Workload("fp8_zipf", 1024, 512, 256, 256, 8, 0, 32, "fp8", ("zipf", 1.1)),  # combine separate
    Workload("fp8_slice", 2000, 256, 256, 256, 8, 0, 4, "fp8"),                  # combine in GEMM2
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_fp8_layer_matches_oracle(moe, w):
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    err = rel_l2(to_np(y), yo)
    print(w.name, f"{err:.3e}")
    assert err <= TOL["fp8"], f"{w.name}: rel L2 {err:.3e}"
    assert moe.moe_layer_gemm_kernel(w.T, w.d, w.f, w.k, w.E, w.E_loc, "fp8", 1) == "cta"


def test_fp8_grouped_mlp_equals_layer(moe):
    """permute -> moe_grouped_mlp -> combine through the entry points gives the layer's y
    bit for bit (same kernels, same per-tensor exponents)."""
    w = SMALL[1]
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "fp8")
    xd, lgd = to_dev(x), to_dev(lg)
    y_layer, _ = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    ids, probs = moe.moe_route_topk(lgd, w.k)
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, "fp8")
    Y2, ws = moe.moe_grouped_mlp(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw)
    y = moe.moe_unpermute_combine(Y2, P["pair_to_row"], "fp8")
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(y, y_layer)


def test_fp8_deterministic(moe):
    w = SMALL[2]
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    a = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    b = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    assert torch.equal(a, b)


def test_fp8_split_calls_equal_layer(moe):
    """route -> permute -> GEMM1 (bf16 h and its amax in the entry's workspace, then h as one
    tensor) -> GEMM2 -> combine through the separate entry points gives the layer's y bit
    for bit; the row-gather GEMM1 entry refuses FP8."""
    from mixture_experts_layer_103_b300 import MoeError
    w = SMALL[1]
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "fp8")
    xd, lgd = to_dev(x), to_dev(lg)
    y_layer, _ = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    ids, probs = moe.moe_route_topk(lgd, w.k)
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, "fp8")
    h, hs, ws1 = moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw)
    Y2, ws2 = moe.moe_expert_gemm2(h, hs, P["offsets"], pw)
    y = moe.moe_unpermute_combine(Y2, P["pair_to_row"], "fp8")
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws1) == 0 and moe.moe_get_device_error(ws2) == 0
    assert torch.equal(y, y_layer)
    M = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, "fp8", maps_only=True)
    with pytest.raises(MoeError) as ei:
        moe.moe_expert_gemm1_swiglu_gather(xd, None, M["row_src_token"], M["offsets"], M["row_prob"], pw)
    assert ei.value.status == 2


# ----------------------------------------------------------------------------- backward
BWD = [
    Workload("fp8b_slice", 300, 256, 128, 16, 4, 4, 8, "fp8"),                       # non-local slots
    Workload("fp8b_skew", 500, 384, 256, 8, 2, 0, 8, "fp8", ("normal", 0.5)),        # ragged segments
    Workload("fp8b_e64", 1024, 256, 256, 64, 8, 0, 64, "fp8", ("normal", 0.5)),      # every slot local
    Workload("fp8b_ep", 1000, 256, 128, 256, 8, 32, 16, "fp8"),                      # dx combined in its GEMM
]


def _bwd(moe, w, x, lg, dy, Wg, Wu, Wd):
    wg, wu, wd = to_dev(Wg), to_dev(Wu), to_dev(Wd)
    pw = moe.moe_pack_weights(wg, wu, wd, "fp8")
    bw = moe.moe_pack_weights_backward_mx(wg, wu, wd, w_exp=pw.w_exp)
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    g, ws = moe.moe_layer_backward_mx(to_dev(x), to_dev(dy), ids, probs, w.E, w.e0, pw, bw)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    return g, pw, bw


@pytest.mark.parametrize("w", BWD, ids=[w.name for w in BWD])
def test_fp8_backward_matches_oracle(moe, w):
    """The per-tensor FP8 layer backward (C ABI) against oracle.moe_backward_fp8: dx, the
    router-logit gradients and the three weight gradients within the FP8 tolerance."""
    from synthetic import gen_dy
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g, _, _ = _bwd(moe, w, x, lg, dy, Wg, Wu, Wd)
    ref = oracle.moe_backward_fp8(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    errs = {key: rel_l2(to_np(g[key]), ref[key]) for key in ("dx", "dlogits", "dW_gate", "dW_up", "dW_down")}
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v <= TOL["fp8"]}
    assert not bad, f"relative L2 above {TOL['fp8']}: {bad}"


def test_fp8_backward_weights_use_forward_exponents(moe):
    """The backward weight layouts (each matrix transposed / re-blocked along the other
    axis) carry the forward pack's exponents: every scale byte of a matrix equals its
    exponent + 127, and the codes equal the oracle's per-tensor codes of that matrix."""
    w = BWD[0]
    Wg, Wu, Wd = gen_weights(w)
    wg, wu, wd = to_dev(Wg), to_dev(Wu), to_dev(Wd)
    pw = moe.moe_pack_weights(wg, wu, wd, "fp8")
    bw = moe.moe_pack_weights_backward_mx(wg, wu, wd, w_exp=pw.w_exp)
    torch.cuda.synchronize()
    w_exp = pw.w_exp.cpu().numpy()
    Wdq = bw.Wd_q.cpu().numpy()  # [E_loc, f, d]: W_down rows, blocks along d
    for e in range(w.E_loc):
        codes, X = oracle.fp8_tensor_quantize(_bf16_values(Wd[e]))
        assert w_exp[2, e] == X
        np.testing.assert_array_equal(Wdq[e], codes)
    S = unpack_w_sf(bw.Wd_scale.cpu().numpy(), w.E_loc, w.f, w.d)
    for e in range(w.E_loc):
        assert (S[e] == w_exp[2, e] + 127).all()


def test_fp8_backward_deterministic(moe):
    from synthetic import gen_dy
    w = BWD[1]
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    a, _, _ = _bwd(moe, w, x, lg, dy, Wg, Wu, Wd)
    b, _, _ = _bwd(moe, w, x, lg, dy, Wg, Wu, Wd)
    for key in a:
        assert torch.equal(a[key], b[key]), key
