"""Parity of the CUDA path (through the C ABI) against the CPU oracle, on a B300.

Bit-exact: routing ids, per-expert counts/offsets, the permutation maps, the permuted
rows (bf16/fp32 copies and MXFP8 codes + scales of x and of the weights).
Within the layer tolerances (relative L2 vs the fp64 oracle): 1e-5 fp32, 2e-2 bf16,
5e-2 MXFP8 -- on small workloads that span several 128-row tiles with ragged tails, on
edge cases (1/127/128/129 rows per expert, one expert holding every token, empty
experts, no local expert), and at full size on sampled tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, Workload, bf16_to_f32, gen_logits, gen_weights, gen_x, sample_tokens
from moe_testlib import TOL, bf16_bits_np, gate_up_rows, rel_l2, to_dev, to_np, unpack_act_sf, unpack_w_sf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported(), "needs compute capability 10.3 (B300)"
    return m


def _logits(kind, T, E, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((T, E)).astype(np.float32)
    if kind == "quarter":  # many exact ties
        return (rng.integers(-6, 6, size=(T, E)) * 0.25).astype(np.float32)
    if kind == "equal":
        return np.full((T, E), 0.5, np.float32)
    if kind == "signed_zero":
        lg = (rng.integers(-1, 2, size=(T, E)) * 0.0).astype(np.float32)
        lg[:, ::3] = -0.0
        lg[:, 1::5] = 0.0
        return lg
    # the router's lanes hold experts e = lane + 32 i: make one or two lanes hold all of a
    # token's top choices (distinct, or tied within the lane)
    if kind in ("one_lane", "one_lane_tied", "two_lanes"):
        lg = (rng.integers(-3, 3, size=(T, E)) * 0.5).astype(np.float32) if kind == "one_lane_tied" else \
            rng.standard_normal((T, E)).astype(np.float32)
        for t in range(T):
            lanes = rng.choice(32, 2 if kind == "two_lanes" else 1, replace=False)
            for ln in lanes:
                if kind == "one_lane_tied":
                    lg[t, ln::32] = 5.0
                else:
                    lg[t, ln::32] += 10.0
        return lg
    raise ValueError(kind)


# ----------------------------------------------------------------------------- route
@pytest.mark.parametrize("T,E,k,kind", [
    (512, 256, 8, "normal"), (300, 64, 8, "normal"), (64, 8, 2, "normal"), (100, 1024, 32, "normal"),
    (77, 37, 5, "normal"), (256, 256, 8, "quarter"), (33, 256, 8, "equal"), (40, 96, 7, "signed_zero"),
    (5, 1, 1, "normal"), (0, 8, 2, "normal"),
    (300, 256, 8, "one_lane"), (300, 256, 8, "one_lane_tied"), (200, 512, 16, "two_lanes"),
    (100, 1024, 32, "one_lane"), (150, 160, 9, "one_lane"), (120, 1024, 32, "quarter"),
])
def test_route_parity(moe, T, E, k, kind):
    lg = _logits(kind, T, E, seed=T + E)
    ids, probs = moe.moe_route_topk(to_dev(lg), k)
    torch.cuda.synchronize()
    oids, oprobs = oracle.route_topk(lg, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    np.testing.assert_allclose(probs.cpu().numpy(), oprobs, rtol=2e-6, atol=1e-7)


# ----------------------------------------------------------------------------- permute
PERM_CASES = [
    # T, E, k, e0, E_loc, d, x dtype
    (300, 64, 8, 0, 64, 256, "bf16"),
    (1000, 256, 8, 32, 32, 128, "bf16"),
    (2048, 256, 8, 0, 4, 512, "bf16"),
    (64, 8, 2, 0, 8, 128, "f32"),
    (257, 16, 4, 5, 1, 64, "f32"),
    (33, 9, 9, 0, 9, 8, "bf16"),
]


@pytest.mark.parametrize("T,E,k,e0,E_loc,d,xdt", PERM_CASES)
def test_permute_parity(moe, T, E, k, e0, E_loc, d, xdt):
    w = Workload("perm", T, d, 32, E, k, e0, E_loc, xdt)
    x = gen_x(w)
    lg = (np.random.default_rng(T).integers(-4, 4, size=(T, E)) * 0.5).astype(np.float32)  # ties
    ids_d, probs_d = moe.moe_route_topk(to_dev(lg), k)
    P = moe.moe_permute(to_dev(x), ids_d, probs_d, e0, E_loc, xdt)
    torch.cuda.synchronize()
    ids = ids_d.cpu().numpy()
    probs = probs_d.cpu().numpy()
    O = oracle.permute(ids, e0, E_loc)
    N = O["N"]
    np.testing.assert_array_equal(P["counts"].cpu().numpy(), O["counts"])
    np.testing.assert_array_equal(P["offsets"].cpu().numpy(), O["offsets"])
    np.testing.assert_array_equal(P["pair_to_row"].cpu().numpy(), O["pair_to_row"])
    rst = P["row_src_token"].cpu().numpy()[:N]
    np.testing.assert_array_equal(rst, O["row_src_token"])
    np.testing.assert_array_equal(P["row_prob"].cpu().numpy()[:N], probs[O["row_src_token"], O["row_slot"]])
    px = P["perm_x"][:N]
    got = bf16_bits_np(px) if xdt == "bf16" else px.cpu().numpy()
    np.testing.assert_array_equal(got, x[O["row_src_token"]])


@pytest.mark.parametrize("T,E,k,e0,E_loc,d,xdt", [
    (300, 64, 8, 0, 64, 256, "bf16"), (700, 256, 8, 0, 32, 384, "bf16"), (129, 8, 2, 2, 4, 128, "f32"),
])
def test_permute_mx_parity(moe, T, E, k, e0, E_loc, d, xdt):
    w = Workload("permmx", T, d, 32, E, k, e0, E_loc, xdt)
    x = gen_x(w)
    x[5] = 0  # an all-zero row: scale code 127
    lg = gen_logits(w)
    ids_d, probs_d = moe.moe_route_topk(to_dev(lg), k)
    P = moe.moe_permute(to_dev(x), ids_d, probs_d, e0, E_loc, "mxfp8")
    torch.cuda.synchronize()
    O = oracle.permute(ids_d.cpu().numpy(), e0, E_loc)
    N = O["N"]
    codes, scales = oracle.mx_quantize(x[O["row_src_token"]], xdt, (N, d, 1))
    np.testing.assert_array_equal(P["perm_x"][:N].cpu().numpy(), codes)
    sf = unpack_act_sf(P["perm_x_scale"].cpu().numpy(), O["offsets"], d, N)
    np.testing.assert_array_equal(sf, scales[:, :, 0])


# ----------------------------------------------------------------------------- pack
@pytest.mark.parametrize("dtype,E_loc,d,f", [("bf16", 3, 256, 96), ("f32", 2, 128, 64), ("mxfp8", 3, 256, 384),
                                             ("mxfp8", 2, 384, 128)])
def test_pack_parity(moe, dtype, E_loc, d, f):
    w = Workload("pack", 1, d, f, E_loc, 1, 0, E_loc, "f32" if dtype == "f32" else "bf16")
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), dtype)
    torch.cuda.synchronize()
    gr, ur = gate_up_rows(f)
    if dtype != "mxfp8":
        get = bf16_bits_np if dtype == "bf16" else (lambda t: t.cpu().numpy())
        Wgu = get(pw.Wgu)
        np.testing.assert_array_equal(Wgu[:, gr, :], np.swapaxes(Wg, 1, 2))
        np.testing.assert_array_equal(Wgu[:, ur, :], np.swapaxes(Wu, 1, 2))
        np.testing.assert_array_equal(get(pw.Wd), np.swapaxes(Wd, 1, 2))
        return
    cg, sg = oracle.mx_quantize(Wg, "bf16", (E_loc, d, f))
    cu, su = oracle.mx_quantize(Wu, "bf16", (E_loc, d, f))
    cd, sd = oracle.mx_quantize(Wd, "bf16", (E_loc, f, d))
    Wgu = pw.Wgu.cpu().numpy()
    np.testing.assert_array_equal(Wgu[:, gr, :], np.swapaxes(cg, 1, 2))
    np.testing.assert_array_equal(Wgu[:, ur, :], np.swapaxes(cu, 1, 2))
    np.testing.assert_array_equal(pw.Wd.cpu().numpy(), np.swapaxes(cd, 1, 2))
    S = unpack_w_sf(pw.Wgu_scale.cpu().numpy(), E_loc, 2 * f, d)
    np.testing.assert_array_equal(S[:, gr, :], np.swapaxes(sg, 1, 2))
    np.testing.assert_array_equal(S[:, ur, :], np.swapaxes(su, 1, 2))
    np.testing.assert_array_equal(unpack_w_sf(pw.Wd_scale.cpu().numpy(), E_loc, d, f), np.swapaxes(sd, 1, 2))


# ----------------------------------------------------------------------------- layer
def oracle_layer(w: Workload, x, lg, Wg, Wu, Wd, tokens=None):
    if w.dtype == "fp8":
        return oracle.moe_forward_fp8(x, lg, w.k, w.e0, w.E_loc, Wg, Wu, Wd, tokens=tokens)
    if w.dtype == "mxfp8":
        cg, sg = oracle.mx_quantize(Wg, "bf16", (w.E_loc, w.d, w.f))
        cu, su = oracle.mx_quantize(Wu, "bf16", (w.E_loc, w.d, w.f))
        cd, sd = oracle.mx_quantize(Wd, "bf16", (w.E_loc, w.f, w.d))
        return oracle.moe_forward(x, "bf16", lg, w.d, w.f, w.E, w.k, w.e0, w.E_loc, cg, cu, cd, "e4m3",
                                  (sg, su, sd), mx_act=True, tokens=tokens)
    return oracle.moe_forward(x, w.act_dtype, lg, w.d, w.f, w.E, w.k, w.e0, w.E_loc, Wg, Wu, Wd, w.act_dtype,
                              tokens=tokens)


def gpu_layer(moe, w: Workload, x, lg, Wg, Wu, Wd):
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), w.dtype)
    y, ws = moe.moe_layer_forward(to_dev(x), to_dev(lg), w.E, w.k, w.e0, pw)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    return y


SMALL = [
    Workload("f32_tiny", 64, 128, 256, 8, 2, 0, 8, "f32"),
    Workload("f32_slice", 200, 64, 96, 16, 4, 4, 8, "f32"),
    Workload("bf16_a", 256, 256, 256, 8, 2, 0, 8, "bf16"),
    Workload("bf16_ragged", 300, 200, 96, 16, 4, 4, 8, "bf16"),
    Workload("bf16_e64", 1024, 512, 512, 64, 8, 0, 64, "bf16", ("normal", 0.5)),
    Workload("bf16_ep64", 4096, 384, 256, 256, 8, 0, 4, "bf16"),
    Workload("bf16_zipf", 512, 256, 128, 256, 8, 0, 32, "bf16", ("zipf", 1.1)),
    Workload("bf16_pair_layer", 2048, 256, 256, 8, 2, 0, 8, "bf16"),   # T*k/E = 512: CTA-pair GEMMs
    Workload("bf16_pair_longk", 512, 4096, 128, 4, 2, 0, 4, "bf16"),   # 256 rows, d >= 4096: pair GEMM1
    Workload("mx_a", 256, 256, 256, 8, 2, 0, 8, "mxfp8"),
    Workload("mx_ragged", 300, 384, 384, 16, 4, 4, 8, "mxfp8"),
    Workload("mx_zipf", 1024, 512, 256, 256, 8, 0, 32, "mxfp8", ("zipf", 1.1)),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_layer_parity_small(moe, w):
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    err = rel_l2(to_np(y), yo)
    assert err <= TOL[w.dtype], f"{w.name}: rel L2 {err:.3e}"


def _forced_logits(counts, E, seed=0):
    """k = 1 logits giving exactly counts[e] tokens to expert e (tokens shuffled)."""
    owner = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int64)
    rng = np.random.default_rng(seed)
    rng.shuffle(owner)
    lg = rng.standard_normal((owner.size, E)).astype(np.float32)
    lg[np.arange(owner.size), owner] = 8.0
    return lg


EDGE = [
    ("rows_1_127_128_129", [1, 127, 128, 129, 0, 255, 0, 2]),
    ("one_expert_all", [0, 0, 0, 700, 0, 0, 0, 0]),
    ("tiny_segments", [1, 1, 1, 1, 1, 1, 1, 1]),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "mxfp8"])
@pytest.mark.parametrize("name,counts", EDGE, ids=[e[0] for e in EDGE])
def test_layer_edge_counts(moe, dtype, name, counts):
    E = len(counts)
    lg = _forced_logits(counts, E)
    T = lg.shape[0]
    w = Workload(name, T, 256, 128, E, 1, 0, E, dtype)
    x = gen_x(w)
    Wg, Wu, Wd = gen_weights(w)
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    assert rel_l2(to_np(y), yo) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_no_local_expert_gives_zeros(moe, dtype):
    E, T = 16, 64
    lg = _forced_logits([T // 4] * 4 + [0] * 12, E)
    w = Workload("nolocal", T, 128, 128, E, 2, 8, 8, dtype)  # experts 8..15 get nothing
    x = gen_x(w)
    Wg, Wu, Wd = gen_weights(w)
    lg[:, 8:] = -8.0
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    assert (to_np(y) == 0).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "mxfp8"])
def test_layer_empty_batch(moe, dtype):
    """T = 0: the fused forward launches nothing that touches rows and reports no error."""
    w = Workload("empty", 0, 256, 128, 8, 2, 0, 8, dtype)
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    assert tuple(y.shape) == (0, w.d)


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_ep_slices_sum_to_full_layer(moe, dtype):
    """Expert parallelism on one GPU: the partial outputs of the disjoint expert slices
    e0 = 0, 32, ..., 224 of a 256-expert top-8 layer (what each GPU of an EP8 group
    computes) sum to the full layer -- the sum-reduce that replaces the exchange step."""
    w = Workload("ep_sum", 256, 256, 128, 256, 8, 0, 256, dtype, ("zipf", 1.1))
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    acc = np.zeros((w.T, w.d))
    for e0 in range(0, 256, 32):
        sl = slice(e0, e0 + 32)
        acc += to_np(gpu_layer(moe, w.replace(e0=e0, E_loc=32), x, lg, Wg[sl], Wu[sl], Wd[sl]))
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    assert rel_l2(acc, yo) <= TOL[dtype]


SPLIT_CASES = [
    Workload("split", 512, 256, 256, 32, 4, 8, 16, "bf16"),           # 2 local slots per token
    Workload("split_slice", 3000, 256, 256, 256, 8, 8, 4, "bf16"),    # 1/8: combine folded into GEMM2
    Workload("split_slice_mx", 3000, 256, 256, 256, 8, 8, 4, "mxfp8"),
]


@pytest.mark.parametrize("w", SPLIT_CASES, ids=[c.name for c in SPLIT_CASES])
def test_split_calls_equal_fused_call(moe, w):
    """route -> permute -> gemm1 -> gemm2 -> combine through the separate entry points
    gives exactly the fused moe_layer_forward result, whichever way the layer combines."""
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), w.dtype)
    xd, lgd = to_dev(x), to_dev(lg)
    y_fused, _ = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    assert moe.moe_layer_fused_combine(w.k, w.E, w.E_loc, w.dtype) == (w.k * w.E_loc < w.E)
    ids, probs = moe.moe_route_topk(lgd, w.k)
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, w.dtype)
    hint = moe.moe_rows_hint(w.T, w.k, w.E)
    h, hs, _ = moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw,
                                           rows_hint=hint)
    Y2, _ = moe.moe_expert_gemm2(h, hs, P["offsets"], pw, rows_hint=hint)
    y = moe.moe_unpermute_combine(Y2, P["pair_to_row"], w.dtype)
    Y2b, _ = moe.moe_grouped_mlp(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw, rows_hint=hint)
    torch.cuda.synchronize()
    assert torch.equal(y, y_fused)
    N = int(P["offsets"][-1])
    assert torch.equal(Y2[:N], Y2b[:N])


# rows_hint values that force a GEMM kernel (moe.h MOE_KERNEL_*)
K_CTA, K_PAIR, K_SWAP = -1, -2, -3

COMBINE_CASES = [
    # workload, rows_hint (K_CTA: 1-CTA GEMM2, 4096: CTA-pair GEMM2, K_SWAP: swapped
    # operands, 0: N_cap / E_loc expected rows, i.e. mostly the swapped kernel here)
    (Workload("cmb_e64", 777, 256, 256, 64, 8, 0, 64, "bf16", ("normal", 0.5)), K_CTA),
    (Workload("cmb_e64_pair", 777, 256, 256, 64, 8, 0, 64, "bf16", ("normal", 0.5)), 4096),
    (Workload("cmb_e64_swap", 777, 256, 256, 64, 8, 0, 64, "bf16", ("normal", 0.5)), K_SWAP),
    (Workload("cmb_slice", 1000, 384, 128, 256, 8, 224, 32, "bf16"), 0),  # tokens with 0, 1 and many slots
    (Workload("cmb_zipf", 1000, 384, 128, 256, 8, 32, 32, "bf16", ("zipf", 1.1)), 0),
    (Workload("cmb_k32", 300, 128, 128, 64, 32, 0, 64, "bf16"), 0),
    (Workload("cmb_tail", 513, 200, 96, 16, 4, 4, 8, "bf16"), K_CTA),  # d % 64 != 0: a partial n-tile
    (Workload("cmb_tail_swap", 513, 200, 96, 16, 4, 4, 8, "bf16"), K_SWAP),  # d % 256: a partial weight tile
    (Workload("cmb_mx", 1024, 512, 256, 256, 8, 0, 32, "mxfp8", ("zipf", 1.1)), 0),
    (Workload("cmb_mx_e8", 700, 256, 256, 8, 4, 0, 8, "mxfp8"), 0),
    (Workload("cmb_mx_e8_swap", 700, 256, 256, 8, 4, 0, 8, "mxfp8"), K_SWAP),
    # rows_hint 1: the pass for few multi-slot tokens, here on a slice where many have several
    (Workload("cmb_sparse_pass", 1000, 384, 128, 256, 8, 0, 64, "bf16", ("zipf", 1.1)), 1),
]


@pytest.mark.parametrize("w,hint", COMBINE_CASES, ids=[c[0].name for c in COMBINE_CASES])
def test_gemm2_combine_equals_separate_kernels(moe, w, hint):
    """GEMM2 with the combine folded in (direct rows for tokens with one local slot, zero
    rows from the GEMM's extra warps, the slot sum for the rest) gives, bit for bit, GEMM2
    followed by the combine kernel, on two calls in a row, and the layer's y matches the
    oracle."""
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), w.dtype)
    xd = to_dev(x)
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, w.dtype)
    h, hs, _ = moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw,
                                           rows_hint=hint)
    Y2, _ = moe.moe_expert_gemm2(h, hs, P["offsets"], pw, rows_hint=hint)
    y_sep = moe.moe_unpermute_combine(Y2, P["pair_to_row"], "bf16")
    y1, ws = moe.moe_expert_gemm2_combine(h, hs, P["offsets"], P["row_src_token"], P["pair_to_row"], pw,
                                          rows_hint=hint)
    y1 = y1.clone()
    y2, _ = moe.moe_expert_gemm2_combine(h, hs, P["offsets"], P["row_src_token"], P["pair_to_row"], pw, ws=ws,
                                         rows_hint=hint)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    nloc = (P["pair_to_row"] >= 0).sum(1).cpu().numpy()
    if w.name == "cmb_slice":
        assert (nloc == 0).any() and (nloc == 1).any() and (nloc > 2).any()
    assert torch.equal(y1, y_sep), int((y1 != y_sep).sum())
    assert torch.equal(y2, y_sep)
    assert (to_np(y1)[nloc == 0] == 0).all()
    yl = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    assert rel_l2(to_np(yl), oracle_layer(w, x, lg, Wg, Wu, Wd)) <= TOL[w.dtype]


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_deterministic(moe, dtype):
    w = Workload("det", 777, 256, 256, 64, 8, 0, 64, dtype, ("normal", 0.5))
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), dtype)
    xd, lgd = to_dev(x), to_dev(lg)
    y1, ws = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    y1 = y1.clone()
    ws.fill_(0xA5)
    y2, _ = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "mxfp8"])
def test_canaries_untouched(moe, dtype):
    """Output and workspace carry guard bands before and after; none may change."""
    w = Workload("canary", 300, 256, 128, 16, 4, 2, 8, dtype)
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), dtype)
    pad = 4096
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    ybig = torch.full((w.T * w.d + 2 * pad,), 7.0, dtype=tdt, device="cuda")
    y = ybig[pad:pad + w.T * w.d].view(w.T, w.d)
    nb = moe.moe_layer_workspace_size(w.T, w.d, w.f, w.E, w.k, w.E_loc, dtype)
    wsbig = torch.full((nb + 2 * 256 * 64,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = wsbig[256 * 64: 256 * 64 + nb]
    moe.moe_layer_forward(to_dev(x), to_dev(lg), w.E, w.k, w.e0, pw, y=y, ws=ws)
    torch.cuda.synchronize()
    assert (ybig[:pad] == 7.0).all() and (ybig[-pad:] == 7.0).all()
    assert (wsbig[:256 * 64] == 0x5A).all() and (wsbig[256 * 64 + nb:] == 0x5A).all()
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    assert rel_l2(to_np(y), yo) <= TOL[dtype]


# ----------------------------------------------------------------------------- full size
FULL = ["tiny_fp32", "bf16_e64", "ep8_zipf_T512", "ep64_T2048", "ep64_T8192", "ep64_T32768",
        "mxfp8_ep8_zipf_T8192", "mxfp8_ep64_T8192", "fp8_ep64_T8192", "dense_bf16_T16384", "dense_mxfp8_T16384"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(moe, name):
    """Full workload through moe_layer_forward; routing and the whole permutation (counts,
    offsets, pair_to_row, row_src_token, row_prob) checked bit for bit for every token, the
    output on a seeded sample of tokens against the oracle."""
    w = WORKLOADS[name]
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    xd, lgd = to_dev(x), to_dev(lg)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), w.dtype)
    y, ws = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    ids, _ = moe.moe_route_topk(lgd, w.k)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    oids, _ = oracle.route_topk(lg, w.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), oids)
    # the permutation maps of the layer's own kernels (moe_permute, maps only) at full size
    probs_d = torch.empty(w.T, w.k, dtype=torch.float32, device="cuda")
    moe.moe_route_topk(lgd, w.k, topk_ids=ids, topk_probs=probs_d)
    P = moe.moe_permute(xd, ids, probs_d, w.e0, w.E_loc, "f32" if w.dtype == "f32" else "bf16", maps_only=True)
    torch.cuda.synchronize()
    O = oracle.permute(oids, w.e0, w.E_loc)
    N = O["N"]
    np.testing.assert_array_equal(P["counts"].cpu().numpy(), O["counts"])
    np.testing.assert_array_equal(P["offsets"].cpu().numpy(), O["offsets"])
    np.testing.assert_array_equal(P["pair_to_row"].cpu().numpy(), O["pair_to_row"])
    np.testing.assert_array_equal(P["row_src_token"].cpu().numpy()[:N], O["row_src_token"])
    np.testing.assert_array_equal(P["row_prob"].cpu().numpy()[:N],
                                  probs_d.cpu().numpy()[O["row_src_token"], O["row_slot"]])
    del P
    tok = sample_tokens(w, 48 if w.T > 64 else w.T)
    # always include tokens with a local expert so the sample is not all zeros
    local = np.where(((oids >= w.e0) & (oids < w.e0 + w.E_loc)).any(1))[0]
    tok = np.unique(np.concatenate([tok, local[:: max(1, local.size // 48)][:48]]))
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd, tokens=tok)
    err = rel_l2(to_np(y)[tok], yo)
    assert err <= TOL[w.dtype], f"{name}: rel L2 {err:.3e}"


# ----------------------------------------------------------------------------- CTA-pair kernel
PAIR_CASES = [
    # name, counts per expert (k = 1), d, f
    ("pair_edges", [1, 127, 128, 129, 255, 256, 257, 600], 256, 256),
    ("pair_tails", [300, 0, 513, 77], 200, 96),      # K and N tails: d % 64 != 0, 2f < 256
    ("pair_one_expert", [0, 0, 1100, 0], 384, 128),
    # 1-CTA cluster units: experts with 1..5 m-tiles (odd and even), odd n-tile counts
    ("odd_units", [1, 129, 300, 640, 0, 385, 128, 257], 192, 160),
]


@pytest.mark.parametrize("name,counts,d,f", PAIR_CASES, ids=[c[0] for c in PAIR_CASES])
def test_pair_kernel_matches_oracle(moe, name, counts, d, f):
    """bf16 GEMMs on token-major CTA pairs (forced by a large rows_hint) and on the
    swapped-operand kernel vs the oracle and vs the 1-CTA kernel."""
    E = len(counts)
    lg = _forced_logits(counts, E, seed=len(name))
    T = lg.shape[0]
    w = Workload(name, T, d, f, E, 1, 0, E, "bf16")
    x = gen_x(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "bf16")
    ids, probs = moe.moe_route_topk(to_dev(lg), 1)
    P = moe.moe_permute(to_dev(x), ids, probs, 0, E, "bf16")
    ys = {}
    for hint in (K_CTA, 4096, K_SWAP):  # 1-CTA kernel, token-major pairs, swapped operands
        Y2, ws = moe.moe_grouped_mlp(P["perm_x"], None, P["offsets"], P["row_prob"], pw, rows_hint=hint)
        ys[hint] = moe.moe_unpermute_combine(Y2, P["pair_to_row"], "bf16")
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    for hint, y in ys.items():
        assert rel_l2(to_np(y), yo) <= TOL["bf16"], hint
    for hint in (4096, K_SWAP):
        assert rel_l2(to_np(ys[hint]), to_np(ys[K_CTA])) <= 1e-2, hint


MX_PAIR_CASES = [
    ("mx_pair_edges", [1, 127, 128, 129, 255, 256, 257, 600], 256, 256),
    ("mx_pair_one_expert", [0, 0, 1100, 0], 384, 128),   # d % 256 == 128: a half-width last n-tile
    ("mx_pair_tails", [300, 0, 513, 77], 512, 384),
]


@pytest.mark.parametrize("name,counts,d,f", MX_PAIR_CASES, ids=[c[0] for c in MX_PAIR_CASES])
def test_mx_pair_kernel_matches_oracle(moe, name, counts, d, f):
    """MXFP8 GEMMs on token-major CTA pairs (block-scaled cta_group::2, forced by rows_hint =
    65536) and on the swapped-operand kernel vs the oracle and vs the 1-CTA MXFP8 kernel."""
    E = len(counts)
    lg = _forced_logits(counts, E, seed=len(name) + 3)
    w = Workload(name, lg.shape[0], d, f, E, 1, 0, E, "mxfp8")
    x = gen_x(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "mxfp8")
    ids, probs = moe.moe_route_topk(to_dev(lg), 1)
    P = moe.moe_permute(to_dev(x), ids, probs, 0, E, "mxfp8")
    ys = {}
    for hint in (K_CTA, 1 << 16, K_SWAP):
        Y2, ws = moe.moe_grouped_mlp(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw, rows_hint=hint)
        ys[hint] = moe.moe_unpermute_combine(Y2, P["pair_to_row"], "mxfp8")
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    for hint, y in ys.items():
        assert rel_l2(to_np(y), yo) <= TOL["mxfp8"], hint
    for hint in (1 << 16, K_SWAP):
        assert rel_l2(to_np(ys[hint]), to_np(ys[K_CTA])) <= 1e-2, hint


# ----------------------------------------------------------------------------- row-gather GEMM1
def _gather_vs_copy(moe, w, x, lg, Wg, Wu, Wd, hint=K_CTA):
    """GEMM1 reading x through row_src_token must equal GEMM1 on the permuted copy, bit for
    bit (same operand values, same MMA order); MXFP8 compares through GEMM2 (h scales live
    in the SF tile layout, whose pad bytes are unspecified)."""
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), w.dtype)
    xd = to_dev(x)
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    P = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, w.dtype)
    M = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, w.dtype, maps_only=True)
    torch.cuda.synchronize()
    N = int(P["offsets"][-1])
    for key in ("counts", "offsets", "pair_to_row"):
        assert torch.equal(P[key], M[key]), key
    assert torch.equal(P["row_src_token"][:N], M["row_src_token"][:N])
    assert torch.equal(P["row_prob"][:N], M["row_prob"][:N])
    h1, hs1, _ = moe.moe_expert_gemm1_swiglu(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw,
                                             rows_hint=hint)
    if w.dtype == "mxfp8":
        xq, xs = moe.moe_quantize_mx_rows(xd, pair_to_row=M["pair_to_row"])
        torch.cuda.synchronize()
        rst = M["row_src_token"][:N].long()
        assert torch.equal(P["perm_x"][:N], xq[rst])  # one quantisation rule, per row or per token
        h2, hs2, ws = moe.moe_expert_gemm1_swiglu_gather(xq, xs, M["row_src_token"], M["offsets"], M["row_prob"], pw)
    else:
        h2, hs2, ws = moe.moe_expert_gemm1_swiglu_gather(xd, None, M["row_src_token"], M["offsets"], M["row_prob"], pw,
                                                         rows_hint=hint)
    Y1, _ = moe.moe_expert_gemm2(h1, hs1, P["offsets"], pw, rows_hint=K_CTA)
    Y2, _ = moe.moe_expert_gemm2(h2, hs2, M["offsets"], pw, rows_hint=K_CTA)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(h1[:N], h2[:N])
    assert torch.equal(Y1[:N], Y2[:N])
    return N


GATHER_SMALL = ["bf16_a", "bf16_ragged", "bf16_e64", "bf16_ep64", "bf16_zipf", "mx_a", "mx_ragged", "mx_zipf"]


@pytest.mark.parametrize("name", GATHER_SMALL)
def test_gather_gemm1_matches_permuted_copy(moe, name):
    w = {c.name: c for c in SMALL}[name]
    Wg, Wu, Wd = gen_weights(w)
    assert _gather_vs_copy(moe, w, gen_x(w), gen_logits(w), Wg, Wu, Wd) > 0


@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_gather_gemm1_odd_units(moe, dtype):
    """Forced segments of 1..5 m-tiles (odd and even) with odd n-tile counts."""
    counts = [1, 129, 300, 640, 0, 385, 128, 257]
    d, f = (256, 256) if dtype == "mxfp8" else (192, 160)
    lg = _forced_logits(counts, len(counts), seed=5)
    w = Workload("gather_odd", lg.shape[0], d, f, len(counts), 1, 0, len(counts), dtype)
    Wg, Wu, Wd = gen_weights(w)
    assert _gather_vs_copy(moe, w, gen_x(w), lg, Wg, Wu, Wd) == sum(counts)


@pytest.mark.parametrize("name,counts,d,f", PAIR_CASES, ids=[c[0] for c in PAIR_CASES])
def test_pair_gather_gemm1_matches_pair_copy(moe, name, counts, d, f):
    """GEMM1 on CTA pairs with each CTA gathering its 128 token rows (the peer's stages
    relayed to the leader) equals GEMM1 on CTA pairs fed by TMA from the permuted copy,
    bit for bit: segment edges at 1/127/128/129/255/256/257 rows, K and N tails, one
    expert holding every token, odd unit counts."""
    E = len(counts)
    lg = _forced_logits(counts, E, seed=len(name) + 1)
    w = Workload(name, lg.shape[0], d, f, E, 1, 0, E, "bf16")
    Wg, Wu, Wd = gen_weights(w)
    assert _gather_vs_copy(moe, w, gen_x(w), lg, Wg, Wu, Wd, hint=4096) == sum(counts)


# ----------------------------------------------------------------------------- swapped operands
SWAP_CASES = [
    # name, counts per expert (k = 1), d, f: segments around the 16-token MMA granule, one and
    # two MMAs per tile (up to 256 / more tokens), experts split over several tiles, K and
    # weight-row tails (d % 64 != 0, 2f % 256 != 0)
    ("swap_edges", [1, 15, 16, 17, 255, 256, 257, 383, 384, 385, 1000], 256, 256),
    ("swap_tails", [300, 0, 513, 77], 200, 96),
    ("swap_small", [3, 64, 0, 40, 9, 64, 1, 33], 512, 384),
]


@pytest.mark.parametrize("name,counts,d,f", SWAP_CASES, ids=[c[0] for c in SWAP_CASES])
@pytest.mark.parametrize("dtype", ["bf16", "mxfp8"])
def test_swap_kernel_matches_oracle(moe, name, counts, d, f, dtype):
    """Both GEMMs on the swapped-operand kernel (weight rows on M, tokens on N) vs the
    oracle and vs the 1-CTA kernel; the bf16 GEMM1 with the token rows gathered from x
    equals the one fed by TMA from the permuted copy, bit for bit."""
    if dtype == "mxfp8":
        d, f = max(128, d // 128 * 128), max(128, f // 128 * 128)
    E = len(counts)
    lg = _forced_logits(counts, E, seed=len(name) + 11)
    w = Workload(name, lg.shape[0], d, f, E, 1, 0, E, dtype)
    x = gen_x(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), dtype)
    ids, probs = moe.moe_route_topk(to_dev(lg), 1)
    P = moe.moe_permute(to_dev(x), ids, probs, 0, E, dtype)
    ys = {}
    for hint in (K_CTA, K_SWAP):
        Y2, ws = moe.moe_grouped_mlp(P["perm_x"], P["perm_x_scale"], P["offsets"], P["row_prob"], pw, rows_hint=hint)
        ys[hint] = moe.moe_unpermute_combine(Y2, P["pair_to_row"], dtype)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd)
    for hint, y in ys.items():
        assert rel_l2(to_np(y), yo) <= TOL[dtype], hint
    assert rel_l2(to_np(ys[K_SWAP]), to_np(ys[K_CTA])) <= 1e-2
    if dtype == "bf16":
        assert _gather_vs_copy(moe, w, x, lg, Wg, Wu, Wd, hint=K_SWAP) == sum(counts)


def test_swap_layer_choice(moe):
    """moe_layer_forward runs the bf16 GEMM1 of the EP64 slice at T = 8192 on the
    swapped-operand kernel (gather mode) and the layer matches the oracle on sampled tokens."""
    w = WORKLOADS["ep64_T8192"]
    assert moe.moe_layer_gemm_kernel(w.T, w.d, w.f, w.k, w.E, w.E_loc, w.dtype, 1) == "swap"
    assert moe.moe_layer_gemm_kernel(w.T, w.d, w.f, w.k, w.E, w.E_loc, w.dtype, 2) == "pair"
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    y = to_np(gpu_layer(moe, w, x, lg, Wg, Wu, Wd))
    oids, _ = oracle.route_topk(lg, w.k)
    local = np.where(((oids >= w.e0) & (oids < w.e0 + w.E_loc)).any(1))[0]
    tok = np.unique(np.concatenate([local[:: max(1, local.size // 40)][:40], sample_tokens(w, 8)]))
    yo = oracle_layer(w, x, lg, Wg, Wu, Wd, tokens=tok)
    assert rel_l2(y[tok], yo) <= TOL["bf16"]


def test_pair_gather_layer(moe):
    """The bf16 layer at 2048 expected rows per expert runs GEMM1 on CTA pairs with the row
    gather (no permuted copy) and matches the oracle."""
    w = Workload("pair_gather_layer", 4096, 256, 256, 16, 8, 0, 16, "bf16", ("normal", 0.5))
    assert moe.moe_layer_gemm1_pairs(w.T, w.d, w.k, w.E, w.E_loc, "bf16")
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    y = gpu_layer(moe, w, x, lg, Wg, Wu, Wd)
    assert rel_l2(to_np(y), oracle_layer(w, x, lg, Wg, Wu, Wd)) <= TOL["bf16"]


def test_quantize_rows_matches_oracle(moe):
    """moe_quantize_mx_rows against the oracle's quantiser (codes and scale bytes)."""
    w = Workload("q", 37, 256, 128, 8, 2, 0, 8, "mxfp8")
    x = gen_x(w)
    xq, xs = moe.moe_quantize_mx_rows(to_dev(x))
    torch.cuda.synchronize()
    assert x.dtype == np.uint16  # bf16 storage
    codes, scales = oracle.mx_quantize(x, "bf16", (w.T, w.d, 1))
    np.testing.assert_array_equal(xq.cpu().numpy(), codes)
    np.testing.assert_array_equal(xs.cpu().numpy(), scales.reshape(w.T, w.d // 32))


# ----------------------------------------------------------------------------- placement plan
def test_eplb_plan_from_device_counts(moe):
    """The placement planner fed by the permute's per-expert counts of the Zipf-skewed
    256-expert routing (all experts local): a valid plan, the oracle's plan, and a lower
    peak GPU load than the contiguous 32-experts-per-GPU placement."""
    from oracle.eplb import eplb_plan
    w = WORKLOADS["ep8_zipf_T512"]
    lg = gen_logits(w)
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    x = torch.zeros(w.T, 64, dtype=torch.bfloat16, device="cuda")
    P = moe.moe_permute(x, ids, probs, 0, w.E, "bf16", maps_only=True)
    counts = P["counts"].cpu().numpy().astype(np.int64)
    oids, _ = oracle.route_topk(lg, w.k)
    np.testing.assert_array_equal(counts, np.bincount(oids.ravel(), minlength=w.E))
    G, S = 8, 40
    slot, rep, gl = moe.moe_eplb_plan(counts, G, S)
    oslot, orep, _ = eplb_plan(counts.tolist(), G, S)
    assert slot.tolist() == oslot and rep.tolist() == orep
    assert abs(gl.sum() - counts.sum()) <= 1e-9 * counts.sum()
    assert gl.max() < counts.reshape(G, -1).sum(1).max()
