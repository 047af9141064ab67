"""Pins of the CPU oracle against things other than itself (CPU only).

* a hand-worked 2-expert example (closed forms, tests/golden/two_expert_example.json);
* an independent numpy brute force (dense evaluation of every expert, full stable sort,
  nearest-code quantiser) on tiny random inputs;
* invariants of the permutation (bijection, monotone offsets, stable order);
* special cases that reduce to a textbook routine (dense SwiGLU MLP by numpy matmul,
  softmax of equal logits = 1/k);
* linearity / homogeneity in W_down, token-permutation equivariance, EP-slice additivity;
* the E4M3 codec against torch's float8_e4m3fn (library routine) and the OCP spec's
  landmark values; the E8M0 scale rule on powers of two, 448 * 2^j, zero and subnormal
  blocks.

Sources: "Wide-EP ... (NVIDIA)" explainer, section "MoE basics"; "Efficient MoE training
for biological foundation models", sections "GroupedLinear Optimizes Expert Computation"
and "MXFP8 Precision Reduces Memory Footprint".
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from synthetic import WORKLOADS, bf16_bits, bf16_to_f32, gen_logits, gen_weights, gen_x

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_expert_example.json")


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def _np_silu(a):
    return a / (1.0 + np.exp(-a))


# ----------------------------------------------------------------------------- golden
@pytest.mark.parametrize("case", ["k1", "k2"])
def test_two_expert_hand_worked(case):
    g = json.load(open(GOLDEN))
    c = g["cases"][case]
    k = int(case[1])
    x = np.array(g["x"], np.float32)
    lg = np.array(g["logits"], np.float32)
    Wg, Wu, Wd = (np.array(g[n], np.float32) for n in ("W_gate", "W_up", "W_down"))
    ids, probs = oracle.route_topk(lg, k)
    assert ids.tolist() == c["ids"]
    np.testing.assert_allclose(probs, c["probs"], rtol=1e-15, atol=0)
    perm = oracle.permute(ids, 0, 2)
    assert perm["counts"].tolist() == c["counts"]
    assert perm["row_src_token"].tolist() == c["row_src_token"]
    y = oracle.moe_forward(x, "f32", lg, 2, 2, 2, k, 0, 2, Wg, Wu, Wd, "f32")
    np.testing.assert_allclose(y, c["y"], rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------- brute force
def _tiny(seed, T, E, d, f, k, e0, E_loc, dtype="f32"):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    Wg = (rng.standard_normal((E_loc, d, f)) / np.sqrt(d)).astype(np.float32)
    Wu = (rng.standard_normal((E_loc, d, f)) / np.sqrt(d)).astype(np.float32)
    Wd = (rng.standard_normal((E_loc, f, d)) / np.sqrt(f)).astype(np.float32)
    if dtype == "bf16":
        x, Wg, Wu, Wd = (bf16_bits(a) for a in (x, Wg, Wu, Wd))
    return x, lg, Wg, Wu, Wd


def _vals(a, dtype):
    return (a if dtype == "f32" else bf16_to_f32(a)).astype(np.float64)


@pytest.mark.parametrize("seed,T,E,d,f,k,e0,E_loc", [
    (1, 16, 8, 16, 16, 1, 0, 8),
    (2, 16, 8, 16, 8, 2, 0, 8),
    (3, 12, 8, 8, 16, 8, 0, 8),      # k = E
    (4, 16, 8, 16, 16, 2, 3, 4),     # local slice
    (5, 9, 5, 4, 12, 3, 1, 2),       # E not a power of two
    (6, 16, 1, 8, 8, 1, 0, 1),       # E = 1
])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_oracle_matches_brute_force(seed, T, E, d, f, k, e0, E_loc, dtype):
    x, lg, Wg, Wu, Wd = _tiny(seed, T, E, d, f, k, e0, E_loc, dtype)
    y = oracle.moe_forward(x, dtype, lg, d, f, E, k, e0, E_loc, Wg, Wu, Wd, dtype)
    yb = brute.forward(_vals(x, dtype), lg, _vals(Wg, dtype), _vals(Wu, dtype), _vals(Wd, dtype), k, e0)
    assert rel_l2(y, yb) <= 1e-12
    np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("seed,T,E,d,f,k,e0,E_loc", [
    (7, 8, 8, 32, 32, 2, 0, 8),
    (8, 6, 8, 64, 32, 3, 2, 4),
])
def test_oracle_mx_matches_brute_force(seed, T, E, d, f, k, e0, E_loc):
    x, lg, Wg, Wu, Wd = _tiny(seed, T, E, d, f, k, e0, E_loc, "bf16")
    # weights: oracle quantiser (per column, blocks of 32 along K) vs the brute quantiser
    cg, sg = oracle.mx_quantize(Wg, "bf16", (E_loc, d, f))
    cu, su = oracle.mx_quantize(Wu, "bf16", (E_loc, d, f))
    cd, sd = oracle.mx_quantize(Wd, "bf16", (E_loc, f, d))
    deq = []
    for W, c, s in ((Wg, cg, sg), (Wu, cu, su), (Wd, cd, sd)):
        wt = np.swapaxes(bf16_to_f32(W).astype(np.float64), 1, 2)  # blocks along K -> last axis
        bc, bs, bd = brute.mx_quantize_rows(wt)
        assert np.array_equal(np.swapaxes(bc, 1, 2), c)
        assert np.array_equal(np.swapaxes(bs, 1, 2), s)
        deq.append(np.swapaxes(bd, 1, 2))
    y = oracle.moe_forward(x, "bf16", lg, d, f, E, k, e0, E_loc, cg, cu, cd, "e4m3", (sg, su, sd), mx_act=True)
    yb = brute.forward(bf16_to_f32(x).astype(np.float64), lg, *deq, k, e0, mx=True)
    # identical rule, fp64 on both sides: the h codes can only differ where the two fp64
    # evaluation orders straddle an E4M3 rounding midpoint (measure zero for random data)
    assert rel_l2(y, yb) <= 1e-12


# ----------------------------------------------------------------------------- routing
def test_route_ties_all_equal():
    T, E, k = 5, 37, 6
    lg = np.full((T, E), 0.75, np.float32)
    ids, p = oracle.route_topk(lg, k)
    assert (ids == np.arange(k)[None, :]).all()
    assert (p == 1.0 / k).all() or np.allclose(p, 1.0 / k, rtol=1e-15, atol=0)


def test_route_forced_ties_quarter_grid():
    rng = np.random.default_rng(11)
    lg = (rng.integers(-8, 8, size=(200, 64)) * 0.25).astype(np.float32)
    ids, _ = oracle.route_topk(lg, 8)
    for t in range(lg.shape[0]):
        bi, _ = brute.topk(lg[t], 8)
        assert ids[t].tolist() == bi.tolist()


def test_route_signed_zero_equal():
    lg = np.zeros((1, 8), np.float32)
    lg[0, 2] = -0.0
    lg[0, 5] = 1.0
    lg[0, 7] = -1.0
    ids, _ = oracle.route_topk(lg, 3)
    assert ids[0].tolist() == [5, 0, 1]


def test_route_rejects_nan():
    lg = np.zeros((2, 4), np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(ValueError):
        oracle.route_topk(lg, 2)


def test_route_infinities_order():
    lg = np.array([[0.0, -np.inf, 3.0, np.inf, -1.0]], np.float32)
    ids, _ = oracle.route_topk(lg, 5)
    assert ids[0].tolist() == [3, 2, 0, 4, 1]


def test_route_probs_sum_to_one():
    lg = gen_logits(WORKLOADS["bf16_e64"], T=256)
    _, p = oracle.route_topk(lg, 8)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    assert (np.diff(p, axis=1) <= 0).all()


# ----------------------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,e0,E_loc", [(300, 64, 8, 0, 64), (257, 256, 8, 32, 32), (100, 256, 8, 0, 4),
                                             (64, 8, 2, 0, 8), (33, 9, 9, 0, 9), (50, 16, 4, 15, 1)])
def test_permutation_invariants(T, E, k, e0, E_loc):
    rng = np.random.default_rng(T + E)
    lg = (rng.integers(-4, 4, size=(T, E)) * 0.5).astype(np.float32)  # many ties
    ids, _ = oracle.route_topk(lg, k)
    P = oracle.permute(ids, e0, E_loc)
    local = (ids >= e0) & (ids < e0 + E_loc)
    assert int(P["counts"].sum()) == int(local.sum()) == P["N"]
    if E_loc == E:
        assert P["N"] == T * k
    off = P["offsets"]
    assert off[0] == 0 and (np.diff(off) == P["counts"]).all()
    p2r = P["pair_to_row"]
    assert ((p2r >= 0) == local).all()
    rows = p2r[local]
    assert sorted(rows.tolist()) == list(range(P["N"]))           # bijection onto [0, N)
    for e in range(E_loc):
        seg = P["row_src_token"][off[e]:off[e + 1]]
        assert (np.diff(seg) > 0).all()                              # stable: ascending tokens
        assert all((ids[t] == e0 + e).any() for t in seg)
    for t in range(T):
        for j in range(k):
            r = p2r[t, j]
            if r >= 0:
                assert P["row_src_token"][r] == t and P["row_slot"][r] == j


# ----------------------------------------------------------------------------- reductions
def test_identical_experts_equal_dense_mlp():
    """All experts identical and local: sum_j p_j = 1, so y = dense SwiGLU MLP(x)."""
    rng = np.random.default_rng(3)
    T, E, d, f, k = 20, 6, 24, 40, 3
    x = rng.standard_normal((T, d)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    wg = rng.standard_normal((d, f)).astype(np.float32) / 5
    wu = rng.standard_normal((d, f)).astype(np.float32) / 5
    wd = rng.standard_normal((f, d)).astype(np.float32) / 6
    rep = lambda a: np.repeat(a[None], E, axis=0)
    y = oracle.moe_forward(x, "f32", lg, d, f, E, k, 0, E, rep(wg), rep(wu), rep(wd), "f32")
    x64 = x.astype(np.float64)
    dense = (_np_silu(x64 @ wg.astype(np.float64)) * (x64 @ wu.astype(np.float64))) @ wd.astype(np.float64)
    np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-13)


def test_k1_is_dense_mlp_of_chosen_expert():
    rng = np.random.default_rng(4)
    T, E, d, f = 16, 4, 8, 16
    x, lg, Wg, Wu, Wd = _tiny(4, T, E, d, f, 1, 0, E)
    y = oracle.moe_forward(x, "f32", lg, d, f, E, 1, 0, E, Wg, Wu, Wd, "f32")
    e = np.argmax(lg, axis=1)
    for t in range(T):
        xt = x[t].astype(np.float64)
        ref = (_np_silu(xt @ Wg[e[t]].astype(np.float64)) * (xt @ Wu[e[t]].astype(np.float64))) @ Wd[e[t]].astype(np.float64)
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-14)


def test_linear_in_w_down_and_homogeneous():
    x, lg, Wg, Wu, Wd = _tiny(9, 12, 8, 16, 16, 2, 0, 8)
    rng = np.random.default_rng(10)
    Wd2 = rng.standard_normal(Wd.shape).astype(np.float32)
    fwd = lambda W: oracle.moe_forward(x, "f32", lg, 16, 16, 8, 2, 0, 8, Wg, Wu, W, "f32")
    np.testing.assert_allclose(fwd(Wd * np.float32(2.0)), 2.0 * fwd(Wd), rtol=1e-13, atol=1e-15)
    s = (Wd.astype(np.float64) + Wd2.astype(np.float64)).astype(np.float32)
    exact = (s.astype(np.float64) == Wd.astype(np.float64) + Wd2.astype(np.float64)).all()
    if exact:
        np.testing.assert_allclose(fwd(s), fwd(Wd) + fwd(Wd2), rtol=1e-12, atol=1e-13)
    else:  # fp32 sum not exact: compare against the exactly-representable pieces
        np.testing.assert_allclose(fwd(s), fwd(Wd) + fwd(Wd2), rtol=1e-6, atol=1e-7)


def test_token_permutation_equivariance():
    x, lg, Wg, Wu, Wd = _tiny(12, 20, 8, 8, 8, 2, 0, 8)
    perm = np.random.default_rng(13).permutation(20)
    y = oracle.moe_forward(x, "f32", lg, 8, 8, 8, 2, 0, 8, Wg, Wu, Wd, "f32")
    yp = oracle.moe_forward(x[perm], "f32", lg[perm], 8, 8, 8, 2, 0, 8, Wg, Wu, Wd, "f32")
    np.testing.assert_array_equal(yp, y[perm])


def test_ep_slice_additivity():
    """Sum over disjoint expert slices of a reduced 256-expert top-8 layer = full layer."""
    w = WORKLOADS["ep8_zipf_T512"].replace(T=24, d=64, f=32, E_loc=256)
    x = gen_x(w)
    lg = gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    full = oracle.moe_forward(x, "bf16", lg, w.d, w.f, w.E, w.k, 0, 256, Wg, Wu, Wd, "bf16")
    acc = np.zeros_like(full)
    for e0 in range(0, 256, 32):
        sl = slice(e0, e0 + 32)
        acc += oracle.moe_forward(x, "bf16", lg, w.d, w.f, w.E, w.k, e0, 32, Wg[sl], Wu[sl], Wd[sl], "bf16")
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-13)


def test_no_local_expert_rows_are_zero():
    x, lg, Wg, Wu, Wd = _tiny(14, 30, 16, 8, 8, 2, 0, 2)
    y = oracle.moe_forward(x, "f32", lg, 8, 8, 16, 2, 0, 2, Wg, Wu, Wd, "f32")
    ids, _ = oracle.route_topk(lg, 2)
    none = ~((ids < 2).any(axis=1))
    assert none.any()
    assert (y[none] == 0).all()


# ----------------------------------------------------------------------------- codec
def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2  # 0x7F and 0xFF only
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_e4m3_landmarks():
    v = oracle.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x38, 0x00, 0x80, 0xFE], np.uint8))
    assert v.tolist() == [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, 0.0, -0.0, -448.0]
    assert np.all(np.diff(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))) > 0)


def test_e4m3_encode_vs_nearest_search_and_torch():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(200_000) * 50,
        rng.standard_normal(200_000) * 2.0 ** -7,
        np.exp2(rng.uniform(-12, 9.2, 200_000)) * rng.choice([-1, 1], 200_000),
    ])
    # every midpoint between adjacent finite codes, and the codes themselves
    tab = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (tab[1:] + tab[:-1]) / 2
    v = np.concatenate([v, mids, -mids, tab, -tab, [460.0, 464.0, 500.0, 1e6, -1e6]])
    ours = oracle.e4m3_encode(v)
    np.testing.assert_array_equal(ours, brute.e4m3_nearest(v))
    # torch converts through fp32, so compare it on fp32-exact values only
    v32 = v.astype(np.float32)
    inr = np.abs(v32) < 448
    ref = torch.from_numpy(v32[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v32[inr].astype(np.float64)), ref)


def test_mx_scale_rule():
    blocks = []
    for j in range(-20, 20):                   # single power of two in a zero block -> exact
        b = np.zeros(32)
        b[j % 32] = 2.0 ** j
        blocks.append(b)
    for j in range(-10, 10):                   # 448 * 2^j, 1.5 * 2^j
        blocks.append(np.full(32, 448.0 * 2.0 ** j))
        blocks.append(np.linspace(-1.5, 1.5, 32) * 2.0 ** j)
    blocks.append(np.zeros(32))                # zero block -> code 127, zero elements
    blocks.append(np.full(32, 2.0 ** -130))    # amax below 2^-119 -> clamped X = -127 (code 0)
    a = np.stack(blocks)
    codes, scales = oracle.mx_quantize(a, "f64", (a.shape[0], 32, 1))
    scales = scales[:, 0, 0].astype(int)
    amax = np.abs(a).max(1)
    for i, m in enumerate(amax):
        if m == 0:
            assert scales[i] == 127 and (codes[i] == 0).all()
        elif m < 2.0 ** -119:
            assert scales[i] == 0
        else:
            assert scales[i] - 127 == int(np.floor(np.log2(m))) - 8
    deq = oracle.e4m3_decode(codes.reshape(a.shape)) * np.exp2(scales - 127.0)[:, None]
    for i in range(40):
        np.testing.assert_array_equal(deq[i], a[i])
    # 448 * 2^j: amax/2^X = 448 * 2^j / 2^(floor(log2 448) + j - 8) = 448 / 2 = 224 -> exact
    for i in range(40, 80, 2):
        np.testing.assert_array_equal(deq[i], a[i])
    # brute quantiser agrees on every block
    bc, bs, _ = brute.mx_quantize_rows(a)
    np.testing.assert_array_equal(bc, codes.reshape(a.shape))
    np.testing.assert_array_equal(bs[:, 0], scales)


# ----------------------------------------------------------------------------- MXFP8 down projection
@pytest.mark.parametrize("w_dtype", ["e4m3", "bf16"])
def test_down_proj_mx_matches_brute(w_dtype):
    """oracle.down_proj_mx (GEMM2 of given MXFP8 h rows) against numpy: the h codes decoded
    from the E4M3 bit fields (brute force's table) times 2^(s - 127) per 32-block along f,
    multiplied by W_down of the row's expert (E4M3 codes decoded the same way with their
    per-column scales along f, or exact bf16 values); a row with an out-of-range expert is
    zero.  A wrong block index, a transposed W_down or a dropped scale fails it."""
    rng = np.random.default_rng(11)
    E_loc, d, f, n = 3, 64, 96, 40
    codes = rng.integers(0, 256, size=(n, f)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11          # no NaN codes
    scales = rng.integers(120, 135, size=(n, f // 32)).astype(np.uint8)
    row_expert = rng.integers(0, E_loc, size=n).astype(np.int32)
    row_expert[[3, 17]] = -1                       # not a local row: zero output
    h = brute.e4m3_value(codes) * np.repeat(np.exp2(scales.astype(np.float64) - 127.0), 32, axis=1)
    Wd32 = (rng.standard_normal((E_loc, f, d)) / np.sqrt(f)).astype(np.float32)
    if w_dtype == "bf16":
        Wd = bf16_bits(Wd32)
        Wd_val = bf16_to_f32(Wd).astype(np.float64)
        Wd_scale = None
    else:
        Wd, Wd_scale = oracle.mx_quantize(Wd32, "f32", (E_loc, f, d))   # blocks along f
        Wd_val = brute.e4m3_value(Wd) * np.repeat(np.exp2(Wd_scale.astype(np.float64) - 127.0), 32, axis=1)
    want = np.zeros((n, d))
    for r in range(n):
        if row_expert[r] >= 0:
            want[r] = h[r] @ Wd_val[row_expert[r]]
    got = oracle.down_proj_mx(codes, scales, row_expert, d, f, E_loc, Wd, w_dtype, Wd_scale)
    assert (got[[3, 17]] == 0).all()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ----------------------------------------------------------------------------- per-tensor FP8
def test_fp8_tensor_exponent_definition():
    """oracle.fp8_tensor_exponent (from the fp64 bit fields) is the smallest integer X with
    amax <= 448 * 2^X, found here by search: at 448 * 2^j exactly, just above and below it,
    powers of two, the 0.875 mantissa edge, subnormals, huge values and 0."""
    probe = [0.0, 448.0, 448.0 * (1 + 2 ** -40), 448.0 * (1 - 2 ** -40), 1.0, 0.5, 2.0 ** -130, 2.0 ** -149,
             3.4e38, 0.875, 0.875 * (1 + 2 ** -30), 1.75, 7.0, 7.0 * (1 + 2 ** -20), 1e-3, 123.456]
    probe += [448.0 * 2.0 ** j for j in range(-20, 21, 3)]
    rng = np.random.default_rng(21)
    probe += list(np.exp(rng.uniform(-60, 60, 200)))
    for a in probe:
        X = oracle.fp8_tensor_exponent(a)
        assert X == brute.fp8_tensor_exponent(a), a
        if a > 0 and -127 < X < 127:
            assert a <= 448.0 * 2.0 ** X and not a <= 448.0 * 2.0 ** (X - 1), a


def test_fp8_tensor_quantize_vs_nearest_search():
    """Per-tensor quantisation: every code is the nearest E4M3 value of v / 2^X (ties to
    even), X from the tensor's largest magnitude; the largest element never saturates; a
    tensor of powers of two within range round-trips exactly; scaling a tensor by 2^s
    shifts X by s and leaves the codes unchanged."""
    rng = np.random.default_rng(22)
    for scale in (1e-3, 1.0, 37.0, 1e4):
        v = rng.standard_normal((17, 40)) * scale
        codes, X = oracle.fp8_tensor_quantize(v)
        bc, bX, bdeq = brute.fp8_tensor_quantize(v)
        assert X == bX
        np.testing.assert_array_equal(codes, bc)
        deq = oracle.e4m3_decode(codes) * 2.0 ** X
        np.testing.assert_array_equal(deq, bdeq)
        assert np.abs(v / 2.0 ** X).max() <= 448.0
        c2, X2 = oracle.fp8_tensor_quantize(v * 2.0 ** 5)
        assert X2 == X + 5
        np.testing.assert_array_equal(c2, codes)
    p2 = 2.0 ** rng.integers(-6, 8, size=50) * rng.choice([-1.0, 1.0], size=50)
    p2[0] = 2.0 ** 8                                 # amax 256 <= 448: X = 0
    codes, X = oracle.fp8_tensor_quantize(p2)
    assert X == 0
    np.testing.assert_array_equal(oracle.e4m3_decode(codes), p2)


@pytest.mark.parametrize("seed,T,E,d,f,k,e0,E_loc", [
    (31, 8, 8, 32, 32, 2, 0, 8),
    (32, 7, 8, 64, 32, 3, 2, 4),
    (33, 5, 4, 32, 64, 1, 1, 2),
])
def test_oracle_fp8_matches_brute_force(seed, T, E, d, f, k, e0, E_loc):
    """oracle.moe_forward_fp8 (vectorised over the permutation, C++ codec, exponent from the
    bit fields) against brute.forward_fp8 (token by token, dense expert evaluation, nearest
    search, exponent by search): a tensor quantised per row or per expert block instead of
    as a whole, a dropped probability or a wrong slot order fails it."""
    x, lg, Wg, Wu, Wd = _tiny(seed, T, E, d, f, k, e0, E_loc, "bf16")
    y = oracle.moe_forward_fp8(x, lg, k, e0, E_loc, Wg, Wu, Wd)
    yb = brute.forward_fp8(bf16_to_f32(x).astype(np.float64), lg, *(bf16_to_f32(w).astype(np.float64)
                                                                    for w in (Wg, Wu, Wd)), k, e0)
    assert rel_l2(y, yb) <= 1e-12


def test_fp8_layer_near_exact_layer():
    """The per-tensor FP8 layer stays near the exact bf16-input layer and is not equal to it:
    E4M3 keeps 3 mantissa bits, so each operand carries ~2-4 % relative rounding and the
    output lands at a few percent (measured 6.5-6.7 % at these sizes, against 7.7-7.9 %
    for the MXFP8 layer, whose power-of-two block scales put amax in [256, 512) and round
    the largest values more coarsely); a per-tensor scale off by a binade, a dropped
    dequantisation factor or unquantised h moves it out of that band."""
    x, lg, Wg, Wu, Wd = _tiny(41, 64, 8, 256, 128, 2, 0, 8, "bf16")
    d, f = 256, 128
    y8 = oracle.moe_forward_fp8(x, lg, 2, 0, 8, Wg, Wu, Wd)
    y = oracle.moe_forward(x, "bf16", lg, d, f, 8, 2, 0, 8, Wg, Wu, Wd, "bf16")
    cg, sg = oracle.mx_quantize(Wg, "bf16", (8, d, f))
    cu, su = oracle.mx_quantize(Wu, "bf16", (8, d, f))
    cd, sd = oracle.mx_quantize(Wd, "bf16", (8, f, d))
    ym = oracle.moe_forward(x, "bf16", lg, d, f, 8, 2, 0, 8, cg, cu, cd, "e4m3", (sg, su, sd), mx_act=True)
    err8, errmx = rel_l2(y8, y), rel_l2(ym, y)
    assert 0.03 < err8 <= 0.1
    assert 0.5 * errmx <= err8 <= errmx
