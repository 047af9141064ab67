"""Pins of the oracle's layer backward (CPU): central finite differences of the forward
oracle in fp64 (itself pinned by test_oracle_pins.py), for x, all three weight tensors and
the router logits, on a slice of local experts (some slots not local) and on all experts.
A dropped term, a wrong sign or a transposed operand in the backward fails here."""
import numpy as np
import pytest

import oracle


def _problem(seed, T, d, f, E, k, E_loc):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E_loc, d, f)) / np.sqrt(d)
    Wu = rng.standard_normal((E_loc, d, f)) / np.sqrt(d)
    Wd = rng.standard_normal((E_loc, f, d)) / np.sqrt(f)
    # logits on a 2^-8 grid with distinct values per token: the top-k stays fixed under
    # the +-2^-12 perturbations below, and every perturbed value is exact in fp32
    lg = np.stack([rng.permutation(np.arange(E)) * 0.25 + rng.integers(-64, 64) / 256.0 for _ in range(T)])
    lg = lg.astype(np.float32)
    dy = rng.standard_normal((T, d))
    return x, lg, Wg, Wu, Wd, dy


def _loss(x, lg, Wg, Wu, Wd, dy, k, e0, E_loc):
    d, f, E = x.shape[1], Wg.shape[2], lg.shape[1]
    y = oracle.moe_forward(x, "f64", lg, d, f, E, k, e0, E_loc, Wg, Wu, Wd, "f64")
    return float((y * dy).sum())


@pytest.mark.parametrize("e0,E_loc", [(1, 2), (0, 4)])
def test_backward_matches_finite_differences(e0, E_loc):
    T, d, f, E, k = 5, 6, 4, 4, 2
    x, lg, Wg, Wu, Wd, dy = _problem(7 + e0, T, d, f, E, k, E_loc)
    g = oracle.moe_backward(x, "f64", lg, dy, "f64", k, e0, E_loc, "f64", Wg, Wu, Wd)
    L = lambda **kw: _loss(kw.get("x", x), kw.get("lg", lg), kw.get("Wg", Wg), kw.get("Wu", Wu),
                           kw.get("Wd", Wd), dy, k, e0, E_loc)
    eps = 1e-5

    def fd(name, arr):
        out = np.empty(arr.shape)
        for idx in np.ndindex(arr.shape):
            a, b = arr.copy(), arr.copy()
            a[idx] += eps
            b[idx] -= eps
            out[idx] = (L(**{name: a}) - L(**{name: b})) / (2 * eps)
        return out

    for name, arr, key in [("x", x, "dx"), ("Wg", Wg, "dW_gate"), ("Wu", Wu, "dW_up"), ("Wd", Wd, "dW_down")]:
        num = fd(name, arr)
        np.testing.assert_allclose(g[key], num, rtol=1e-6, atol=1e-8, err_msg=key)
    # router logits (fp32): perturb by 2^-12, exact on the 2^-8 grid
    h = 2.0 ** -12
    num = np.empty(lg.shape)
    for idx in np.ndindex(lg.shape):
        a, b = lg.copy(), lg.copy()
        a[idx] += np.float32(h)
        b[idx] -= np.float32(h)
        num[idx] = (L(lg=a) - L(lg=b)) / (2 * h)
    np.testing.assert_allclose(g["dlogits"], num, rtol=1e-5, atol=1e-7)


def test_backward_structure():
    """Linear in dy; logit gradients only on the k selected logits and summing to zero
    (softmax Jacobian); a token with no local expert gets zero dx."""
    T, d, f, E, k, e0, E_loc = 6, 5, 3, 4, 2, 2, 2
    x, lg, Wg, Wu, Wd, dy = _problem(3, T, d, f, E, k, E_loc)
    g1 = oracle.moe_backward(x, "f64", lg, dy, "f64", k, e0, E_loc, "f64", Wg, Wu, Wd)
    g2 = oracle.moe_backward(x, "f64", lg, 2.5 * dy, "f64", k, e0, E_loc, "f64", Wg, Wu, Wd)
    for key in ("dx", "dlogits", "dW_gate", "dW_up", "dW_down"):
        np.testing.assert_allclose(g2[key], 2.5 * g1[key], rtol=1e-12, atol=1e-14)
    ids, _ = oracle.route_topk(lg, k)
    for t in range(T):
        sel = set(ids[t].tolist())
        assert all(g1["dlogits"][t, q] == 0.0 for q in range(E) if q not in sel)
        assert abs(g1["dlogits"][t].sum()) < 1e-12
        if not any(e0 <= i < e0 + E_loc for i in ids[t]):
            assert (g1["dx"][t] == 0.0).all()


# ----------------------------------------------------------------------------- MXFP8 backward
# The MXFP8 backward is not differentiable through its quantisers, so it is pinned by an
# independent brute force of the same definition (oracle/brute.py: nearest-code quantiser,
# experts collected by a token scan, per-token rows, per-token outer products for the
# weight gradients) and by its distance to the unquantised backward.
from synthetic import Workload, bf16_to_f32, gen_dy, gen_logits, gen_weights, gen_x  # noqa: E402
from oracle import brute  # noqa: E402

MX_BWD = [
    Workload("mx_bwd_slice", 40, 64, 32, 8, 2, 2, 4, "mxfp8"),                    # non-local slots
    Workload("mx_bwd_skew", 70, 96, 64, 6, 3, 0, 6, "mxfp8", ("normal", 0.5)),    # ragged segments
]


@pytest.mark.parametrize("w", MX_BWD, ids=[w.name for w in MX_BWD])
def test_mx_backward_matches_brute_force(w):
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    got = oracle.moe_backward_mx(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    v = lambda a: bf16_to_f32(a).astype(np.float64)
    ref = brute.backward_mx(v(x), lg, v(dy), v(Wg), v(Wu), v(Wd), w.k, w.e0)
    for key in ref:
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert err <= 1e-12, (key, err)


@pytest.mark.parametrize("w", MX_BWD, ids=[w.name for w in MX_BWD])
def test_mx_backward_near_unquantised(w):
    """Same gradients as the bf16 backward up to the E4M3 rounding of the GEMM operands:
    relative L2 between 1 % and 15 % (quantisation happened, nothing larger broke)."""
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    got = oracle.moe_backward_mx(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    ref = oracle.moe_backward(x, "bf16", lg, dy, "bf16", w.k, w.e0, w.E_loc, "bf16", Wg, Wu, Wd)
    for key in ("dx", "dlogits", "dW_gate", "dW_up", "dW_down"):
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert 0.01 <= err <= 0.15, (key, err)


FP8_BWD = [
    Workload("fp8_bwd_slice", 40, 64, 32, 8, 2, 2, 4, "fp8"),                     # non-local slots
    Workload("fp8_bwd_skew", 70, 96, 64, 6, 3, 0, 6, "fp8", ("normal", 0.5)),     # ragged segments
]


@pytest.mark.parametrize("w", FP8_BWD, ids=[w.name for w in FP8_BWD])
def test_fp8_backward_matches_brute_force(w):
    """oracle.moe_backward_fp8 (vectorised over the permutation, C++ codec) against
    brute.backward_fp8 (token by token, nearest-code quantiser, exponent by search): a
    tensor quantised per expert or per row instead of as a whole, [dg du] split into two
    tensors, or h left unquantised fails it."""
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    got = oracle.moe_backward_fp8(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    v = lambda a: bf16_to_f32(a).astype(np.float64)
    ref = brute.backward_fp8(v(x), lg, v(dy), v(Wg), v(Wu), v(Wd), w.k, w.e0)
    for key in ref:
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert err <= 1e-12, (key, err)


@pytest.mark.parametrize("w", FP8_BWD, ids=[w.name for w in FP8_BWD])
def test_fp8_backward_near_unquantised(w):
    """Same gradients as the bf16 backward up to the E4M3 rounding of the GEMM operands:
    relative L2 between 1 % and 15 %."""
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    got = oracle.moe_backward_fp8(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    ref = oracle.moe_backward(x, "bf16", lg, dy, "bf16", w.k, w.e0, w.E_loc, "bf16", Wg, Wu, Wd)
    for key in ("dx", "dlogits", "dW_gate", "dW_up", "dW_down"):
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert 0.01 <= err <= 0.15, (key, err)
