"""Parity of the layer backward (bf16, through the C ABI) against the oracle's fp64
backward, on a B300: dx, the router-logit gradients and the three expert weight
gradients, relative L2 <= 2e-2 (the forward's bf16 tolerance: the backward rounds the
recomputed pre-activations, dg/du and h to bf16 once each), on workloads spanning several
128-row tiles with ragged tails, a local expert slice, forced segment sizes, and full size
on sampled tokens and experts; determinism."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, Workload, gen_dy, gen_logits, gen_weights, gen_x, sample_tokens
from moe_testlib import rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu
TOL_BWD = 2e-2


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported()
    return m


def _run(moe, w, x, lg, dy, Wg, Wu, Wd):
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "bf16")
    WguT = moe.moe_pack_weights_backward(to_dev(Wg), to_dev(Wu))
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    g, ws = moe.moe_layer_backward(to_dev(x), to_dev(dy), ids, probs, w.E, w.e0, pw, to_dev(Wd), WguT)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    return g


def _check(g, ref, tokens=None, experts=None):
    sel_t = slice(None) if tokens is None else tokens
    sel_e = slice(None) if experts is None else experts
    errs = {
        "dx": rel_l2(to_np(g["dx"])[sel_t], ref["dx"]),
        "dlogits": rel_l2(to_np(g["dlogits"])[sel_t], ref["dlogits"]),
        "dW_gate": rel_l2(to_np(g["dW_gate"])[sel_e], ref["dW_gate"]),
        "dW_up": rel_l2(to_np(g["dW_up"])[sel_e], ref["dW_up"]),
        "dW_down": rel_l2(to_np(g["dW_down"])[sel_e], ref["dW_down"]),
    }
    bad = {k: v for k, v in errs.items() if not v <= TOL_BWD}
    assert not bad, errs


SMALL = [
    Workload("b_tiny", 64, 128, 96, 8, 2, 0, 8, "bf16"),
    Workload("b_slice", 200, 256, 128, 16, 4, 4, 8, "bf16"),
    Workload("b_e64", 1024, 512, 512, 64, 8, 0, 64, "bf16", ("normal", 0.5)),
    Workload("b_zipf", 512, 256, 128, 256, 8, 0, 32, "bf16", ("zipf", 1.1)),
    # under one local slot per token (k E_loc < E): the dx GEMM writes single-slot tokens'
    # rows and the zero rows itself, a sparse pass sums the rest
    Workload("b_ep", 1000, 256, 128, 256, 8, 32, 16, "bf16"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_backward_matches_oracle(moe, w):
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    ref = oracle.moe_backward(x, "bf16", lg, dy, "bf16", w.k, w.e0, w.E_loc, "bf16", Wg, Wu, Wd)
    _check(g, ref)


def _forced_logits(counts, E, seed=0):
    owner = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int64)
    rng = np.random.default_rng(seed)
    rng.shuffle(owner)
    lg = rng.standard_normal((owner.size, E)).astype(np.float32)
    lg[np.arange(owner.size), owner] = 8.0
    return lg


def test_backward_forced_segments(moe):
    """Segments of 0, 1, 127, 128, 129 and 300 rows (k = 1): ragged tiles, empty experts
    (their weight gradients must be exactly zero)."""
    counts = [1, 0, 127, 128, 129, 0, 300, 5]
    lg = _forced_logits(counts, len(counts), seed=3)
    w = Workload("b_forced", lg.shape[0], 192, 160, len(counts), 1, 0, len(counts), "bf16")
    x, dy = gen_x(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    ref = oracle.moe_backward(x, "bf16", lg, dy, "bf16", 1, 0, len(counts), "bf16", Wg, Wu, Wd)
    _check(g, ref)
    for e in (1, 5):
        assert (g["dW_gate"][e] == 0).all() and (g["dW_up"][e] == 0).all() and (g["dW_down"][e] == 0).all()


def test_backward_empty_batch(moe):
    """T = 0: no routed rows, so every weight gradient is exactly zero."""
    w = Workload("b_empty", 0, 128, 96, 8, 2, 0, 8, "bf16")
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    assert tuple(g["dx"].shape) == (0, w.d) and tuple(g["dlogits"].shape) == (0, w.E)
    for key in ("dW_gate", "dW_up", "dW_down"):
        assert (g[key] == 0).all(), key


def test_backward_deterministic(moe):
    w = SMALL[2]
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g1 = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    g1 = {k: v.clone() for k, v in g1.items()}
    g2 = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_backward_full_size_sampled(moe):
    """bf16_e64 at full size: dx and dlogits on sampled tokens, weight gradients of two
    experts (the oracle sums over all 4096 tokens for them)."""
    w = WORKLOADS["bf16_e64"]
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    tok = sample_tokens(w, 32)
    experts = np.array([3, 41], np.int32)
    ref = oracle.moe_backward(x, "bf16", lg, dy, "bf16", w.k, w.e0, w.E_loc, "bf16", Wg, Wu, Wd, tokens=tok,
                              experts=experts)
    _check(g, ref, tokens=tok, experts=experts)


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], Workload("b_pair", 512, 4096, 128, 4, 2, 0, 4, "bf16")],
                         ids=["b_slice", "b_e64", "b_pair_longk"])
def test_training_forward_saves_preactivations(moe, w):
    """moe_layer_forward_train: y bit-identical to moe_layer_forward, routing equal to
    moe_route_topk, and the backward on its saved g/u bit-identical to the backward that
    recomputes them."""
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "bf16")
    WguT = moe.moe_pack_weights_backward(to_dev(Wg), to_dev(Wu))
    xd, lgd, dyd = to_dev(x), to_dev(lg), to_dev(dy)
    y_t, ids, probs, gu, ws = moe.moe_layer_forward_train(xd, lgd, w.E, w.k, w.e0, pw)
    y, _ = moe.moe_layer_forward(xd, lgd, w.E, w.k, w.e0, pw)
    ids2, probs2 = moe.moe_route_topk(lgd, w.k)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(y_t, y) and torch.equal(ids, ids2) and torch.equal(probs, probs2)
    g_saved, ws1 = moe.moe_layer_backward(xd, dyd, ids, probs, w.E, w.e0, pw, to_dev(Wd), WguT, gu_saved=gu)
    g_saved = {k: v.clone() for k, v in g_saved.items()}
    g_recomp, ws2 = moe.moe_layer_backward(xd, dyd, ids, probs, w.E, w.e0, pw, to_dev(Wd), WguT)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws1) == 0 and moe.moe_get_device_error(ws2) == 0
    for key in g_saved:
        assert torch.equal(g_saved[key], g_recomp[key]), key
