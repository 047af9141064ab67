"""Parity of the MXFP8 layer backward (through the C ABI) against the oracle's MXFP8
backward (oracle.moe_backward_mx, fp64 over the oracle's own E4M3/E8M0 codec), on a B300:
dx, the router-logit gradients and the three expert weight gradients within the MXFP8
tolerance (relative L2 <= 5e-2), on small workloads with non-local slots, ragged segments
and all experts local, and on the EP64 MXFP8 slice at full size.

"Efficient MoE training for biological foundation models", section "GroupedLinear
Optimizes Expert Computation" (the fused GroupedMLP's backward) and section "MXFP8
Precision Reduces Memory Footprint" (8-bit values, one scale per 32 consecutive values).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, Workload, gen_dy, gen_logits, gen_weights, gen_x
from moe_testlib import TOL, rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported()
    return m


def _run(moe, w, x, lg, dy, Wg, Wu, Wd):
    wg, wu, wd = to_dev(Wg), to_dev(Wu), to_dev(Wd)
    pw = moe.moe_pack_weights(wg, wu, wd, "mxfp8")
    bw = moe.moe_pack_weights_backward_mx(wg, wu, wd)
    ids, probs = moe.moe_route_topk(to_dev(lg), w.k)
    g, ws = moe.moe_layer_backward_mx(to_dev(x), to_dev(dy), ids, probs, w.E, w.e0, pw, bw)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    return g


def _check(g, ref, tol=TOL["mxfp8"]):
    errs = {key: rel_l2(to_np(g[key]), ref[key]) for key in ("dx", "dlogits", "dW_gate", "dW_up", "dW_down")}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"relative L2 above {tol}: {bad} (all: {errs})"
    return errs


SMALL = [
    Workload("mxb_slice", 300, 256, 128, 16, 4, 4, 8, "mxfp8"),                        # non-local slots
    Workload("mxb_skew", 500, 384, 256, 8, 2, 0, 8, "mxfp8", ("normal", 0.5)),         # ragged segments
    Workload("mxb_e64", 1024, 256, 256, 64, 8, 0, 64, "mxfp8", ("normal", 0.5)),       # every slot local
    Workload("mxb_ep", 1000, 256, 128, 256, 8, 32, 16, "mxfp8"),                       # dx combined in its GEMM
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_mx_backward_matches_oracle(moe, w):
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    ref = oracle.moe_backward_mx(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    errs = _check(g, ref)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_mx_backward_full_size_ep64(moe):
    """The EP64 MXFP8 slice (T = 8192, d = 7168, f = 2048, 4 of 256 experts) at full size."""
    w = WORKLOADS["mxfp8_ep64_T8192"]
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    g = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    ref = oracle.moe_backward_mx(x, lg, dy, w.k, w.e0, w.E_loc, Wg, Wu, Wd)
    errs = _check(g, ref)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_mx_backward_deterministic(moe):
    w = SMALL[1]
    x, lg, dy = gen_x(w), gen_logits(w), gen_dy(w)
    Wg, Wu, Wd = gen_weights(w)
    a = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    b = _run(moe, w, x, lg, dy, Wg, Wu, Wd)
    for key in a:
        assert torch.equal(a[key], b[key]), key
