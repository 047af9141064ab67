"""Failure detection without a GPU fault: every pipelined kernel waits on mbarriers with
a bounded wait; when the bound runs out it records MOE_ERR_TIMEOUT in the caller's error
word and returns.  The self-test entry point waits on a barrier nothing arrives on (a
flag that nothing sets); the status must come back as a timeout and the context must stay
usable for the next layer call."""
import time

import numpy as np
import pytest
import torch

import oracle
from synthetic import Workload, gen_logits, gen_weights, gen_x
from moe_testlib import TOL, rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported()
    return m


def test_bounded_wait_reports_timeout_and_context_survives(moe):
    t0 = time.perf_counter()
    code = moe.moe_selftest_wait_timeout(20_000_000)  # 20 ms
    dt = time.perf_counter() - t0
    assert code == 5  # MOE_ERR_TIMEOUT
    assert 0.015 <= dt < 5.0
    # the context is intact: a layer call right after runs and is correct
    w = Workload("after_timeout", 256, 256, 128, 8, 2, 0, 8, "bf16")
    x, lg = gen_x(w), gen_logits(w)
    Wg, Wu, Wd = gen_weights(w)
    pw = moe.moe_pack_weights(to_dev(Wg), to_dev(Wu), to_dev(Wd), "bf16")
    y, ws = moe.moe_layer_forward(to_dev(x), to_dev(lg), w.E, w.k, w.e0, pw)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    ref = oracle.moe_forward(x, "bf16", lg, w.d, w.f, w.E, w.k, w.e0, w.E_loc, Wg, Wu, Wd, "bf16")
    assert rel_l2(to_np(y), ref) <= TOL["bf16"]
