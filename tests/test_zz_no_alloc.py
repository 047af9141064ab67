"""moe_permute_noalloc: the permute for callers that cannot allocate device memory when
they run it (a serving engine whose free memory already belongs to its KV-cache pool, a
host recording a CUDA graph).  Its scratch lives in a static device array inside the
library, so it takes no workspace.  It must produce exactly what moe_permute (with a
caller workspace) produces, call after call, and refuse inputs whose scratch would not fit.

This file is collected last so that a stop-at-first-failure run has already run every
other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from synthetic import Workload, gen_logits, gen_x
from moe_testlib import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    assert m.moe_supported()
    return m


def _compare(moe, w, perm_dtype):
    x, lg = gen_x(w), gen_logits(w)
    xd, lgd = to_dev(x), to_dev(lg)
    ids, probs = moe.moe_route_topk(lgd, w.k)
    ref = moe.moe_permute(xd, ids, probs, w.e0, w.E_loc, perm_dtype)
    got = moe.moe_permute_noalloc(xd, ids, probs, w.e0, w.E_loc, perm_dtype)
    torch.cuda.synchronize()
    N = int(ref["offsets"][-1])
    for key in ("counts", "offsets", "pair_to_row"):
        assert torch.equal(got[key], ref[key]), key
    for key in ("row_src_token", "row_prob", "perm_x"):
        assert torch.equal(got[key][:N], ref[key][:N]), key
    if perm_dtype == "mxfp8":
        assert torch.equal(got["perm_x_scale"], ref["perm_x_scale"]) or N == 0 or _sf_equal(ref, got, w, N)
    return N


def _sf_equal(ref, got, w, N):
    from moe_testlib import unpack_act_sf
    off = ref["offsets"].cpu().numpy()
    a = unpack_act_sf(ref["perm_x_scale"].cpu().numpy(), off, w.d, N)
    b = unpack_act_sf(got["perm_x_scale"].cpu().numpy(), off, w.d, N)
    return np.array_equal(a, b)


def test_noalloc_permute_matches_workspace_permute_twice(moe):
    # two calls in a row with different shapes: the static scratch keeps the previous
    # call's contents, which must not leak into the next result
    w1 = Workload("na1", 3000, 256, 32, 64, 8, 0, 64, "bf16", ("normal", 0.5))
    w2 = Workload("na2", 700, 128, 32, 256, 8, 32, 32, "bf16", ("zipf", 1.1))
    assert _compare(moe, w1, "bf16") > 0
    assert _compare(moe, w2, "bf16") > 0


def test_noalloc_permute_mxfp8_twice(moe):
    w = Workload("na3", 513, 256, 32, 16, 4, 4, 8, "bf16")
    _compare(moe, w, "mxfp8")
    _compare(moe, w.replace(seed=1), "mxfp8")


def test_noalloc_permute_rejects_oversized_scratch(moe):
    # ceil(70000/256) * 1024 tile counts need more than the 1 MiB static array
    T, k, E_loc = 70000, 8, 1024
    assert moe.moe_permute_workspace_size(T, k, E_loc) > (1 << 20)
    one = torch.empty(16, dtype=torch.int32, device="cuda")
    p = moe._ptr(one)
    st = moe.lib().moe_permute_noalloc(p, 1, 1, T, 64, p, p, k, 0, E_loc, p, None, p, p, p, p, p, moe._stream())
    assert st == 3  # MOE_ERR_WORKSPACE, nothing launched
