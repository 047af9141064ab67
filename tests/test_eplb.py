"""Expert placement / replication plan (host code, no GPU): the oracle against hand-derived
plans, the mathematics of its replication step and its invariants; the library's
moe_eplb_plan against the oracle."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle.eplb import eplb_plan

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    with open(os.path.join(HERE, "golden", "eplb_examples.json")) as fh:
        return json.load(fh)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: str(c["load"]))
def test_oracle_matches_hand_derived_plans(case):
    slot, rep, gl = eplb_plan(case["load"], case["G"], case["S"])
    assert slot == case["slot_expert"]
    assert rep == case["replicas"]
    assert [float(v) for v in gl] == [float(v) for v in case["gpu_load"]]


def _instances(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        G = int(rng.integers(1, 6))
        S = int(rng.integers(1, 5))
        E = int(rng.integers(1, G * S + 1))
        kind = rng.integers(3)
        if kind == 0:
            load = rng.integers(0, 50, E)
        elif kind == 1:  # Zipf-like skew
            load = (1000.0 / np.arange(1, E + 1) ** 1.1).astype(np.int64)[rng.permutation(E)]
        else:  # ties everywhere
            load = np.full(E, int(rng.integers(0, 5)))
        yield [int(v) for v in load], G, S


def test_oracle_invariants():
    for load, G, S in _instances(300, 1):
        E = len(load)
        slot, rep, gl = eplb_plan(load, G, S)
        flat = [e for row in slot for e in row if e >= 0]
        assert sorted(set(flat)) == list(range(E))                     # every expert placed
        assert all(1 <= rep[e] <= G for e in range(E))
        assert [flat.count(e) for e in range(E)] == rep
        for row in slot:
            es = [e for e in row if e >= 0]
            assert len(es) == len(set(es)) and len(row) == S             # one copy per GPU at most
            assert row[len(es):] == [-1] * (S - len(es))                 # filled from slot 0 up
        assert sum(gl, Fraction(0)) == sum(load)                          # load conserved exactly
        if G * S == E:
            assert rep == [1] * E


def test_replication_step_minimises_the_largest_load_per_copy():
    """Brute force over every copy vector (1..G copies each, sum = slots or all at G): the
    greedy's largest load per copy is the minimum achievable."""
    checked = 0
    for load, G, S in _instances(150, 2):
        E = len(load)
        if E > 5:
            continue
        _, rep, _ = eplb_plan(load, G, S)
        target = min(G * S, E * G)
        best = None
        for vec in itertools.product(range(1, G + 1), repeat=E):
            if sum(vec) != target:
                continue
            worst = max(Fraction(load[e], vec[e]) for e in range(E))
            best = worst if best is None else min(best, worst)
        got = max(Fraction(load[e], rep[e]) for e in range(E))
        # copies the placement dropped only happen when no GPU could take them
        if sum(rep) == target:
            assert got == best
            checked += 1
    assert checked >= 40


def test_uniform_load_balances_exactly():
    for G, S in [(2, 2), (4, 3), (8, 4)]:
        slot, rep, gl = eplb_plan([7] * (G * S), G, S)
        assert rep == [1] * (G * S)
        assert all(v == 7 * S for v in gl)


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_103_b300 import build
    build.build()
    import mixture_experts_layer_103_b300 as m
    return m


def test_library_matches_oracle(moe):
    n = 0
    for load, G, S in _instances(400, 3):
        slot, rep, gl = moe.moe_eplb_plan(load, G, S)
        oslot, orep, ogl = eplb_plan(load, G, S)
        assert slot.tolist() == oslot, (load, G, S)
        assert rep.tolist() == orep
        np.testing.assert_allclose(gl, [float(v) for v in ogl], rtol=1e-12, atol=1e-9)
        n += 1
    assert n == 400


def test_library_validation(moe):
    import ctypes
    L = moe.lib()
    P = ctypes.c_void_p(256)
    assert L.moe_eplb_plan(None, 4, 2, 2, P, P, P) == 1
    assert L.moe_eplb_plan(P, 5, 2, 2, P, P, P) == 1     # E > G * S
    assert L.moe_eplb_plan(P, 0, 2, 2, P, P, P) == 1
    with pytest.raises(RuntimeError):
        moe.moe_eplb_plan([3, -1], 2, 1)                  # negative load
