"""The route comparison rule of the GPU parity tests, on the CPU: a row
whose ids differ from the oracle's passes only when the difference lies
inside the oracle's key gap tolerance, with weights taken from the
oracle's own scores of the chosen set."""
import numpy as np
import pytest

import oracle
from moe_expert_router_02_gb300 import synth
from tests.helpers import PARITY_LOG, check_routes


def _case():
    # row 0: experts 2 and 5 tie at the k / k+1 boundary within 1e-7;
    # row 1: clear gaps everywhere
    lg = np.array([[3.0, 2.0, 1.0, -1.0, -2.0, 1.0 - 1e-7],
                   [3.0, 2.5, 2.0, 1.0, 0.0, -1.0]])
    case = dict(k=3, act=synth.SOFTMAX, bias=None)
    idx, w, keys = oracle.select(lg, 3, synth.SOFTMAX)
    ref = dict(idx=idx, w=w, keys=keys, logits=lg)
    return case, ref


def _weights(lg, ids):
    p = np.exp(lg[ids] - lg.max())
    return (p / p.sum()).astype(np.float32)


def test_identical_routes_pass_and_are_counted():
    case, ref = _case()
    n = len(PARITY_LOG)
    assert check_routes(ref["idx"], ref["w"].astype(np.float32), ref, case, label="t") == 0
    assert PARITY_LOG[n] == ("t", 2, 1, 0)


def test_near_tie_swap_passes_with_its_own_weights():
    case, ref = _case()
    gi = ref["idx"].copy()
    assert list(gi[0]) == [0, 1, 2]
    gi[0, 2] = 5  # the other side of the near tie
    gw = ref["w"].astype(np.float32).copy()
    gw[0] = _weights(ref["logits"][0], gi[0])
    assert check_routes(gi, gw, ref, case, label="swap") == 1


def test_near_tie_row_with_old_weights_fails():
    case, ref = _case()
    gi = ref["idx"].copy()
    gi[0, 2] = 5
    gw = ref["w"].astype(np.float32).copy()
    gw[0] = [0.5, 0.3, 0.2]
    with pytest.raises(AssertionError, match="weight"):
        check_routes(gi, gw, ref, case)


def test_far_expert_on_a_near_tie_row_fails():
    case, ref = _case()
    gi = ref["idx"].copy()
    gi[0, 2] = 4  # key -2, far below the k-th
    gw = ref["w"].astype(np.float32).copy()
    gw[0] = _weights(ref["logits"][0], gi[0])
    with pytest.raises(AssertionError, match="k-th key"):
        check_routes(gi, gw, ref, case)


def test_misordered_slots_fail():
    case, ref = _case()
    gi = ref["idx"].copy()
    gi[0] = [1, 0, 2]  # same set, slots 0 and 1 swapped across a gap of 1
    gw = ref["w"].astype(np.float32).copy()
    gw[0] = _weights(ref["logits"][0], gi[0])
    with pytest.raises(AssertionError, match="misordered"):
        check_routes(gi, gw, ref, case)


def test_changed_set_on_a_clear_row_fails():
    case, ref = _case()
    gi = ref["idx"].copy()
    gi[1, 2] = 3
    gw = ref["w"].astype(np.float32).copy()
    gw[1] = _weights(ref["logits"][1], gi[1])
    with pytest.raises(AssertionError):
        check_routes(gi, gw, ref, case)


def test_repeated_or_out_of_range_experts_fail():
    case, ref = _case()
    for bad in ([0, 0, 1], [0, 1, 6]):
        gi = ref["idx"].copy()
        gi[1] = bad
        with pytest.raises(AssertionError):
            check_routes(gi, ref["w"].astype(np.float32), ref, case)
