"""The GPU parity checker's routing rule, on the CPU with made-up routings:
expert sets must match exactly, slot order only where neighbouring oracle
choice scores are at least the 1e-6 margin apart."""
import numpy as np
import pytest

from _parity import MARGIN, check_routing, tie_runs
from group_limited_routed_gb300.inputs import CONFIGS

CFG = CONFIGS["tiny"].replace(topk=4, topk_groups=2)


def _routing(c_rows, idx_rows):
    T, E = len(c_rows), CFG.n_experts
    c = np.zeros((T, E), np.float32)
    for t, row in enumerate(c_rows):
        c[t, : len(row)] = row
    idx = np.array(idx_rows, np.int32)
    w = np.full(idx.shape, CFG.routed_scale / idx.shape[1], np.float32)
    return {"c": c, "idx": idx, "w": w, "expert_margin": np.ones(T), "group_margin": np.ones(T)}


def test_tie_runs():
    assert tie_runs([4.0, 3.0, 2.0]) == [(0, 1), (1, 2), (2, 3)]
    assert tie_runs([4.0, 4.0 - MARGIN / 4, 2.0]) == [(0, 2), (2, 3)]


def test_order_inside_a_near_tie_may_differ_but_sets_may_not():
    # experts 0..3 in group 0 (8 experts per group); 1 and 2 nearly tied
    c = [0.9, 0.5 + 1e-7, 0.5, 0.1]
    r = _routing([c], [[0, 1, 2, 3]])
    check_routing(CFG, np.array([[0, 2, 1, 3]]), r["w"], r)        # swap inside the tie
    with pytest.raises(AssertionError):
        check_routing(CFG, np.array([[1, 0, 2, 3]]), r["w"], r)    # swap across a real margin
    with pytest.raises(AssertionError):
        check_routing(CFG, np.array([[0, 1, 2, 4]]), r["w"], r)    # another expert
