"""The GPU parity checker's host logic, on the CPU with made-up routings:
expert sets must match exactly, slot order only where neighbouring oracle
choice scores are at least the 1e-6 margin apart; a near-tie token is
compared on the oracle's alternative routing for the set the GPU chose; the
output sample of a large batch reaches every expert's last token block."""
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


def test_near_tie_token_is_compared_on_the_gpus_valid_alternative():
    """A token whose k-th and (k+1)-th choice scores are 2e-7 apart: a GPU
    that took the (k+1)-th expert is compared on the oracle's routing for
    that set (weights from the oracle's own scores); a set outside the tie
    fails; a token routed like the oracle keeps the oracle's routing."""
    import oracle
    from _parity import output_routing
    cfg = CONFIGS["tiny"]
    E = cfg.n_experts
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((2, E)).astype(np.float32)
    r = oracle.route(lg, np.zeros(E, np.float32), cfg.n_groups, cfg.topk_groups, cfg.topk,
                     cfg.routed_scale)
    # bias the token-0 scores so that the best unchosen candidate sits 2e-7
    # below the k-th chosen one
    c = r["c"][0].astype(np.float64)
    kth = r["idx"][0, -1]
    cand = [e for e in range(E) if r["keep"][0, e // (E // cfg.n_groups)]
            and e not in r["idx"][0]]
    nxt = max(cand, key=lambda e: c[e])
    bias = np.zeros((E,), np.float32)
    bias[nxt] = np.float32(c[kth] - c[nxt] - 2e-7)
    r = oracle.route(lg, bias, cfg.n_groups, cfg.topk_groups, cfg.topk, cfg.routed_scale)
    assert r["expert_margin"][0] < MARGIN and nxt not in r["idx"][0]
    gpu = r["idx"].copy()
    gpu[0, -1] = nxt
    idx, w = output_routing(cfg, r, gpu)
    assert set(idx[0].tolist()) == set(gpu[0].tolist())
    assert abs(float(w[0].sum()) - cfg.routed_scale) < 1e-5
    assert np.array_equal(idx[1], r["idx"][1]) and np.array_equal(w[1], r["w"][1])
    bad = r["idx"].copy()
    bad[0, -1] = min(cand, key=lambda e: c[e])          # far below the cut
    if bad[0, -1] != nxt:
        with pytest.raises(AssertionError):
            output_routing(cfg, r, bad)


def test_block_sample_reaches_every_experts_last_block():
    from _parity import block_sample
    cfg = CONFIGS["tiny"]
    rng = np.random.default_rng(0)
    T, k, E = 3000, cfg.topk, cfg.n_experts
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    rows = block_sample(cfg, idx, 200, seed=1, nt=256)
    assert len(rows) >= 200 and rows[0] == 0 and rows[-1] == T - 1
    assert np.all(np.diff(rows) > 0)
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    starts = np.concatenate([[0], np.cumsum(counts)])
    chosen = set(rows.tolist())
    for e in range(E):
        c = counts[e]
        nb = -(-c // 256)
        bs = min(256, (-(-c // nb) + 15) // 16 * 16)
        last = [int(order[starts[e] + p]) // k for p in range((nb - 1) * bs, c)]
        assert chosen & set(last), e              # a row of the last (ragged) block
        assert int(order[starts[e] + c - 1]) // k in chosen
