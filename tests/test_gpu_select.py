"""The group-limited selection runs with a block per token below 256 tokens
and with a warp per token from 256 on.  Both follow one rule (scores desc,
lower index first among equals, for groups and experts alike), so on the same
logits they must give the same indices and the same weights bit for bit; and
both must match the oracle's selection.  Logits and biases are drawn from a
few values so that ties are everywhere."""
import numpy as np
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs
import oracle

from _parity import W_RTOL_SELECT, check_routing, host

pytestmark = pytest.mark.gpu

SHAPES = [(64, 8, 4, 8), (256, 8, 4, 8), (256, 128, 16, 8), (256, 16, 4, 32), (96, 3, 2, 4),
          (32, 16, 3, 5), (64, 2, 1, 6)]


def _cfg(E, G, kg, k, T):
    return inputs.MoEConfig(name="sel", T=T, d=128, d_ff=128, n_experts=E, n_groups=G,
                            topk_groups=kg, topk=k, routed_scale=2.5)


def _tied_inputs(T, E, seed, levels):
    rng = np.random.default_rng(seed)
    lg = rng.choice(np.linspace(-3, 3, levels).astype(np.float32), size=(T, E))
    bias = rng.choice(np.float32([-0.05, 0.0, 0.03]), size=E).astype(np.float32)
    return lg.astype(np.float32), bias


@pytest.mark.parametrize("E,G,kg,k", SHAPES)
def test_block_and_warp_selection_agree_bitwise(E, G, kg, k):
    lg, bias = _tied_inputs(256, E, seed=E + 7 * G + k, levels=5)
    b = torch.from_numpy(bias).cuda()
    idx_w, w_w = pkg.select(_cfg(E, G, kg, k, 256), torch.from_numpy(lg).cuda(), b)
    idx_b, w_b = pkg.select(_cfg(E, G, kg, k, 255), torch.from_numpy(lg[:255]).cuda(), b)
    assert torch.equal(idx_w[:255], idx_b)
    assert torch.equal(w_w[:255].view(torch.int32), w_b.view(torch.int32))


@pytest.mark.parametrize("E,G,kg,k", SHAPES)
def test_warp_selection_matches_oracle(E, G, kg, k):
    """Continuous logits (the oracle's FP64 sigmoid and the GPU's FP32 one may
    round apart, so exact ties are left to the bitwise test above): indices
    exact except where a margin is below 1e-6, weights within 1e-6."""
    T = 700
    rng = np.random.default_rng(3 * E + G)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    bias = rng.uniform(-0.05, 0.05, E).astype(np.float32)
    cfg = _cfg(E, G, kg, k, T)
    idx, w = pkg.select(cfg, torch.from_numpy(lg).cuda(), torch.from_numpy(bias).cuda())
    r = oracle.route(lg, bias, G, kg, k, 2.5)
    check_routing(cfg, host(idx), host(w), r, w_rtol=W_RTOL_SELECT)


def test_all_equal_scores_follow_the_tie_rule_at_300_tokens():
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cuda", T=300)
    idx, w = pkg.route(cfg, t["hidden"], torch.zeros_like(t["router_w"]),
                       torch.zeros_like(t["corr_bias"]))
    assert np.array_equal(host(idx), np.tile(np.arange(8), (300, 1)))
    assert np.all(host(w) == np.float32(2.5 / 8))
