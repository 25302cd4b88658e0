"""GPU parity at the full Beam layer sizes (d=5120, 256 experts, d_ff=2560),
in the launch configuration the benchmark times.  Routing is compared on
every token; expert outputs on every token of the decode batch and on a
seeded sample of tokens of the larger batches (the oracle computes them one
by one)."""
import gc

import numpy as np
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import check_logits, check_out, check_routing, exempt_tokens, host, oracle_out, \
    oracle_route

pytestmark = pytest.mark.gpu


def _sample(T, n, seed):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    s = np.sort(rng.choice(T, n - 2, replace=False))
    return np.unique(np.concatenate([[0, T - 1], s]))   # first and last token always


@pytest.mark.parametrize("name,n_sample", [("decode", 32), ("prefill", 8), ("skewed", 8)])
def test_beam_config_parity(name, n_sample):
    cfg = inputs.CONFIGS[name]
    t = inputs.generate(cfg, "cuda")
    try:
        lg, r = oracle_route(cfg, t)
        ws = pkg.Workspace(cfg, cfg.T)
        idx, w, logits = pkg.route(cfg, t["hidden"], t["router_w"], t["corr_bias"], ws=ws,
                                   want_logits=True)
        check_logits(host(logits), lg)
        check_routing(cfg, host(idx), host(w), r)
        out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"],
                          t["w_up"], t["w_down"], ws=ws)
        assert pkg.check_status(ws) == 0
        rows = _sample(cfg.T, n_sample, seed=len(name))
        rows = rows[~exempt_tokens(r)[rows]]
        ref = oracle_out(cfg, t, r["idx"], r["w"], tokens=rows)
        err, rms, same = check_out(out, ref, rows=rows)
        print(f"{name}: {len(rows)} tokens, max|err| {err:.3e}, RMS {rms:.3e}, "
              f"bit-identical {same:.4f}")
        if name == "skewed":
            counts = np.bincount(host(idx).reshape(-1), minlength=cfg.n_experts)
            assert counts.max() > cfg.T // 2       # a few experts take most tokens
    finally:
        del t
        gc.collect()
        torch.cuda.empty_cache()


def test_beam_largest_batch():
    """65536 tokens (524288 token rows, 2048 per expert): row offsets past
    2^31 elements in the FP32 expert outputs, the counting sort over 512
    chunks, 40960 GEMM tiles.  Routing on every token, outputs on a sample
    that includes the first and last tokens."""
    cfg = inputs.CONFIGS["prefill"].replace(T=65536, seed=21)
    t = inputs.generate(cfg, "cuda")
    try:
        lg, r = oracle_route(cfg, t)
        ws = pkg.Workspace(cfg, cfg.T)
        out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"],
                          t["w_up"], t["w_down"], ws=ws)
        assert pkg.check_status(ws) == 0
        idx = host(ws.view("topk_idx", torch.int32, (cfg.T, cfg.topk)))
        w = host(ws.view("topk_w", torch.float32, (cfg.T, cfg.topk)))
        check_routing(cfg, idx, w, r)
        rows = _sample(cfg.T, 8, seed=3)
        rows = rows[~exempt_tokens(r)[rows]]
        err, rms, same = check_out(out, oracle_out(cfg, t, r["idx"], r["w"], tokens=rows),
                                   rows=rows)
        print(f"T=65536: {len(rows)} tokens, max|err| {err:.3e}, RMS {rms:.3e}")
    finally:
        del t
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [256, 640, 1500, 2051])
def test_router_k_splits_at_beam_shapes(T):
    """Batches whose router tiles leave SMs idle split K over CTAs (256 tokens:
    4 tiles, 10 splits of 8 K ranges; 2051: 34 tiles, 4 splits, a ragged last
    tile) and the selection adds the partials: logits and routing still meet
    the FP32 bounds on every token."""
    cfg = inputs.CONFIGS["prefill"].replace(T=T, seed=300 + T)
    t = inputs.generate(cfg, "cuda", weights=False)
    lg, r = oracle_route(cfg, t)
    idx, w, logits = pkg.route(cfg, t["hidden"], t["router_w"], t["corr_bias"], want_logits=True)
    check_logits(host(logits), lg)
    check_routing(cfg, host(idx), host(w), r)
