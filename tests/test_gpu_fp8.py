"""GPU parity of the dynamic FP8 expert path against the CPU oracle: the
per-row E4M3 quantisation of BF16 rows (bit-exact: both sides take the same
FP32 decisions), the quantised token rows inside a layer call, and the layer
output against the oracle's exact output (plus the BF16 output's half step).

Output bound.  The token codes are bit-exact; an h code differs only where
the GPU's h (FP32 accumulation in the tensor cores' order) and the oracle's
(FP64) round to BF16 on opposite sides of a boundary and that moves the E4M3
code: a near tie, both codes being correct roundings.  Such a flip changes
one h element by one E4M3 step, at most 32 * scale = amax / 14 of its row,
and so every output element of the token by w * (amax / 14) * W_d[i, f].
With the Beam draws (h amax up to about 20, w up to about 0.5, |W_d| up to
4 * 0.02) that is below 4e-2 * RMS(out).  So: 99 % of the elements within
the BF16 path's 1e-2 * RMS, and all within 4e-2 * RMS."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import check_out, check_routing, exempt_tokens, half_ulp_bf16, host, oracle_route

pytestmark = pytest.mark.gpu
FP8_TOL = 1e-2         # the BF16 path's bound, for 99 % of the elements
FP8_FLIP_TOL = 4e-2    # every element: one flipped h code at the row's largest value
FP8_WITHIN = 0.99


def check_fp8_out(out, ref, rows=None):
    err, rms, same = check_out(out, ref, rows=rows, tol=FP8_FLIP_TOL)
    bits, exact = ref
    g = out.double().cpu().numpy()
    if rows is not None:
        g, exact = g[rows], exact[rows]
    if g.size:
        inside = np.abs(g - exact) <= FP8_TOL * rms + half_ulp_bf16(exact)
        print(f"  within {FP8_TOL} * RMS: {inside.mean():.5f} of the elements")
        assert inside.mean() >= FP8_WITHIN
    return err, rms, same


TINY = inputs.CONFIGS["tiny"].replace(name="tiny_fp8", weight_fmt="fp8", seed=12)


def _weights(t):
    return [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]


def _to(t, dev):
    out = {}
    for k, v in t.items():
        if isinstance(v, dict):
            out[k] = {kk: vv.to(dev) for kk, vv in v.items()}
        elif isinstance(v, torch.Tensor):
            out[k] = v.to(dev)
        else:
            out[k] = v
    return out


def _oracle_fp8(cfg, t, r, tokens=None):
    rows = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)})
    proj = {}
    for n in ("w_gate", "w_up", "w_down"):
        proj[n] = {"q": {e: host(t[n]["q"][e]) for e in need},
                   "s": {e: host(t[n]["s"][e]) for e in need}}
    return oracle.experts_fp8(host(t["hidden"]), r["idx"], r["w"], proj["w_gate"], proj["w_up"],
                              proj["w_down"], cfg.n_experts, act_quant=True,
                              tokens=None if tokens is None else rows, exact=True)


@pytest.mark.parametrize("n,cols", [(67, 8), (67, 2560), (67, 5120), (2051, 40), (2051, 2560),
                                    (2051, 3072)])
def test_row_quantiser_is_bit_exact(n, cols):
    """One block per row (67 rows, or rows longer than 3072 values) and one
    warp per row (2051 rows of up to 3072: a ragged last block of four)."""
    g = torch.Generator().manual_seed(5)
    mag = torch.exp(torch.empty(n, 1).uniform_(-14, 8, generator=g))
    x = (torch.randn(n, cols, generator=g) * mag)
    x[5] = 0.0                                     # scale 1, all codes 0
    x[6, ::2] = -0.0
    x[7, :] = 1.0
    x[7, 3] = 448.0                                # scale exactly 1
    x[8, :] = 2.0 ** -30                           # tiny values, subnormal codes after scaling
    x[8, 0] = 2.0 ** -20
    xb = x.to(torch.bfloat16)
    q, sc = pkg.fp8_quantize_rows(xb.cuda())
    q_ref, sc_ref = oracle.fp8_quantize_rows(inputs.bf16_bits(xb))
    assert np.array_equal(host(sc), sc_ref)
    assert np.array_equal(host(q), q_ref)


@pytest.fixture(scope="module")
def tiny_fp8():
    t = _to(inputs.generate(TINY.replace(cpu_generator=True), "cpu"), "cuda")
    lg, r = oracle_route(TINY, t)
    return t, lg, r


def test_quantised_token_rows_in_the_layer_are_bit_exact(tiny_fp8):
    t, lg, r = tiny_fp8
    cfg = TINY
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.FP8)
    pkg.forward_fp8(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    xq = host(ws.view("x_fp8", torch.uint8, (cfg.T, cfg.d)))
    xs = host(ws.view("x_scale", torch.float32, (cfg.T,)))
    q_ref, s_ref = oracle.fp8_quantize_rows(host(t["hidden"]))
    assert np.array_equal(xq, q_ref) and np.array_equal(xs, s_ref)


def test_fp8_forward_matches_oracle(tiny_fp8):
    t, lg, r = tiny_fp8
    ws = pkg.Workspace(TINY, TINY.T, weight_fmt=pkg.FP8)
    out = pkg.forward_fp8(TINY, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    idx = host(ws.view("topk_idx", torch.int32, (TINY.T, TINY.topk)))
    w = host(ws.view("topk_w", torch.float32, (TINY.T, TINY.topk)))
    check_routing(TINY, idx, w, r)
    err, rms, same = check_fp8_out(out, _oracle_fp8(TINY, t, r), rows=~exempt_tokens(r))
    print(f"fp8 tiny: max|err| {err:.3e}, RMS {rms:.3e}, identical {same:.3f}")


@pytest.mark.parametrize("T", [1, 37, 300])
def test_fp8_ragged_and_wide_token_blocks(T):
    """300 tokens (2400 rows over 64 experts) take the 256-row token blocks,
    the gathered token codes and the paired down tiles."""
    cfg = TINY.replace(T=T, seed=80 + T)
    t = _to(inputs.generate(cfg.replace(cpu_generator=True), "cpu"), "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
    out = pkg.forward_fp8(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    rows = np.nonzero(~exempt_tokens(r))[0][:48]
    check_fp8_out(out, _oracle_fp8(cfg, t, r, tokens=rows), rows=rows)


@pytest.mark.parametrize("name,T", [("fp8", None), ("fp8_prefill", 2048)])
def test_fp8_beam_workloads(name, T):
    """Beam shapes: the decode batch (16-row token blocks, rows gathered in
    the GEMM) and a 2048-token batch (256-row blocks), sampled tokens."""
    cfg = inputs.CONFIGS[name]
    cfg = cfg if T is None else cfg.replace(T=T)
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.FP8)
    out = pkg.forward_fp8(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    idx = host(ws.view("topk_idx", torch.int32, (cfg.T, cfg.topk)))
    w = host(ws.view("topk_w", torch.float32, (cfg.T, cfg.topk)))
    check_routing(cfg, idx, w, r)
    rng = np.random.default_rng(13)
    rows = np.sort(rng.choice(cfg.T, 12, replace=False))
    rows = rows[~exempt_tokens(r)[rows]]
    err, rms, same = check_fp8_out(out, _oracle_fp8(cfg, t, r, tokens=rows), rows=rows)
    print(f"{name} T={cfg.T}: {len(rows)} tokens, max|err| {err:.3e}, RMS {rms:.3e}")
