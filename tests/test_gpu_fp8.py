"""GPU parity of the dynamic FP8 expert path against the CPU oracle: the
per-row E4M3 quantisation of BF16 rows (bit-exact: both sides take the same
FP32 decisions), the quantised token rows inside a layer call, and the layer
output against the oracle's exact output (plus the BF16 output's half step).

Output bound.  The token codes are bit-exact; an h code can differ only where
the GPU's FP32 h (tensor-core accumulation order, fast SiLU) and the
oracle's lie on opposite sides of a BF16 rounding midpoint and the two BF16
values quantise to different E4M3 codes: a near tie, both codes correct.
The oracle lists those itself: every h element within 2^-16 of its value
of a BF16 midpoint, and what taking the other BF16 value would change.  The
bound per output is the BF16 path's 1e-2 * RMS plus the summed effect of its
token's listed ties (usually none).  A token whose row scale itself sits at
such a tie (the amax element) is held to 4e-2 * RMS: one E4M3 step at the
row's largest value, amax / 14, times w and |W_d| stays below that with the
Beam draws (h amax up to about 20, w up to about 0.5, |W_d| up to 4 * 0.02)."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import block_sample, check_out, check_routing, gpu_routing, host, oracle_route, \
    output_routing

pytestmark = pytest.mark.gpu
FP8_TOL = 1e-2             # the BF16 path's bound, plus each token's near-tie slack
FP8_SCALE_TIE_TOL = 4e-2   # tokens whose row scale sits at a tie


def check_fp8_out(out, ref, rows=None):
    """ref = (bits, exact, slack, scale_tie) from the oracle with its near
    ties listed.  Every compared token is held to 1e-2 * RMS + half a BF16
    step + its slack; tokens flagged with a scale tie to 4e-2 * RMS."""
    bits, exact, slack, scale_tie = ref
    rows = np.arange(exact.shape[0]) if rows is None else np.asarray(rows)
    if rows.dtype == bool:
        rows = np.nonzero(rows)[0]
    rms = float(np.sqrt((exact[rows] ** 2).mean())) if rows.size else 0.0
    tight, loose = rows[~scale_tie[rows]], rows[scale_tie[rows]]
    n_slack = int((slack[tight].max(axis=1) > 0).sum()) if tight.size else 0
    print(f"  {n_slack} of {tight.size} tokens carry near-tie slack; {loose.size} scale ties")
    err, _, same = check_out(out, (bits, exact), rows=tight, tol=FP8_TOL, slack=slack, rms=rms)
    if loose.size:
        err = max(err, check_out(out, (bits, exact), rows=loose, tol=FP8_SCALE_TIE_TOL,
                                 rms=rms)[0])
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


def _oracle_fp8(cfg, t, r, tokens=None, gpu_idx=None):
    """The oracle's FP8 layer with its near ties listed, on `tokens` (all by
    default); with gpu_idx, near-tie tokens the GPU routed to another valid
    set take the oracle's matching alternative routing."""
    if gpu_idx is not None:
        idx, w = output_routing(cfg, r, gpu_idx, tokens)
        r = dict(r, idx=idx, w=w)
    rows = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)})
    proj = {}
    for n in ("w_gate", "w_up", "w_down"):
        proj[n] = {"q": {e: host(t[n]["q"][e]) for e in need},
                   "s": {e: host(t[n]["s"][e]) for e in need}}
    return oracle.experts_fp8(host(t["hidden"]), r["idx"], r["w"], proj["w_gate"], proj["w_up"],
                              proj["w_down"], cfg.n_experts, act_quant=True,
                              tokens=None if tokens is None else rows, exact=True, ties=True)


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
    err, rms, same = check_fp8_out(out, _oracle_fp8(TINY, t, r, gpu_idx=idx))
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
    rows = block_sample(cfg, r["idx"], 96, seed=T,
                        nt=16 if T * cfg.topk <= 4 * cfg.n_experts else 256)
    check_fp8_out(out, _oracle_fp8(cfg, t, r, tokens=rows, gpu_idx=gpu_routing(ws, cfg, T)),
                  rows=rows)


@pytest.mark.parametrize("name,T,n_sample", [("fp8", None, 32), ("fp8_prefill", 2048, 512)])
def test_fp8_beam_workloads(name, T, n_sample):
    """Beam shapes: the decode batch (16-row token blocks, rows gathered in
    the GEMM; every token compared) and a 2048-token batch (256-row blocks;
    512 tokens that include every expert's first and last token block)."""
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
    rows = block_sample(cfg, r["idx"], n_sample, seed=13,
                        nt=16 if cfg.T * cfg.topk <= 4 * cfg.n_experts else 256)
    err, rms, same = check_fp8_out(out, _oracle_fp8(cfg, t, r, tokens=rows, gpu_idx=idx),
                                   rows=rows)
    print(f"{name} T={cfg.T}: {len(rows)} tokens, max|err| {err:.3e}, RMS {rms:.3e}")
