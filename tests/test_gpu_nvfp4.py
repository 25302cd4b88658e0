"""GPU parity of the NVFP4 expert path against the CPU oracle: the scale
packing (exact), the quantised token rows (bit-exact: both sides take the
same FP32 decisions), and the layer output within the NVFP4 bound
(max-abs 2e-2 * RMS(out), read like the BF16 bound: arithmetic error
against the oracle's exact output, plus the BF16 output's half step)."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import block_sample, check_out, check_routing, gpu_routing, host, oracle_route, \
    output_routing

pytestmark = pytest.mark.gpu
FP4_TOL = 2e-2
TINY = inputs.CONFIGS["tiny"].replace(name="tiny_fp4", weight_fmt="nvfp4", seed=7)


def _nt(cfg, T):
    # token-block width of the NVFP4 and W4A16 GEMMs at this batch
    return 16 if T * cfg.topk <= 4 * cfg.n_experts else 32


def _weights(t, stream=None):
    return [pkg.Fp4Weight.of(t[n], stream) for n in ("w_gate", "w_up", "w_down")]


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


def _oracle_fp4(cfg, t, r, tokens=None, gpu_idx=None):
    """The oracle's NVFP4 layer on `tokens` (all by default); with gpu_idx,
    near-tie tokens the GPU routed to another valid set take the oracle's
    matching alternative routing."""
    if gpu_idx is not None:
        idx, w = output_routing(cfg, r, gpu_idx, tokens)
        r = dict(r, idx=idx, w=w)
    rows = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)})
    proj = {}
    for n in ("w_gate", "w_up", "w_down"):
        proj[n] = {"q": {e: host(t[n]["q"][e]) for e in need},
                   "sf": {e: host(t[n]["sf"][e]) for e in need},
                   "gs": host(t[n]["gs"])}
    return oracle.experts_nvfp4(host(t["hidden"]), r["idx"], r["w"], proj["w_gate"], proj["w_up"],
                                proj["w_down"], cfg.n_experts, act_quant=True,
                                tokens=None if tokens is None else rows, exact=True)


def test_pack_scales_matches_the_blocked_order():
    rows, S = 256, 40
    g = torch.Generator().manual_seed(3)
    sf = torch.randint(0, 256, (rows, S), generator=g, dtype=torch.uint8)
    got = host(pkg.pack_scales(sf.cuda())).reshape(-1)
    ref = np.zeros(rows * S, np.uint8)
    src = sf.numpy()
    for row in range(rows):
        for s in range(S):
            blk = (row // 128) * (S // 4) + s // 4
            r = row % 128
            ref[blk * 512 + (r % 32) * 16 + (r // 32) * 4 + s % 4] = src[row, s]
    assert np.array_equal(got, ref)


@pytest.fixture(scope="module")
def tiny_fp4():
    t = _to(inputs.generate(TINY.replace(cpu_generator=True), "cpu"), "cuda")
    lg, r = oracle_route(TINY, t)
    return t, lg, r


def test_quantised_token_rows_are_bit_exact(tiny_fp4):
    t, lg, r = tiny_fp4
    cfg = TINY
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.NVFP4)
    pkg.forward_nvfp4(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    TK = cfg.T * cfg.topk
    perm = host(ws.view("perm_src", torch.int32, (TK,)))
    xq = host(ws.view("x_fp4", torch.uint8, (TK, cfg.d // 2)))
    # 16-byte slot per 64 elements: the 4 scales, then padding
    xsf = host(ws.view("x_sf", torch.uint8, (TK, cfg.d // 64, 16)))[:, :, :4].reshape(TK, -1)
    x = t["hidden"].float().cpu().numpy()
    dec = np.array([oracle.e2m1_value(c) for c in range(16)])
    for row in range(TK):
        q, sf = oracle.nvfp4_quantize(x[perm[row] // cfg.topk])
        assert np.array_equal(xsf[row], sf), row
        a = np.stack([xq[row] & 15, xq[row] >> 4], 1).reshape(-1)
        b = np.stack([q & 15, q >> 4], 1).reshape(-1)
        assert np.array_equal(dec[a], dec[b]), row        # +0 / -0 decode alike


def test_nvfp4_forward_matches_oracle(tiny_fp4):
    t, lg, r = tiny_fp4
    ws = pkg.Workspace(TINY, TINY.T, weight_fmt=pkg.NVFP4)
    out = pkg.forward_nvfp4(TINY, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t),
                            ws=ws)
    ref = _oracle_fp4(TINY, t, r, gpu_idx=gpu_routing(ws, TINY, TINY.T))
    check_out(out, ref, tol=FP4_TOL)


@pytest.mark.parametrize("T", [1, 37, 300])
def test_nvfp4_ragged_and_wide_token_blocks(T):
    """300 tokens take the 32-row token blocks."""
    cfg = TINY.replace(T=T, seed=60 + T)
    t = _to(inputs.generate(cfg.replace(cpu_generator=True), "cpu"), "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, T, weight_fmt=pkg.NVFP4)
    out = pkg.forward_nvfp4(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    rows = block_sample(cfg, r["idx"], 96, seed=T, nt=_nt(cfg, T))
    check_out(out, _oracle_fp4(cfg, t, r, tokens=rows, gpu_idx=gpu_routing(ws, cfg, T)),
              rows=rows, tol=FP4_TOL)


def test_nvfp4_beam_workload():
    cfg = inputs.CONFIGS["nvfp4"]
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.NVFP4)
    out = pkg.forward_nvfp4(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t), ws=ws)
    assert pkg.check_status(ws) == 0
    idx = host(ws.view("topk_idx", torch.int32, (cfg.T, cfg.topk)))
    w = host(ws.view("topk_w", torch.float32, (cfg.T, cfg.topk)))
    check_routing(cfg, idx, w, r)
    err, rms, same = check_out(out, _oracle_fp4(cfg, t, r, gpu_idx=idx), tol=FP4_TOL)
    print(f"nvfp4 beam: all {cfg.T} tokens, max|err| {err:.3e}, RMS {rms:.3e}")


# ----------------------------------------------- W4A16 (NVFP4 weights, F16 activations)
A16_TOL = 1e-2


def _oracle_a16(cfg, t, r, tokens=None, gpu_idx=None):
    if gpu_idx is not None:
        idx, w = output_routing(cfg, r, gpu_idx, tokens)
        r = dict(r, idx=idx, w=w)
    rows = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)})
    proj = {}
    for n in ("w_gate", "w_up", "w_down"):
        proj[n] = {"q": {e: host(t[n]["q"][e]) for e in need},
                   "sf": {e: host(t[n]["sf"][e]) for e in need},
                   "gs": host(t[n]["gs"])}
    return oracle.experts_nvfp4(host(t["hidden"]), r["idx"], r["w"], proj["w_gate"], proj["w_up"],
                                proj["w_down"], cfg.n_experts, act_quant=oracle.ACT_F16,
                                tokens=None if tokens is None else rows, exact=True)


@pytest.mark.parametrize("T", [64, 1, 37, 300])
def test_w4a16_forward_matches_oracle(T):
    """16 and 32-row token blocks (300 tokens); the BF16 output tolerance:
    activations are not quantised."""
    cfg = TINY.replace(T=T, seed=80 + T)
    t = _to(inputs.generate(cfg.replace(cpu_generator=True), "cpu"), "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.NVFP4_A16)
    out = pkg.forward_nvfp4_a16(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t),
                                ws=ws)
    assert pkg.check_status(ws) == 0
    rows = block_sample(cfg, r["idx"], 96, seed=T, nt=_nt(cfg, T))
    err, rms, same = check_out(out, _oracle_a16(cfg, t, r, tokens=rows,
                                                gpu_idx=gpu_routing(ws, cfg, T)),
                               rows=rows, tol=A16_TOL)
    print(f"w4a16 T={T}: max|err| {err:.3e}, RMS {rms:.3e}, identical {same:.3f}")


def test_w4a16_beam_workload():
    cfg = inputs.CONFIGS["nvfp4"]
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.NVFP4_A16)
    out = pkg.forward_nvfp4_a16(cfg, t["hidden"], t["router_w"], t["corr_bias"], *_weights(t),
                                ws=ws)
    assert pkg.check_status(ws) == 0
    idx = gpu_routing(ws, cfg, cfg.T)
    w = host(ws.view("topk_w", torch.float32, (cfg.T, cfg.topk)))
    check_routing(cfg, idx, w, r)
    err, rms, same = check_out(out, _oracle_a16(cfg, t, r, gpu_idx=idx), tol=A16_TOL)
    print(f"w4a16 beam: all {cfg.T} tokens, max|err| {err:.3e}, RMS {rms:.3e}")
