"""GPU parity at the smallest layer shapes each expert format accepts: K loops
of one or two blocks in every GEMM (BF16 and FP8 at d = d_ff = 128, NVFP4,
W4A16 and MXFP8 at 256), 32 experts in 4 groups of 8, top-2 groups, top-4, and
ragged token counts on both sides of the 16-row / 256-row block switch
(T * topk > 4 * E from T = 33 on).  Bounds: the BF16 path's 1e-2 * RMS,
NVFP4's 2e-2 * RMS, FP8's 1e-2 * RMS plus the oracle's near-tie slack of
each token (4e-2 * RMS for a token whose row scale sits at a tie), each
against the oracle's exact output plus half a BF16 step.  Every token is
compared, near-tie tokens on the oracle's routing that the GPU chose."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import check_out, check_routing, gpu_routing, host, oracle_out, oracle_route, \
    output_routing

pytestmark = pytest.mark.gpu

SMALL = dict(n_experts=32, n_groups=4, topk_groups=2, topk=4, routed_scale=2.5,
             cpu_generator=True)


def _cfg(fmt, T, d, seed):
    return inputs.MoEConfig(name=f"small_{fmt}", T=T, d=d, d_ff=d, seed=seed,
                            weight_fmt="nvfp4" if fmt == "a16" else fmt, **SMALL)


def _to(t, dev):
    return {k: ({kk: vv.to(dev) for kk, vv in v.items()} if isinstance(v, dict)
                else v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def _proj(t, need, keys):
    return {n: {k: {e: host(t[n][k][e]) for e in need} for k in keys}
            for n in ("w_gate", "w_up", "w_down")}


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4", "a16", "mxfp8"])
@pytest.mark.parametrize("T", [1, 20, 33, 70])
def test_smallest_shapes(fmt, T):
    d = 256 if fmt in ("nvfp4", "a16", "mxfp8") else 128
    cfg = _cfg(fmt, T, d, seed=7 * T + len(fmt))
    t = _to(inputs.generate(cfg, "cpu"), "cuda")
    lg, r = oracle_route(cfg, t)
    x = host(t["hidden"])
    args = (cfg, t["hidden"], t["router_w"], t["corr_bias"])
    if fmt == "bf16":
        ws = pkg.Workspace(cfg, T)
        out = pkg.forward(*args, t["w_gate"], t["w_up"], t["w_down"], ws=ws)
    elif fmt == "fp8":
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
        out = pkg.forward_fp8(*args, *[pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up",
                                                                         "w_down")], ws=ws)
    elif fmt == "mxfp8":
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.MXFP8)
        out = pkg.forward_mxfp8(*args, *[pkg.Mxfp8Weight.of(t[n]) for n in ("w_gate", "w_up",
                                                                             "w_down")], ws=ws)
    else:
        a16 = fmt == "a16"
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.NVFP4_A16 if a16 else pkg.NVFP4)
        wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
        fwd = pkg.forward_nvfp4_a16 if a16 else pkg.forward_nvfp4
        out = fwd(*args, *wts, ws=ws)
    assert pkg.check_status(ws) == 0
    idx = gpu_routing(ws, cfg, T)
    w = host(ws.view("topk_w", torch.float32, (T, cfg.topk)))
    check_routing(cfg, idx, w, r)
    oi, ow = output_routing(cfg, r, idx)
    need = sorted({int(e) for e in oi.reshape(-1)})
    if fmt == "bf16":
        check_out(out, oracle_out(cfg, t, oi, ow))
    elif fmt in ("fp8", "mxfp8"):
        p = _proj(t, need, ("q", "s"))
        fn = oracle.experts_fp8 if fmt == "fp8" else oracle.experts_mxfp8
        bits, exact, slack, scale_tie = fn(
            x, oi, ow, p["w_gate"], p["w_up"], p["w_down"], cfg.n_experts, act_quant=True,
            exact=True, ties=True)
        rms = float(np.sqrt((exact ** 2).mean()))
        rows = np.arange(T)
        check_out(out, (bits, exact), rows=rows[~scale_tie], slack=slack, rms=rms)
        if scale_tie.any():
            check_out(out, (bits, exact), rows=rows[scale_tie], tol=4e-2, rms=rms)
    else:
        p = _proj(t, need, ("q", "sf"))
        for n in p:
            p[n]["gs"] = host(t[n]["gs"])
        ref = oracle.experts_nvfp4(x, oi, ow, p["w_gate"], p["w_up"], p["w_down"],
                                   cfg.n_experts, act_quant=oracle.ACT_F16 if a16 else True,
                                   exact=True)
        check_out(out, ref, tol=1e-2 if a16 else 2e-2)


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4", "a16", "mxfp8"])
def test_repeated_calls_are_bit_identical(fmt):
    """Every reduction runs in a fixed order: two calls on the same inputs
    give the same bits, at both token-block widths (the W4A16 partial sums of
    its four MMA issuers included)."""
    for T in (20, 70):
        d = 256 if fmt in ("nvfp4", "a16", "mxfp8") else 128
        cfg = _cfg(fmt, T, d, seed=3 * T + len(fmt))
        t = _to(inputs.generate(cfg, "cpu"), "cuda")
        args = (cfg, t["hidden"], t["router_w"], t["corr_bias"])
        if fmt == "bf16":
            run = lambda: pkg.forward(*args, t["w_gate"], t["w_up"], t["w_down"])
        elif fmt == "fp8":
            wts = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
            run = lambda: pkg.forward_fp8(*args, *wts)
        elif fmt == "mxfp8":
            wts = [pkg.Mxfp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
            run = lambda: pkg.forward_mxfp8(*args, *wts)
        else:
            wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
            fwd = pkg.forward_nvfp4_a16 if fmt == "a16" else pkg.forward_nvfp4
            run = lambda: fwd(*args, *wts)
        a, b = run(), run()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (fmt, T)
