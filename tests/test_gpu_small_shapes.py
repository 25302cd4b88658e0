"""GPU parity at the smallest layer shapes each expert format accepts: K loops
of one or two blocks in every GEMM (BF16 and FP8 at d = d_ff = 128, NVFP4
and W4A16 at 256), 32 experts in 4 groups of 8, top-2 groups, top-4, and
ragged token counts on both sides of the 16-row / 256-row block switch
(T * topk > 4 * E from T = 33 on).  Bounds: the BF16 path's 1e-2 * RMS,
NVFP4's 2e-2 * RMS, FP8's two-part bound (99 % within 1e-2 * RMS, all within
4e-2 * RMS), each against the oracle's exact output plus half a BF16 step."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import check_out, check_routing, exempt_tokens, half_ulp_bf16, host, oracle_out, \
    oracle_route

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


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4", "a16"])
@pytest.mark.parametrize("T", [1, 20, 33, 70])
def test_smallest_shapes(fmt, T):
    d = 256 if fmt in ("nvfp4", "a16") else 128
    cfg = _cfg(fmt, T, d, seed=7 * T + len(fmt))
    t = _to(inputs.generate(cfg, "cpu"), "cuda")
    lg, r = oracle_route(cfg, t)
    rows = np.nonzero(~exempt_tokens(r))[0]
    need = sorted({int(e) for e in r["idx"][rows].reshape(-1)}) if rows.size else []
    x = host(t["hidden"])
    args = (cfg, t["hidden"], t["router_w"], t["corr_bias"])
    if fmt == "bf16":
        ws = pkg.Workspace(cfg, T)
        out = pkg.forward(*args, t["w_gate"], t["w_up"], t["w_down"], ws=ws)
        ref = oracle_out(cfg, t, r["idx"], r["w"], tokens=rows)
        tol, flip = 1e-2, None
    elif fmt == "fp8":
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
        out = pkg.forward_fp8(*args, *[pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up",
                                                                         "w_down")], ws=ws)
        p = _proj(t, need, ("q", "s"))
        ref = oracle.experts_fp8(x, r["idx"], r["w"], p["w_gate"], p["w_up"], p["w_down"],
                                 cfg.n_experts, act_quant=True, tokens=rows, exact=True)
        tol, flip = 1e-2, 4e-2
    else:
        a16 = fmt == "a16"
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.NVFP4_A16 if a16 else pkg.NVFP4)
        wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
        fwd = pkg.forward_nvfp4_a16 if a16 else pkg.forward_nvfp4
        out = fwd(*args, *wts, ws=ws)
        p = _proj(t, need, ("q", "sf"))
        for n in p:
            p[n]["gs"] = host(t[n]["gs"])
        ref = oracle.experts_nvfp4(x, r["idx"], r["w"], p["w_gate"], p["w_up"], p["w_down"],
                                   cfg.n_experts, act_quant=oracle.ACT_F16 if a16 else True,
                                   tokens=rows, exact=True)
        tol, flip = (1e-2 if a16 else 2e-2), None
    assert pkg.check_status(ws) == 0
    idx = host(ws.view("topk_idx", torch.int32, (T, cfg.topk)))
    w = host(ws.view("topk_w", torch.float32, (T, cfg.topk)))
    check_routing(cfg, idx, w, r)
    if flip is None:
        check_out(out, ref, rows=rows, tol=tol)
    else:
        err, rms, _ = check_out(out, ref, rows=rows, tol=flip)
        g = out.double().cpu().numpy()[rows]
        exact = ref[1][rows]
        if g.size:
            inside = np.abs(g - exact) <= tol * rms + half_ulp_bf16(exact)
            assert inside.mean() >= 0.99


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4", "a16"])
def test_repeated_calls_are_bit_identical(fmt):
    """Every reduction runs in a fixed order: two calls on the same inputs
    give the same bits, at both token-block widths (the W4A16 partial sums of
    its four MMA issuers included)."""
    for T in (20, 70):
        d = 256 if fmt in ("nvfp4", "a16") else 128
        cfg = _cfg(fmt, T, d, seed=3 * T + len(fmt))
        t = _to(inputs.generate(cfg, "cpu"), "cuda")
        args = (cfg, t["hidden"], t["router_w"], t["corr_bias"])
        if fmt == "bf16":
            run = lambda: pkg.forward(*args, t["w_gate"], t["w_up"], t["w_down"])
        elif fmt == "fp8":
            wts = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
            run = lambda: pkg.forward_fp8(*args, *wts)
        else:
            wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
            fwd = pkg.forward_nvfp4_a16 if fmt == "a16" else pkg.forward_nvfp4
            run = lambda: fwd(*args, *wts)
        a, b = run(), run()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (fmt, T)
