"""The layer inside a CUDA graph: every entry point enqueues on the caller's
stream with no host synchronisation and no allocation, so a forward call can
be captured once and replayed; each replay must equal an eager call bit for
bit (fixed-order sums throughout), including after the inputs change in
place between replays."""
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm up on a side stream (first-call set-up, kernel attributes), then
    capture one call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("name,T", [("tiny", 64), ("tiny", 300), ("decode", 32)])
def test_forward_replays_match_eager(name, T):
    """T = 64 and 32 take the cooperative routing launch, T = 300 the
    separate routing kernels and the 256-token tiles."""
    cfg = inputs.CONFIGS[name].replace(T=T)
    t = inputs.generate(cfg, "cuda")
    ws = pkg.Workspace(cfg, T)
    out = torch.empty(T, cfg.d, dtype=torch.bfloat16, device="cuda")
    x = t["hidden"].clone()

    def call():
        pkg.forward(cfg, x, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"], t["w_down"],
                    out=out, ws=ws, stream=torch.cuda.current_stream())

    g = _capture(call)
    for step in range(3):
        if step:
            x.copy_(inputs.generate(cfg.replace(seed=cfg.seed + 17 * step), "cuda",
                                    weights=False)["hidden"])
        g.replay()
        torch.cuda.synchronize()
        ref = pkg.forward(cfg, x, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                          t["w_down"])
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), step
    assert pkg.check_status(ws) == 0


def test_nvfp4_and_boundary_replays_match_eager():
    cfg = inputs.CONFIGS["tiny"].replace(weight_fmt="nvfp4", seed=31, cpu_generator=True)
    t = inputs.generate(cfg, "cpu")
    t = {k: ({kk: vv.cuda() for kk, vv in v.items()} if isinstance(v, dict)
             else v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    wts = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
    ws = pkg.Workspace(cfg, cfg.T, weight_fmt=pkg.NVFP4)
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: pkg.forward_nvfp4(cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts,
                                           out=out, ws=ws, stream=torch.cuda.current_stream()))
    g.replay()
    torch.cuda.synchronize()
    ref = pkg.forward_nvfp4(cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))

    bcfg = inputs.CONFIGS["tiny"]
    tb = inputs.generate(bcfg, "cuda")
    h0 = torch.randn(bcfg.T, bcfg.d, device="cuda").to(torch.bfloat16)
    gam = torch.ones(bcfg.d, dtype=torch.bfloat16, device="cuda")
    res = h0.clone()
    wsb = pkg.Workspace(bcfg, bcfg.T)
    o2 = torch.empty(bcfg.T, bcfg.d, dtype=torch.bfloat16, device="cuda")
    nx = torch.empty_like(o2)

    def bcall():
        pkg.forward_boundary(bcfg, tb["hidden"], tb["router_w"], tb["corr_bias"], tb["w_gate"],
                             tb["w_up"], tb["w_down"], res, gam, gam, 1e-6, 5, out=o2,
                             next_input=nx, ws=wsb, stream=torch.cuda.current_stream())

    g2 = _capture(bcall)
    res.copy_(h0)
    g2.replay()
    torch.cuda.synchronize()
    res_ref = h0.clone()
    o_ref, nx_ref = pkg.forward_boundary(bcfg, tb["hidden"], tb["router_w"], tb["corr_bias"],
                                         tb["w_gate"], tb["w_up"], tb["w_down"], res_ref, gam,
                                         gam, 1e-6, 5)
    for a, b in ((o2, o_ref), (res, res_ref), (nx, nx_ref)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_replays_match_eager():
    """Both token-block widths: 64 tokens (16-row blocks) and 300 (256-row
    blocks with the gathered token codes)."""
    for T in (64, 300):
        cfg = inputs.CONFIGS["tiny"].replace(weight_fmt="fp8", T=T, seed=40 + T)
        t = inputs.generate(cfg, "cuda")
        wts = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
        out = torch.empty(T, cfg.d, dtype=torch.bfloat16, device="cuda")
        g = _capture(lambda: pkg.forward_fp8(cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts,
                                             out=out, ws=ws, stream=torch.cuda.current_stream()))
        g.replay()
        torch.cuda.synchronize()
        ref = pkg.forward_fp8(cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), T
        assert pkg.check_status(ws) == 0
