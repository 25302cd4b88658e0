"""GPU parity of the expert-parallel entry points.  The R ranks are run one
after another on one GPU, and the all-to-all is done on the host side by
slicing and concatenating device tensors (no kernel waits for another
rank).  The layer's per-row arithmetic does not depend on which rows share
a tile, so R ranks must reproduce beam_moe_forward bit for bit; the output
is also checked against the oracle."""
import numpy as np
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import ep, inputs

from _parity import check_out, gpu_routing, oracle_out, oracle_route, output_routing

pytestmark = pytest.mark.gpu


def _bf16_experts(cfg, t):
    def run(R, q, x, e, w):
        sl = ep.expert_slice(cfg, R, q)
        return pkg.ep_experts(cfg, R, q, x, e, w, t["w_gate"][sl], t["w_up"][sl], t["w_down"][sl])
    return run


def _emulate(cfg, t, Ts, experts=None):
    """Every rank's input rows, its output of the expert-parallel layer (ranks
    in sequence) and the expert indices the ranks' routing chose, in token
    order."""
    experts = _bf16_experts(cfg, t) if experts is None else experts
    R = len(Ts)
    starts = np.concatenate([[0], np.cumsum(Ts)])
    hid = [t["hidden"][starts[r]:starts[r + 1]] for r in range(R)]
    disp = [pkg.ep_dispatch(cfg, h, t["router_w"], t["corr_bias"], R) for h in hid]
    counts = [d[3].cpu().numpy() for d in disp]                 # [src][dst]
    offs = [np.concatenate([[0], np.cumsum(c)]) for c in counts]
    y_recv = []
    for q in range(R):
        parts = [(disp[r][0][offs[r][q]:offs[r][q + 1]], disp[r][1][offs[r][q]:offs[r][q + 1]],
                  disp[r][2][offs[r][q]:offs[r][q + 1]]) for r in range(R)]
        x = torch.cat([p[0] for p in parts]).contiguous()
        e = torch.cat([p[1] for p in parts]).contiguous()
        w = torch.cat([p[2] for p in parts]).contiguous()
        y_recv.append(experts(R, q, x, e, w))
    outs, routing = [], []
    for r in range(R):
        # rows come back per destination rank, in the order they were sent
        back = []
        for q in range(R):
            first = sum(int(counts[s][q]) for s in range(r))
            back.append(y_recv[q][first:first + int(counts[r][q])])
        y_back = torch.cat(back).contiguous() if back else None
        ws = disp[r][4]
        outs.append(pkg.ep_combine(cfg, y_back, Ts[r], ws))
        assert pkg.check_status(ws) == 0
        routing.append(gpu_routing(ws, cfg, Ts[r]))
    return hid, outs, np.concatenate(routing)


@pytest.mark.parametrize("Ts", [[40, 24], [16, 0, 33, 5], [9, 1, 0, 30, 7, 12, 3, 20]])
def test_emulated_ranks_reproduce_the_layer(Ts):
    cfg = inputs.CONFIGS["tiny"].replace(seed=70 + len(Ts))
    t = inputs.generate(cfg, "cuda", T=sum(Ts))
    hid, outs, gidx = _emulate(cfg, t, Ts)
    for h, o in zip(hid, outs):
        ref = pkg.forward(cfg, h, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                          t["w_down"])
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    # and the oracle on all tokens
    full = torch.cat(outs)
    c2 = cfg.replace(T=sum(Ts))
    lg, r = oracle_route(c2, t)
    check_out(full, oracle_out(c2, t, *output_routing(c2, r, gidx)))


def test_emulated_ranks_beam_decode():
    """Beam shapes, eight ranks of 32 experts, 32 tokens per rank."""
    cfg = inputs.CONFIGS["decode"]
    t = inputs.generate(cfg, "cuda", T=8 * 32)
    hid, outs, _ = _emulate(cfg, t, [32] * 8)
    for h, o in zip(hid, outs):
        ref = pkg.forward(cfg, h, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                          t["w_down"])
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def test_foreign_expert_latches_device_check():
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cuda", T=4)
    R, q = 2, 1
    sl = ep.expert_slice(cfg, R, q)
    x = t["hidden"].repeat_interleave(2, 0).contiguous()
    e = torch.full((8,), sl.start, dtype=torch.int32, device="cuda")
    e[3] = 0                                   # owned by rank 0
    w = torch.full((8,), 0.5, device="cuda")
    ws = pkg.EpWorkspace(cfg, R, 8)
    pkg.ep_experts(cfg, R, q, x, e, w, t["w_gate"][sl], t["w_up"][sl], t["w_down"][sl], ws=ws)
    assert pkg.check_status(ws) == 6


@pytest.mark.parametrize("Ts", [[40, 24], [16, 0, 33, 5]])
def test_emulated_ranks_nvfp4_experts(Ts):
    """NVFP4 experts on each rank (the pages' MegaMoE path runs Beam's NVFP4
    experts): every rank's output equals beam_moe_forward_nvfp4 on its tokens
    bit for bit."""
    cfg = inputs.CONFIGS["tiny"].replace(weight_fmt="nvfp4", seed=90 + len(Ts),
                                         cpu_generator=True)
    t = inputs.generate(cfg, "cpu", T=sum(Ts))
    t = {k: ({kk: vv.cuda() for kk, vv in v.items()} if isinstance(v, dict)
             else v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    full = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
    R = len(Ts)
    local = []
    for q in range(R):
        sl = ep.expert_slice(cfg, R, q)
        local.append([pkg.Fp4Weight.of({k: v[sl] for k, v in t[n].items()})
                      for n in ("w_gate", "w_up", "w_down")])

    def run(R_, q, x, e, w):
        return pkg.ep_experts_nvfp4(cfg, R_, q, x, e, w, *local[q])

    hid, outs, _ = _emulate(cfg, t, Ts, experts=run)
    for h, o in zip(hid, outs):
        if h.shape[0] == 0:
            continue
        ref = pkg.forward_nvfp4(cfg, h.contiguous(), t["router_w"], t["corr_bias"], *full)
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("Ts", [[40, 24], [16, 0, 33, 5]])
def test_emulated_ranks_fp8_experts(Ts):
    """Dynamic FP8 experts on each rank: every received row is quantised with
    its own scale, which is its token's, so every rank's output equals
    beam_moe_forward_fp8 on its tokens bit for bit."""
    cfg = inputs.CONFIGS["tiny"].replace(weight_fmt="fp8", seed=95 + len(Ts), cpu_generator=True)
    t = inputs.generate(cfg, "cpu", T=sum(Ts))
    t = {k: ({kk: vv.cuda() for kk, vv in v.items()} if isinstance(v, dict)
             else v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    full = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
    R = len(Ts)
    local = []
    for q in range(R):
        sl = ep.expert_slice(cfg, R, q)
        local.append([pkg.Fp8Weight(t[n]["q"][sl], t[n]["s"][sl])
                      for n in ("w_gate", "w_up", "w_down")])

    def run(R_, q, x, e, w):
        return pkg.ep_experts_fp8(cfg, R_, q, x, e, w, *local[q])

    hid, outs, _ = _emulate(cfg, t, Ts, experts=run)
    for h, o in zip(hid, outs):
        if h.shape[0] == 0:
            continue
        ref = pkg.forward_fp8(cfg, h.contiguous(), t["router_w"], t["corr_bias"], *full)
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
