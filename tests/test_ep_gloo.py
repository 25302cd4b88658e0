"""The expert-parallel exchange of ``group_limited_routed_gb300.ep`` on CPU
ranks (gloo).  The three library calls are replaced by stand-ins built from
the oracle (this test's own code, CPU only), so what is checked here is the
host logic: split sizes, the order rows travel in and come back in, ranks
without tokens, and that R ranks give exactly the single-rank result."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from group_limited_routed_gb300 import ep, inputs

CFG = inputs.CONFIGS["tiny"].replace(cpu_generator=True, seed=21)


class OracleOps:
    """ep_dispatch / ep_experts / ep_combine on the CPU, from the oracle."""

    def ep_dispatch(self, cfg, hidden, router_w, corr_bias, R):
        x = inputs.bf16_bits(hidden)
        lg = oracle.router_logits(x, router_w.numpy())
        r = oracle.route(lg, corr_bias.numpy(), cfg.n_groups, cfg.topk_groups, cfg.topk,
                         cfg.routed_scale)
        flat = r["idx"].reshape(-1)
        order = np.argsort(flat, kind="stable")          # (expert, token, slot)
        send_x = hidden[torch.from_numpy(order // cfg.topk)]
        send_e = torch.from_numpy(flat[order].astype(np.int32))
        send_w = torch.from_numpy(r["w"].reshape(-1)[order].astype(np.float32))
        per = cfg.n_experts // R
        counts = torch.bincount(send_e.long() // per, minlength=R).to(torch.int32)
        return send_x, send_e, send_w, counts, {"order": order}

    def ep_experts(self, cfg, R, q, x_recv, e_recv, w_recv, w_gate, w_up, w_down):
        M = x_recv.shape[0]
        if M == 0:
            return torch.zeros(0, cfg.d, dtype=torch.float32)
        per = cfg.n_experts // R
        idx = (e_recv.numpy() - q * per).reshape(-1, 1).astype(np.int32)
        assert idx.min() >= 0 and idx.max() < per
        need = sorted(set(idx.reshape(-1).tolist()))
        pick = lambda wt: {e: inputs.bf16_bits(wt[e]) for e in need}  # noqa: E731
        _, exact = oracle.experts_bf16(inputs.bf16_bits(x_recv), idx, w_recv.numpy().reshape(-1, 1),
                                       pick(w_gate), pick(w_up), pick(w_down), per, exact=True)
        return torch.from_numpy(exact.astype(np.float32))

    def ep_combine(self, cfg, y_back, T, ws):
        order = ws["order"]
        pos = np.empty_like(order)
        pos[order] = np.arange(len(order))
        y = y_back.numpy()[pos].reshape(T, cfg.topk, cfg.d)
        acc = np.zeros((T, cfg.d), np.float32)
        for j in range(cfg.topk):                         # FP32, slot order
            acc += y[:, j]
        return torch.from_numpy(acc).to(torch.bfloat16)


def _layer():
    t = inputs.generate(CFG, "cpu", T=1)
    return t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"], t["w_down"]


def _hidden(rank, T):
    g = torch.Generator().manual_seed(1000 + rank)
    return torch.randn(T, CFG.d, generator=g).to(torch.bfloat16)


def _single_rank(hidden, router_w, bias, wg, wu, wd):
    ops = OracleOps()
    sx, se, sw, counts, ws = ops.ep_dispatch(CFG, hidden, router_w, bias, 1)
    y = ops.ep_experts(CFG, 1, 0, sx, se, sw, wg, wu, wd)
    return ops.ep_combine(CFG, y, hidden.shape[0], ws)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, Ts, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.set_num_threads(1)     # the ranks share the host's cores
    oracle.set_threads(2)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        router_w, bias, wg, wu, wd = _layer()
        sl = ep.expert_slice(CFG, world, rank)
        h = _hidden(rank, Ts[rank])
        out = ep.forward_ep(CFG, h, router_w, bias, wg[sl], wu[sl], wd[sl], ops=OracleOps())
        ref = _single_rank(h, router_w, bias, wg, wu, wd)
        q.put((rank, tuple(out.shape), bool(torch.equal(out.view(torch.int16),
                                                       ref.view(torch.int16)))))
    finally:
        dist.destroy_process_group()


def _run(Ts):
    world = len(Ts)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, Ts, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = dict((r, (shape, same)) for r, shape, same in (q.get(timeout=10) for _ in range(world)))
    for r in range(world):
        assert res[r] == ((Ts[r], CFG.d), True), (r, res[r])


@pytest.mark.parametrize("Ts", [[20, 7], [0, 12]])
def test_two_ranks_match_the_single_rank_layer(Ts):
    """Uneven token counts, and a rank without tokens that still serves its
    experts."""
    _run(Ts)


def test_four_ranks_match_the_single_rank_layer():
    _run([5, 0, 9, 3])


def test_stand_in_combine_matches_the_oracle_layer():
    """The single-rank stand-in pipeline is the oracle layer up to the FP32
    rounding of each weighted row (it sums FP32 rows; the oracle sums FP64)."""
    router_w, bias, wg, wu, wd = _layer()
    h = _hidden(7, 11)
    got = _single_rank(h, router_w, bias, wg, wu, wd).float().numpy()
    ref, _, _ = oracle.forward_bf16(inputs.bf16_bits(h), router_w.numpy(), bias.numpy(),
                                    inputs.bf16_bits(wg), inputs.bf16_bits(wu),
                                    inputs.bf16_bits(wd), CFG.n_groups, CFG.topk_groups,
                                    CFG.topk, CFG.routed_scale)
    ref = oracle.bf16_to_f64(ref)
    # at most one BF16 step apart
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
