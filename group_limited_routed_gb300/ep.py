"""Expert-parallel Beam MoE layer over a ``torch.distributed`` process group.

Rank q of R owns experts [q*E/R, (q+1)*E/R) and holds only their weights.
Each rank routes its own tokens; the rows of its (token, slot) pairs go to
the ranks owning their experts with explicit expert ids and routing
weights; every rank runs its experts on what it received (also when it has
no tokens of its own); the weighted FP32 rows come back in the order they
were sent, and the token's owner sums them in slot order and rounds once to
BF16.  ("SGLang 原生支持 Reflection 的 Beam 并驱动其生产 API", section "Fusion
Optimizations": the MegaMoE item and the token-ownership figure after it.)

The exchange is five ``all_to_all_single`` calls (counts, rows, expert ids,
weights, and the rows back) and one host read of the send counts, which the
variable-size all-to-all needs.  Every computation runs in the CUDA library;
this module moves buffers between ranks only.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def forward_ep(cfg, hidden, router_w, corr_bias, w_gate, w_up, w_down, group=None, ops=None):
    """This rank's tokens through the expert-parallel layer -> out [T, d] bf16.

    ``w_gate`` / ``w_up`` [E/R, d_ff, d] and ``w_down`` [E/R, d, d_ff] hold
    this rank's experts, BF16 tensors, ``api.Fp4Weight`` (NVFP4, as the
    pages' MegaMoE path) or ``api.Fp8Weight`` (dynamic FP8).  ``ops``
    supplies ``ep_dispatch``, ``ep_experts``, ``ep_experts_nvfp4``,
    ``ep_experts_fp8`` and ``ep_combine`` (default: the CUDA library)."""
    ops = api if ops is None else ops
    R = dist.get_world_size(group)
    r = dist.get_rank(group)
    if cfg.n_experts % R:
        raise ValueError(f"{R} ranks do not divide {cfg.n_experts} experts")
    T = hidden.shape[0]
    send_x, send_e, send_w, counts, ws = ops.ep_dispatch(cfg, hidden, router_w, corr_bias, R)

    recv_counts = torch.empty_like(counts)
    dist.all_to_all_single(recv_counts, counts, group=group)
    send_split = [int(v) for v in counts.tolist()]
    recv_split = [int(v) for v in recv_counts.tolist()]
    M = sum(recv_split)

    recv_x = send_x.new_empty(M, cfg.d)
    recv_e = send_e.new_empty(M)
    recv_w = send_w.new_empty(M)
    dist.all_to_all_single(recv_x, send_x, recv_split, send_split, group=group)
    dist.all_to_all_single(recv_e, send_e, recv_split, send_split, group=group)
    dist.all_to_all_single(recv_w, send_w, recv_split, send_split, group=group)

    experts = (ops.ep_experts_nvfp4 if isinstance(w_gate, api.Fp4Weight)
               else ops.ep_experts_fp8 if isinstance(w_gate, api.Fp8Weight) else ops.ep_experts)
    y_recv = experts(cfg, R, r, recv_x, recv_e, recv_w, w_gate, w_up, w_down)

    y_back = y_recv.new_empty(T * cfg.topk, cfg.d)
    dist.all_to_all_single(y_back, y_recv, send_split, recv_split, group=group)
    return ops.ep_combine(cfg, y_back, T, ws)


def expert_slice(cfg, R: int, q: int):
    """The expert range rank q of R owns, as a slice of the expert axis."""
    per = cfg.n_experts // R
    return slice(q * per, (q + 1) * per)
