"""Out-of-range and foreign routed indices on the larger-batch paths.

A routed index outside the expert range (or, with expert parallelism, owned
by another rank) gets no permuted row: the permutation marks it with row -1,
latches the device check (status 6) and the entry contributes nothing.  The
kernels that write token rows to their permuted rows (the per-token scatter
of BF16 rows and of E4M3 codes, and the NVFP4 token quantisation) must skip
such an entry rather than write before their buffer.  Each test plants one bad
entry and compares every other output bit for bit with a call whose bad entry
is replaced by a valid one: the per-row arithmetic does not depend on which
rows share a tile, so the valid rows must not move."""
import numpy as np
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import ep, inputs

pytestmark = pytest.mark.gpu
TINY = inputs.CONFIGS["tiny"]


def _on_cuda(t):
    return {k: ({kk: vv.cuda() for kk, vv in v.items()} if isinstance(v, dict)
                else v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def _routing(cfg, T, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(cfg.n_experts, generator=g)[:cfg.topk] for _ in range(T)])
    w = torch.rand(T, cfg.topk, generator=g) + 0.1
    return idx.to(torch.int32).cuda(), w.cuda()


@pytest.mark.parametrize("T", [40, 100])
def test_forward_routed_bad_index_large_batch(T):
    """T * k > 4 E: the BF16 token rows go through the per-token scatter."""
    cfg = TINY.replace(T=T, seed=300 + T)
    assert T * cfg.topk > 4 * cfg.n_experts
    t = inputs.generate(cfg, "cuda")
    idx, w = _routing(cfg, T, T)
    bad_t, bad_s = T // 3, 5
    good_idx = idx.clone()
    idx[bad_t, bad_s] = cfg.n_experts + 7
    ws = pkg.Workspace(cfg, T)
    out = pkg.forward_routed(cfg, t["hidden"], idx, w, t["w_gate"], t["w_up"], t["w_down"], ws=ws)
    assert pkg.check_status(ws) == 6
    # the permuted weights of the valid entries are intact (the buffer sits
    # just before the permuted token rows)
    n_valid = T * cfg.topk - 1
    flat_i = idx.reshape(-1).cpu().numpy()
    flat_w = w.reshape(-1).cpu().numpy()
    ok = flat_i < cfg.n_experts
    order = np.argsort(flat_i[ok], kind="stable")
    perm_w = ws.view("perm_w", torch.float32, (T * cfg.topk,)).cpu().numpy()
    assert np.array_equal(perm_w[:n_valid], flat_w[ok][order])
    ref = pkg.forward_routed(cfg, t["hidden"], good_idx, w, t["w_gate"], t["w_up"], t["w_down"])
    keep = torch.ones(T, dtype=torch.bool, device="cuda")
    keep[bad_t] = False
    assert torch.equal(out[keep].view(torch.int16), ref[keep].view(torch.int16))


def _ep_case(M, R=2, q=1, seed=0):
    sl = ep.expert_slice(TINY, R, q)
    g = torch.Generator().manual_seed(seed)
    e = (torch.randint(0, sl.stop - sl.start, (M,), generator=g) + sl.start).to(torch.int32)
    w = torch.rand(M, generator=g) + 0.1
    return sl, e.cuda(), w.cuda()


@pytest.mark.parametrize("M", [40, 200])
def test_ep_experts_foreign_expert(M):
    """BF16 expert-parallel rows; M = 200 > 4 * 32 local experts takes the
    per-token scatter."""
    R, q = 2, 1
    t = inputs.generate(TINY, "cuda", T=M)
    sl, e, w = _ep_case(M, R, q, seed=M)
    x = t["hidden"]
    bad = M // 2
    e_bad = e.clone()
    e_bad[bad] = 0                                     # owned by rank 0
    ws = pkg.EpWorkspace(TINY, R, M)
    y = pkg.ep_experts(TINY, R, q, x, e_bad, w, t["w_gate"][sl], t["w_up"][sl],
                       t["w_down"][sl], ws=ws)
    assert pkg.check_status(ws) == 6
    ref = pkg.ep_experts(TINY, R, q, x, e, w, t["w_gate"][sl], t["w_up"][sl], t["w_down"][sl])
    keep = torch.ones(M, dtype=torch.bool, device="cuda")
    keep[bad] = False
    assert torch.equal(y[keep], ref[keep])


@pytest.mark.parametrize("M", [40, 200])
def test_ep_experts_fp8_foreign_expert(M):
    """Dynamic-FP8 expert-parallel rows; M = 200 scatters the E4M3 codes."""
    R, q = 2, 1
    cfg = TINY.replace(weight_fmt="fp8", seed=310)
    t = _on_cuda(inputs.generate(cfg, "cpu", T=M))
    sl, e, w = _ep_case(M, R, q, seed=M + 1)
    loc = [pkg.Fp8Weight(t[n]["q"][sl], t[n]["s"][sl]) for n in ("w_gate", "w_up", "w_down")]
    bad = M // 3
    e_bad = e.clone()
    e_bad[bad] = 3                                     # owned by rank 0
    ws = pkg.EpWorkspace(cfg, R, M, weight_fmt=pkg.FP8)
    y = pkg.ep_experts_fp8(cfg, R, q, t["hidden"], e_bad, w, *loc, ws=ws)
    assert pkg.check_status(ws) == 6
    ref = pkg.ep_experts_fp8(cfg, R, q, t["hidden"], e, w, *loc)
    keep = torch.ones(M, dtype=torch.bool, device="cuda")
    keep[bad] = False
    assert torch.equal(y[keep], ref[keep])


@pytest.mark.parametrize("M", [24, 200])
def test_ep_experts_nvfp4_foreign_expert(M):
    """NVFP4 expert-parallel rows: the token quantisation writes each row's
    codes and scales to its permuted rows at every batch size."""
    R, q = 2, 0
    cfg = TINY.replace(weight_fmt="nvfp4", seed=320)
    t = _on_cuda(inputs.generate(cfg, "cpu", T=M))
    sl, e, w = _ep_case(M, R, q, seed=M + 2)
    loc = [pkg.Fp4Weight.of({k: v[sl] for k, v in t[n].items()})
           for n in ("w_gate", "w_up", "w_down")]
    bad = M - 1
    e_bad = e.clone()
    e_bad[bad] = TINY.n_experts - 1                    # owned by rank 1
    ws = pkg.EpWorkspace(cfg, R, M, weight_fmt=pkg.NVFP4)
    y = pkg.ep_experts_nvfp4(cfg, R, q, t["hidden"], e_bad, w, *loc, ws=ws)
    assert pkg.check_status(ws) == 6
    ref = pkg.ep_experts_nvfp4(cfg, R, q, t["hidden"], e, w, *loc)
    keep = torch.ones(M, dtype=torch.bool, device="cuda")
    keep[bad] = False
    assert torch.equal(y[keep], ref[keep])
