"""GPU parity on the small workload and its variants: every step of the CUDA
path against the CPU oracle on the same seeded inputs, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import (W_RTOL_SELECT, check_logits, check_out, check_routing, gpu_routing, host,
                     oracle_out, oracle_route, output_routing)

pytestmark = pytest.mark.gpu
CFG = inputs.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny():
    dev = torch.device("cuda")
    t = inputs.generate(CFG, dev)
    lg, r = oracle_route(CFG, t)
    return t, lg, r


def test_route_matches_oracle(tiny):
    t, lg, r = tiny
    idx, w, logits = pkg.route(CFG, t["hidden"], t["router_w"], t["corr_bias"], want_logits=True)
    check_logits(host(logits), lg)
    check_routing(CFG, host(idx), host(w), r)


def test_select_alone_on_oracle_logits(tiny):
    t, lg, r = tiny
    idx, w = pkg.select(CFG, torch.from_numpy(lg).cuda(), t["corr_bias"])
    check_routing(CFG, host(idx), host(w), r, w_rtol=W_RTOL_SELECT)


def test_forward_routed_matches_oracle(tiny):
    t, lg, r = tiny
    out = pkg.forward_routed(CFG, t["hidden"], torch.from_numpy(r["idx"]).cuda(),
                             torch.from_numpy(r["w"]).cuda(), t["w_gate"], t["w_up"], t["w_down"])
    ref = oracle_out(CFG, t, r["idx"], r["w"])
    check_out(out, ref)


def test_forward_matches_oracle(tiny):
    t, lg, r = tiny
    ws = pkg.Workspace(CFG, CFG.T)
    out = pkg.forward(CFG, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                      t["w_down"], ws=ws)
    assert pkg.check_status(ws) == 0
    ref = oracle_out(CFG, t, *output_routing(CFG, r, gpu_routing(ws, CFG, CFG.T)))
    check_out(out, ref)


def test_permutation_is_a_stable_counting_sort(tiny):
    t, lg, r = tiny
    ws = pkg.Workspace(CFG, CFG.T)
    pkg.forward_routed(CFG, t["hidden"], torch.from_numpy(r["idx"]).cuda(),
                       torch.from_numpy(r["w"]).cuda(), t["w_gate"], t["w_up"], t["w_down"], ws=ws)
    torch.cuda.synchronize()
    TK = CFG.T * CFG.topk
    E = CFG.n_experts
    flat = r["idx"].reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(host(ws.view("counts", torch.int32, (E,))), counts)
    assert np.array_equal(host(ws.view("offsets", torch.int32, (E + 1,))),
                          np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(host(ws.view("perm_src", torch.int32, (TK,))), order)
    inv = np.empty(TK, np.int64)
    inv[order] = np.arange(TK)
    assert np.array_equal(host(ws.view("pair_row", torch.int32, (TK,))), inv)
    assert np.array_equal(host(ws.view("perm_w", torch.float32, (TK,))), r["w"].reshape(-1)[order])


@pytest.mark.parametrize("T,skew", [(1100, False), (2051, True)])
def test_large_permutation_is_the_same_stable_sort(T, skew):
    """From 8192 entries on the permutation is a counting sort over chunks of
    1024 entries (ragged last chunk here); it must give the same stable
    (expert, token, slot) order, also when a few experts take most rows."""
    cfg = CFG.replace(T=T, seed=T)
    t = inputs.generate(cfg, "cuda")
    rng = np.random.default_rng(T)
    E, k = cfg.n_experts, cfg.topk
    p = rng.dirichlet(np.full(E, 0.05 if skew else 5.0))
    idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 0.5, (T, k)).astype(np.float32)
    ws = pkg.Workspace(cfg, T)
    out = pkg.forward_routed(cfg, t["hidden"], torch.from_numpy(idx).cuda(),
                             torch.from_numpy(w).cuda(), t["w_gate"], t["w_up"], t["w_down"],
                             ws=ws)
    assert pkg.check_status(ws) == 0
    TK = T * k
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(host(ws.view("counts", torch.int32, (E,))), counts)
    assert np.array_equal(host(ws.view("offsets", torch.int32, (E + 1,))),
                          np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(host(ws.view("perm_src", torch.int32, (TK,))), order)
    inv = np.empty(TK, np.int64)
    inv[order] = np.arange(TK)
    assert np.array_equal(host(ws.view("pair_row", torch.int32, (TK,))), inv)
    assert np.array_equal(host(ws.view("perm_w", torch.float32, (TK,))), w.reshape(-1)[order])
    rows = np.sort(rng.choice(T, 40, replace=False))
    check_out(out, oracle_out(cfg, t, idx, w, tokens=rows), rows=rows)


def test_deterministic_bitwise(tiny):
    t, _, _ = tiny
    args = (CFG, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"], t["w_down"])
    a = pkg.forward(*args)
    b = pkg.forward(*args)
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [1, 2, 5, 37, 130, 300])
def test_ragged_token_counts(T):
    """Token counts that fill no tile evenly (and, at 300, the 128-wide tile)."""
    cfg = CFG.replace(T=T, seed=10 + T)
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, T)
    out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                      t["w_down"], ws=ws)
    ref = oracle_out(cfg, t, *output_routing(cfg, r, gpu_routing(ws, cfg, T)))
    check_out(out, ref)
    idx, w = pkg.route(cfg, t["hidden"], t["router_w"], t["corr_bias"])
    check_routing(cfg, host(idx), host(w), r)


def test_zero_tokens_is_a_no_op():
    t = inputs.generate(CFG, "cuda", T=4)
    out = torch.full((0, CFG.d), 7, dtype=torch.bfloat16, device="cuda")
    x = t["hidden"][:0]
    o = pkg.forward(CFG, x, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"], t["w_down"],
                    out=out)
    assert o.shape == (0, CFG.d)


def test_all_tokens_on_one_expert_and_idle_experts():
    """Bias forces every token onto the same 8 experts: one expert gets all T
    rows (several token tiles), 56 experts get none."""
    cfg = CFG.replace(T=300, seed=77)
    t = inputs.generate(cfg, "cuda")
    b = t["corr_bias"].clone()
    b[[3, 4, 9, 12, 17, 18, 25, 26]] += 5.0
    t["corr_bias"] = b
    lg, r = oracle_route(cfg, t)
    assert np.all(np.sort(r["idx"], 1) == [3, 4, 9, 12, 17, 18, 25, 26])
    ws = pkg.Workspace(cfg, cfg.T)
    out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                      t["w_down"], ws=ws)
    ref = oracle_out(cfg, t, *output_routing(cfg, r, gpu_routing(ws, cfg, cfg.T)))
    check_out(out, ref)


def test_all_equal_scores_follow_the_tie_rule():
    """Zero router and zero bias: every score ties; lower indices win."""
    t = inputs.generate(CFG, "cuda", T=33)
    idx, w = pkg.route(CFG, t["hidden"], torch.zeros_like(t["router_w"]),
                       torch.zeros_like(t["corr_bias"]))
    assert np.array_equal(host(idx), np.tile(np.arange(8), (33, 1)))
    assert np.all(host(w) == np.float32(2.5 / 8))


def test_identical_experts_give_scaled_single_expert():
    """All experts equal => out = bf16(2.5 * y(x)) whatever the routing."""
    cfg = CFG.replace(T=40, seed=5)
    t = inputs.generate(cfg, "cuda")
    for k in ("w_gate", "w_up", "w_down"):
        t[k] = t[k][:1].expand_as(t[k]).contiguous()
    out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                      t["w_down"])
    one = np.zeros((cfg.T, 1), np.int32)
    ref = oracle.experts_bf16(host(t["hidden"]), one, np.full((cfg.T, 1), 2.5, np.float32),
                              {0: host(t["w_gate"][0])}, {0: host(t["w_up"][0])},
                              {0: host(t["w_down"][0])}, cfg.n_experts, exact=True)
    check_out(out, ref)


def test_invalid_routed_index_latches_device_check():
    t = inputs.generate(CFG, "cuda", T=8)
    ws = pkg.Workspace(CFG, 8)
    idx = torch.zeros(8, CFG.topk, dtype=torch.int32, device="cuda")
    idx[:, :] = torch.arange(CFG.topk, dtype=torch.int32, device="cuda")
    idx[3, 2] = CFG.n_experts + 5
    w = torch.full((8, CFG.topk), 0.25, device="cuda")
    pkg.forward_routed(CFG, t["hidden"], idx, w, t["w_gate"], t["w_up"], t["w_down"], ws=ws)
    assert pkg.check_status(ws) == 6
    assert pkg.check_status(ws) == 0   # cleared by the read


def test_host_side_argument_errors():
    t = inputs.generate(CFG, "cuda", T=4)
    bad = CFG.replace(d=500)
    with pytest.raises(pkg.BeamError) as e:
        pkg.workspace_size(bad, 4)
    assert e.value.code == 1
    ws = pkg.Workspace(CFG, 2)
    with pytest.raises(pkg.BeamError) as e:
        pkg.forward(CFG, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                    t["w_down"], ws=ws)
    assert e.value.code == 3


@pytest.mark.parametrize("T", [256, 300, 1000])
def test_tensor_core_router_mid_sized_layer(T):
    """From 256 tokens on (E a multiple of 128) the router runs as a BF16x3
    tensor-core GEMM; its logits must still meet the FP32 tolerance."""
    cfg = CFG.replace(T=T, n_experts=128, d=512, d_ff=256, seed=40 + T)
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    idx, w, logits = pkg.route(cfg, t["hidden"], t["router_w"], t["corr_bias"], want_logits=True)
    check_logits(host(logits), lg)
    check_routing(cfg, host(idx), host(w), r)
    ws = pkg.Workspace(cfg, T)
    out = pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                      t["w_down"], ws=ws)
    rows = np.arange(min(T, 64))
    ref = oracle_out(cfg, t, *output_routing(cfg, r, gpu_routing(ws, cfg, T), rows), tokens=rows)
    check_out(out, ref, rows=rows)


@pytest.mark.parametrize("E,G,kg,k", [(256, 128, 16, 8), (128, 64, 8, 8), (64, 2, 1, 6),
                                      (96, 3, 2, 4), (256, 16, 4, 8), (32, 16, 3, 5)])
def test_group_shapes(E, G, kg, k):
    """Selection for group sizes from 2 to 32 experts and up to 128 groups,
    alone on the oracle's logits and inside the fused decode-sized routing of
    a forward call."""
    cfg = CFG.replace(T=20, n_experts=E, n_groups=G, topk_groups=kg, topk=k, seed=E + G + k)
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    idx, w = pkg.select(cfg, torch.from_numpy(lg).cuda(), t["corr_bias"])
    check_routing(cfg, host(idx), host(w), r, w_rtol=W_RTOL_SELECT)
    ws = pkg.Workspace(cfg, cfg.T)
    pkg.forward(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                t["w_down"], ws=ws)
    assert pkg.check_status(ws) == 0
    check_routing(cfg, host(ws.view("topk_idx", torch.int32, (cfg.T, k))),
                  host(ws.view("topk_w", torch.float32, (cfg.T, k))), r)


@pytest.mark.parametrize("T", [32, 300])
def test_expert_gemms_alone(T):
    """Each expert GEMM from its own inputs: h of the gate/up GEMM against the
    oracle's SwiGLU rows (one BF16 step apart at most, where the fast exp
    lands a product on the other side of a rounding boundary), and y of the
    down GEMM against an FP64 matmul of the GPU's own h times the routing
    weight.  T = 32 takes the 16-row blocks, T = 300 the 256-row blocks and
    the paired down GEMM."""
    cfg = CFG.replace(T=T, seed=200 + T)
    t = inputs.generate(cfg, "cuda")
    lg, r = oracle_route(cfg, t)
    ws = pkg.Workspace(cfg, T)
    pkg.forward_routed(cfg, t["hidden"], torch.from_numpy(r["idx"]).cuda(),
                       torch.from_numpy(r["w"]).cuda(), t["w_gate"], t["w_up"], t["w_down"],
                       ws=ws)
    assert pkg.check_status(ws) == 0
    TK, F, d, k = T * cfg.topk, cfg.d_ff, cfg.d, cfg.topk
    perm = host(ws.view("perm_src", torch.int32, (TK,)))
    h = host(ws.view("h", torch.bfloat16, (TK, F)))
    y = ws.view("y", torch.float32, (TK, d)).cpu().double().numpy()
    x = host(t["hidden"])
    rows = np.random.default_rng(T).choice(TK, 48, replace=False)
    flat = r["idx"].reshape(-1)
    wflat = r["w"].reshape(-1)
    for row in rows:
        e, tok = int(flat[perm[row]]), int(perm[row] // k)
        ref = oracle.swiglu_bf16(x[tok:tok + 1], host(t["w_gate"][e]), host(t["w_up"][e]))[0]
        a = h[row].astype(np.int32)
        b = ref.astype(np.int32)
        a = np.where(a & 0x8000, 0x8000 - a, a)
        b = np.where(b & 0x8000, 0x8000 - b, b)
        assert np.abs(a - b).max() <= 1, row
        assert (a != b).mean() < 0.02, row
        hv = torch.from_numpy(h[row].view(np.int16)).view(torch.bfloat16).double()
        wd = t["w_down"][e].cpu().double()
        prod = wd * hv[None, :]
        yref = float(wflat[perm[row]]) * prod.sum(1).numpy()
        bound = 1e-4 * abs(float(wflat[perm[row]])) * prod.abs().sum(1).numpy() + 1e-30
        assert np.all(np.abs(y[row] - yref) <= bound), row
