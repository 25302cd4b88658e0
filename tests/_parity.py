"""Shared helpers of the GPU parity tests: run the oracle on the same seeded
inputs and compare with the tolerances the layer's specification states
(router logits within 1e-5 relative; expert indices exact except where the
oracle's k-th/(k+1)-th margin is below 1e-6; BF16 outputs within
max-abs 1e-2 * RMS(out)).

Output tolerance, as read here: the bound 1e-2 * RMS(out) applies to the
arithmetic error, measured against the oracle's exact (float64) output
before its final rounding; the BF16 output format adds its own rounding of
at most half a unit in the last place of each value on top (one BF16 step
of a value above about 2.6 * RMS is already larger than 1e-2 * RMS, so no
BF16 result could meet the bound against a BF16-rounded reference)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from group_limited_routed_gb300 import inputs

LOGIT_RTOL = 1e-5
MARGIN = 1e-6
OUT_TOL = 1e-2


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return inputs.bf16_bits(t)
    return t.detach().cpu().numpy()


def oracle_route(cfg, tens):
    lg = oracle.router_logits(host(tens["hidden"]), host(tens["router_w"]))
    r = oracle.route(lg, host(tens["corr_bias"]), cfg.n_groups, cfg.topk_groups, cfg.topk,
                     cfg.routed_scale)
    return lg, r


def check_logits(got: np.ndarray, ref: np.ndarray):
    """|got - ref| <= 1e-5 * max(|ref|, RMS of the reference row)."""
    rms = np.sqrt((ref.astype(np.float64) ** 2).mean(axis=1, keepdims=True))
    bound = LOGIT_RTOL * np.maximum(np.abs(ref), rms)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = err > bound
    print(f"  logits: max |err| {err.max():.3g}, worst {(err / bound).max():.3g} of the bound")
    assert not bad.any(), f"{bad.sum()} logits out of tolerance; worst {(err / bound).max():.3g}x"


def exempt_tokens(r) -> np.ndarray:
    """Tokens whose expert indices are exempt from the bit-exact comparison
    (the oracle's k-th/(k+1)-th or kg-th/(kg+1)-th margin below 1e-6)."""
    return (r["expert_margin"] < MARGIN) | (r["group_margin"] < MARGIN)


# Scores the oracle reads as tied when it lists a near-tie token's other
# valid routings: the exemption margin with room for the GPU's FP32 score
# error (the same slack check_routing allows an exempt token's choice).
NEAR_TIE_TOL = 4 * MARGIN


def gpu_routing(ws, cfg, T) -> np.ndarray:
    """The expert indices a layer call left in its workspace."""
    return host(ws.view("topk_idx", torch.int32, (T, cfg.topk)))


def output_routing(cfg, r, gpu_idx, tokens=None):
    """(idx, w) to compute the oracle's output with, per token: the oracle's
    own routing where the GPU chose the same expert set; elsewhere (a token
    near a tie) the one of the oracle's near-tie routings, listed from its
    own scores, whose set equals the GPU's.  A token whose GPU set is none of
    them fails.  No value comes from the GPU: its set only picks which of
    the oracle's routings the output is compared with."""
    idx, w = r["idx"].copy(), r["w"].copy()
    rows = range(idx.shape[0]) if tokens is None else np.asarray(tokens).tolist()
    moved = 0
    for t in rows:
        g = set(np.asarray(gpu_idx[t]).tolist())
        if g == set(r["idx"][t].tolist()):
            continue
        alts = oracle.route_alternatives(r, t, cfg.n_groups, cfg.topk_groups, cfg.topk,
                                         cfg.routed_scale, NEAR_TIE_TOL)
        match = [a for a in alts if set(a["idx"].tolist()) == g]
        assert match, (f"token {t}: GPU experts {sorted(g)} are none of the oracle's "
                       f"{len(alts)} near-tie routings (its own: {r['idx'][t].tolist()})")
        idx[t], w[t] = match[0]["idx"], match[0]["w"]
        moved += 1
    if moved:
        print(f"  {moved} near-tie tokens compared on the oracle's alternative routing")
    return idx, w


def block_sample(cfg, idx, n, seed, nt):
    """A seeded sample of at least min(n, T) tokens for output checks of a
    large batch that reaches every kind of GEMM tile: the first and last
    tokens and, for every expert, the tokens of its first permuted row and of
    the first, middle and last rows of its last token block.  Rows are in
    the stable (expert, token, slot) order; an expert's n_e rows are cut
    into ceil(n_e / nt) blocks of equal size rounded up to 16 rows, the last
    one ragged.  Seeded random tokens fill the sample up to n."""
    T, k = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=cfg.n_experts)
    starts = np.concatenate([[0], np.cumsum(counts)])
    picks = {0, T - 1}
    for e in range(cfg.n_experts):
        c = int(counts[e])
        if c == 0:
            continue
        nb = -(-c // nt)
        bs = min(nt, (-(-c // nb) + 15) // 16 * 16)
        last0 = (nb - 1) * bs
        for p in (0, last0, (last0 + c - 1) // 2, c - 1):
            picks.add(int(order[starts[e] + p]) // k)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.fromiter(picks, np.int64))
    fill = max(0, min(n, T) - len(picks))
    if fill:
        picks.update(rng.choice(rest, min(fill, rest.size), replace=False).tolist())
    return np.array(sorted(picks), np.int64)


# Routing-weight tolerance when the GPU computed its own logits: a logit off
# by up to 1e-5 * max(|logit|, RMS) moves s = sigmoid(logit) by (1 - s) times
# that, relatively, and w = 2.5 s / sum(s) by at most twice it; logits reach a
# few units, so 1e-4 covers it.  Fed the oracle's logits, only the FP32
# sigmoid's last-place differences remain (1e-6).
W_RTOL_ROUTE = 1e-4
W_RTOL_SELECT = 1e-6


def tie_runs(cs) -> list[tuple[int, int]]:
    """Runs of slots whose neighbouring oracle choice scores (slot order,
    descending) differ by less than the margin: inside a run the slot order
    is not fixed, since a choice-score error below the margin may swap it."""
    runs, start = [], 0
    for j in range(1, len(cs)):
        if cs[j - 1] - cs[j] >= MARGIN:
            runs.append((start, j))
            start = j
    runs.append((start, len(cs)))
    return runs


def check_routing(cfg, idx: np.ndarray, w: np.ndarray, r, w_rtol=W_RTOL_ROUTE):
    """Non-exempt tokens: the expert set bit-exact, and the slot order too
    wherever neighbouring oracle choice scores are at least the margin apart
    (inside a near-tie run only the run's set is fixed); weights close, matched
    by expert.  Exempt tokens must still pick a valid near-tie set."""
    ex = exempt_tokens(r)
    ok = ~ex
    bad = []
    for t in np.nonzero(ok & ~np.all(idx == r["idx"], axis=1))[0]:
        cs = r["c"][t][r["idx"][t]].astype(np.float64)
        if any(set(idx[t, a:b].tolist()) != set(r["idx"][t, a:b].tolist())
               for a, b in tie_runs(cs)):
            bad.append(t)
    if bad:
        t = bad[0]
        raise AssertionError(
            f"{len(bad)} tokens route differently; token {t}: GPU {idx[t].tolist()}, oracle "
            f"{r['idx'][t].tolist()}, oracle c of the GPU's {r['c'][t][idx[t]].tolist()} "
            f"and of its own {r['c'][t][r['idx'][t]].tolist()}, expert margin "
            f"{r['expert_margin'][t]:.3g}, group margin {r['group_margin'][t]:.3g}")
    wg = np.take_along_axis(w[ok], np.argsort(idx[ok], 1), 1)
    wr = np.take_along_axis(r["w"][ok], np.argsort(r["idx"][ok], 1), 1)
    assert np.allclose(wg, wr, rtol=w_rtol, atol=0)
    S = cfg.n_experts // cfg.n_groups
    for t in np.nonzero(ex)[0]:
        row = idx[t]
        assert len(set(row.tolist())) == cfg.topk
        c = r["c"][t]
        kth = np.sort(c[r["idx"][t]])[0]
        # every chosen expert is at most a margin away from the oracle's k-th
        assert np.all(c[row] >= kth - 4 * MARGIN)
        assert len({int(e) // S for e in row}) <= cfg.topk_groups
    assert np.all(np.abs(w.astype(np.float64).sum(1) - cfg.routed_scale) <= 1e-5)
    return ex


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half the BF16 spacing at |v| (8 significant bits)."""
    _, e = np.frexp(np.abs(v))
    return np.where(v == 0, 0.0, np.ldexp(1.0, e - 9))


def check_out(got, ref, rows=None, tol=OUT_TOL, slack=None, rms=None):
    """ref = (bf16 bits, exact float64) as the oracle returns them.  Asserts
    |got - exact| <= tol * RMS(exact) + half a BF16 step of exact (+ slack, a
    per-element allowance the oracle computed, when given); RMS is taken over
    the compared rows unless given; returns (max |got - exact|, RMS, fraction
    bit-identical to the oracle's BF16)."""
    bits, exact = ref[0], ref[1]
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    o16 = oracle.bf16_to_f64(bits)
    extra = np.zeros_like(exact) if slack is None else slack
    if rows is not None:
        g, exact, o16, extra = g[rows], exact[rows], o16[rows], extra[rows]
    if g.size == 0:
        return 0.0, 0.0, 1.0
    rms = np.sqrt((exact ** 2).mean()) if rms is None else rms
    err = np.abs(g - exact)
    excess = err - (tol * rms + half_ulp_bf16(exact) + extra)
    print(f"  arithmetic error beyond BF16 rounding: {max(0.0, float((err - half_ulp_bf16(exact)).max())) / rms:.2e} * RMS")
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"err {err[worst]:.4g} at {worst} (value {exact[worst]:.4g}) > "
                               f"{tol} * RMS {rms:.4g} + half BF16 step")
    return float(err.max()), float(rms), float((g == o16).mean())


def expert_weights_host(tens, experts):
    """Host copies of the BF16 weights of the listed experts (dict e -> arr)."""
    wg, wu, wd = {}, {}, {}
    for e in sorted({int(x) for x in experts}):
        wg[e] = host(tens["w_gate"][e])
        wu[e] = host(tens["w_up"][e])
        wd[e] = host(tens["w_down"][e])
    return wg, wu, wd


def oracle_out(cfg, tens, idx, w, tokens=None):
    """Oracle expert output for the given routing, only for `tokens` rows
    (None = all), fetching only the weights those rows use."""
    rows = np.arange(idx.shape[0]) if tokens is None else np.asarray(tokens)
    wg, wu, wd = expert_weights_host(tens, idx[rows].reshape(-1))
    return oracle.experts_bf16(host(tens["hidden"]), idx, w, wg, wu, wd, cfg.n_experts,
                               tokens=None if tokens is None else rows, exact=True)
