"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- a library routine, brute force, a closed form, an invariant or
a special case the pages fix.  CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from group_limited_routed_gb300 import inputs

RNG = np.random.default_rng(1234)


def f32_ulp_close(a, b, ulps=1):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    sp = np.spacing(np.maximum(np.abs(a), np.abs(b))).astype(np.float64)
    return np.all(np.abs(a.astype(np.float64) - b.astype(np.float64)) <= ulps * sp)


def bf16_nearest(v) -> np.ndarray:
    """BF16 bits of the nearest BF16 value of each float64 in v, ties to even,
    in one rounding.  Exact: |v| / spacing is a scaling by a power of two, and
    numpy's rint rounds half to even (normal BF16 range)."""
    v = np.asarray(v, np.float64)
    _, e = np.frexp(np.abs(v))                 # |v| in [2^(e-1), 2^e)
    step = np.ldexp(1.0, e - 8)                # 8 significant bits
    r = np.where(v == 0, v, np.copysign(np.rint(np.abs(v) / step) * step, v))
    return inputs.bf16_bits(torch.from_numpy(r).float().to(torch.bfloat16))


# ---------------------------------------------------------------- formats
def test_bf16_round_matches_torch():
    vals = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        RNG.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
        # exact ties: lower 16 bits == 0x8000 with both parities of the kept lsb
        (np.arange(0x3f800000, 0x3f800000 + 64 * 0x10000, 0x10000, dtype=np.uint32)
         + np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, np.inf, -np.inf], np.float32),
    ])
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def _minifloat(code, ebits, mbits, bias):
    """Generic minifloat decoder (sign | exponent | mantissa), no inf/nan."""
    sign = -1.0 if code >> (ebits + mbits) & 1 else 1.0
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        return sign * (m / (1 << mbits)) * 2.0 ** (1 - bias)
    return sign * (1 + m / (1 << mbits)) * 2.0 ** (e - bias)


def test_e2m1_values_from_format_definition():
    for c in range(16):
        assert oracle.e2m1_value(c) == _minifloat(c, 2, 1, 1)
    mags = sorted({abs(oracle.e2m1_value(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e4m3_all_256_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == float(ref[c]), (c, v, ref[c])


def test_e4m3_encode_vs_torch_rne():
    v = np.concatenate([
        np.exp(RNG.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)).astype(np.float32),
        # midpoints between neighbouring codes (ties)
        np.array([(oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2 for c in range(0, 126)],
                 np.float32),
        np.array([0.0, 448.0, 2.0 ** -9, 2.0 ** -10], np.float32),
    ])
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], np.uint8)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # satfinite above the largest finite value, sign kept
    assert oracle.e4m3_encode(1000.0) == 0x7E
    assert oracle.e4m3_encode(-1000.0) == 0xFE


def test_e2m1_encode_vs_independent_rounding():
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([RNG.uniform(-7, 7, 5000), mids, -mids, grid, -grid[1:], [6.5, -9.0]])
    v = v.astype(np.float32)
    got = np.array([oracle.e2m1_encode(float(x)) for x in v], np.uint8)
    ref = inputs._e2m1_codes(torch.from_numpy(v)).numpy()
    # +0 and -0 decode alike; compare the decoded values and the codes elsewhere
    dec_got = np.array([oracle.e2m1_value(int(c)) for c in got])
    dec_ref = np.array([oracle.e2m1_value(int(c)) for c in ref])
    assert np.array_equal(dec_got, dec_ref)
    nz = dec_got != 0
    assert np.array_equal(got[nz], ref[nz])
    # ties go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    for x, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
                    (5.0, 4.0), (7.0, 6.0)]:
        assert oracle.e2m1_value(oracle.e2m1_encode(x)) == want


def test_nvfp4_activation_quantizer_vs_torch():
    v = (RNG.standard_normal(16 * 512) * np.repeat(np.exp(RNG.uniform(-6, 3, 512)), 16))
    v = v.astype(np.float32)
    v[:16] = 0.0                      # an all-zero block
    q, sf = oracle.nvfp4_quantize(v)
    tv = torch.from_numpy(v).reshape(-1, 16)
    amax = tv.abs().amax(dim=1)
    sf_ref = (amax / 6.0).to(torch.float8_e4m3fn)
    scale = sf_ref.float().unsqueeze(1)
    codes_ref = torch.where(scale > 0, inputs._e2m1_codes(tv / torch.where(scale > 0, scale, 1.0)),
                            torch.zeros_like(tv, dtype=torch.uint8))
    assert np.array_equal(sf, sf_ref.view(torch.uint8).numpy())
    codes = np.stack([q & 15, q >> 4], axis=1).reshape(-1)
    dec = np.array([oracle.e2m1_value(int(c)) for c in codes])
    dec_ref = np.array([oracle.e2m1_value(int(c)) for c in codes_ref.reshape(-1).numpy()])
    assert np.array_equal(dec, dec_ref)


# ---------------------------------------------------------------- router
def _bf16_matrix(shape, scale=1.0):
    a = torch.from_numpy((RNG.standard_normal(shape) * scale).astype(np.float32))
    return a.to(torch.bfloat16)


def test_router_logits_vs_numpy_fp64():
    x = _bf16_matrix((37, 512))
    wr = (RNG.standard_normal((64, 512)) / np.sqrt(512)).astype(np.float32)
    got = oracle.router_logits(inputs.bf16_bits(x), wr)
    ref = (x.double().numpy() @ wr.astype(np.float64).T).astype(np.float32)
    assert f32_ulp_close(got, ref, 1)


def test_router_one_hot_picks_a_weight_column():
    d, E = 256, 32
    wr = (RNG.standard_normal((E, d))).astype(np.float32)
    x = torch.zeros(d, d, dtype=torch.bfloat16)
    x[torch.arange(d), torch.arange(d)] = 1.0
    got = oracle.router_logits(inputs.bf16_bits(x), wr)
    assert np.array_equal(got, wr.T)


# ---------------------------------------------------------------- selection
def _route(logits, bias, G, kg, k, alpha=2.5):
    return oracle.route(logits.astype(np.float32), bias.astype(np.float32), G, kg, k, alpha)


def test_sigmoid_scores_vs_scipy():
    from scipy.special import expit
    lg = np.concatenate([RNG.standard_normal((50, 64)) * 4, np.zeros((1, 64))]).astype(np.float32)
    r = _route(lg, np.zeros(64), 8, 4, 8)
    ref = expit(lg.astype(np.float64)).astype(np.float32)
    assert f32_ulp_close(r["s"], ref, 1)
    assert np.all(r["s"][-1] == np.float32(0.5))


def _brute_force(c, G, kg, k):
    """Best kg groups by the sum of the group scores (each the best pair sum
    in the group), then best k experts by the sum of their c."""
    E = c.size
    S = E // G
    gs = []
    for g in range(G):
        m = c[g * S:(g + 1) * S]
        gs.append(max(np.float32(m[i]) + np.float32(m[j])
                      for i in range(S) for j in range(S) if i != j))
    best_groups = max(itertools.combinations(range(G), kg),
                      key=lambda sub: sum(float(gs[g]) for g in sub))
    cand = [e for e in range(E) if e // S in best_groups]
    best = max(itertools.combinations(cand, k), key=lambda sub: sum(float(c[e]) for e in sub))
    return set(best_groups), set(best)


@pytest.mark.parametrize("E,G,kg,k", [(16, 8, 4, 3), (32, 4, 2, 4), (24, 6, 3, 5), (64, 8, 4, 8)])
def test_selection_brute_force(E, G, kg, k):
    T = 40 if E < 64 else 6
    lg = (RNG.standard_normal((T, E)) * 1.5).astype(np.float32)
    bias = RNG.uniform(-0.05, 0.05, E).astype(np.float32)
    r = _route(lg, bias, G, kg, k)
    for t in range(T):
        if E == 64:
            # C(32,8) subsets is too many: brute-force the groups only, then
            # check the experts are the k best candidates by a sort.
            S = E // G
            gsets, _ = _brute_force(r["c"][t], G, kg, 1)
            cand = np.array([e for e in range(E) if e // S in gsets])
            order = cand[np.argsort(-r["c"][t][cand], kind="stable")]
            assert set(r["idx"][t]) == set(order[:k])
        else:
            gsets, eset = _brute_force(r["c"][t], G, kg, k)
            assert set(np.nonzero(r["keep"][t])[0]) == gsets
            assert set(r["idx"][t]) == eset


def test_keep_all_groups_is_plain_topk():
    E, G, k = 64, 8, 8
    lg = (RNG.standard_normal((100, E)) * 2).astype(np.float32)
    bias = RNG.uniform(-0.05, 0.05, E).astype(np.float32)
    r = _route(lg, bias, G, G, k)
    ref = np.argsort(-r["c"], axis=1, kind="stable")[:, :k]
    assert np.array_equal(r["idx"], ref)
    assert np.all(np.isinf(r["group_margin"]))


def test_all_equal_scores_tie_rule():
    for E, G in [(64, 8), (256, 8)]:
        r = _route(np.zeros((3, E)), np.zeros(E), G, 4, 8)
        assert np.array_equal(r["idx"], np.tile(np.arange(8), (3, 1)))
        assert np.array_equal(r["keep"], np.tile(np.arange(G) < 4, (3, 1)))
        assert np.all(r["w"] == np.float32(2.5 / 8))
        assert np.all(r["expert_margin"] == 0) and np.all(r["group_margin"] == 0)


def test_combine_weights_use_scores_not_bias():
    from scipy.special import expit
    E = 64
    lg = (RNG.standard_normal((20, E))).astype(np.float32)
    bias = RNG.uniform(-0.05, 0.05, E).astype(np.float32)
    bias[:8] += 3.0       # forces the choice, must not leak into the weights
    r = _route(lg, bias, 8, 4, 8)
    s = expit(lg.astype(np.float64))
    sel = np.take_along_axis(s, r["idx"].astype(np.int64), 1)
    ref = 2.5 * sel / sel.sum(1, keepdims=True)
    assert np.allclose(r["w"], ref, rtol=2e-7, atol=0)
    assert np.all(np.sort(r["idx"], 1) == np.arange(8))


def test_invariants_on_tiny_config():
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cpu", weights=False)
    lg = oracle.router_logits(inputs.bf16_bits(t["hidden"]), t["router_w"].numpy())
    r = oracle.route(lg, t["corr_bias"].numpy(), cfg.n_groups, cfg.topk_groups, cfg.topk,
                     cfg.routed_scale)
    S = cfg.n_experts // cfg.n_groups
    idx = r["idx"]
    for row, keep in zip(idx, r["keep"]):
        assert len(set(row)) == cfg.topk
        assert all(keep[e // S] for e in row)
        assert keep.sum() == cfg.topk_groups
    assert np.all(r["w"] > 0)
    assert np.all(np.abs(r["w"].astype(np.float64).sum(1) - 2.5) <= 1e-6)
    assert np.all(r["expert_margin"] >= 0) and np.all(r["group_margin"] >= 0)
    # slots in descending choice score
    cs = np.take_along_axis(r["c"], idx.astype(np.int64), 1)
    assert np.all(np.diff(cs, axis=1) <= 0)


# ---------------------------------------------------------------- experts
def _torch_expert(x, wg, wu, wd):
    """Dense SwiGLU expert in float64 with the layer's rounding points,
    using torch's matmul and silu."""
    g = (x.double() @ wg.double().T).float().double()
    u = (x.double() @ wu.double().T).float().double()
    h = (torch.nn.functional.silu(g) * u).float().to(torch.bfloat16)
    return h.double() @ wd.double().T


def _tiny_weights(E, F, d):
    wg = _bf16_matrix((E, F, d), 0.02)
    wu = _bf16_matrix((E, F, d), 0.02)
    wd = _bf16_matrix((E, d, F), 0.02)
    return wg, wu, wd


def test_identical_experts_closed_form():
    T, d, F, E = 12, 128, 64, 16
    x = _bf16_matrix((T, d))
    wg, wu, wd = _tiny_weights(1, F, d)
    wg, wu, wd = (a.expand(E, *a.shape[1:]).contiguous() for a in (wg, wu, wd))
    lg = (RNG.standard_normal((T, E))).astype(np.float32)
    r = _route(lg, RNG.uniform(-0.05, 0.05, E), 8, 4, 4)
    out = oracle.experts_bf16(inputs.bf16_bits(x), r["idx"], r["w"], inputs.bf16_bits(wg),
                              inputs.bf16_bits(wu), inputs.bf16_bits(wd), E)
    y = _torch_expert(x, wg[0], wu[0], wd[0])
    ref = torch.from_numpy(bf16_nearest((2.5 * y).numpy()).view(np.int16)).view(torch.bfloat16)
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)
    # the weights sum to 2.5 up to FP32 rounding: at most one BF16 step apart
    diff = (got.float() - ref.float()).abs()
    assert torch.all(diff <= ref.float().abs() * 2 ** -7 + 1e-30)
    assert (got == ref).float().mean() > 0.97


def test_forced_routing_matches_dense_torch_experts():
    T, d, F, E, G = 10, 128, 64, 32, 8
    x = _bf16_matrix((T, d))
    wg, wu, wd = _tiny_weights(E, F, d)
    chosen = [1, 2, 9, 10, 17, 18, 30, 31]          # groups 0, 2, 4, 7 (S=4)
    bias = RNG.uniform(-0.05, 0.05, E).astype(np.float32)
    bias[chosen] += 10.0
    lg = oracle.router_logits(inputs.bf16_bits(x), (RNG.standard_normal((E, d)) / 12).astype(np.float32))
    r = _route(lg, bias, G, 4, 8)
    assert np.all(np.sort(r["idx"], 1) == chosen)
    out, ex = oracle.experts_bf16(inputs.bf16_bits(x), r["idx"], r["w"], inputs.bf16_bits(wg),
                                  inputs.bf16_bits(wu), inputs.bf16_bits(wd), E, exact=True)
    ref = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(8):
            e = int(r["idx"][t, j])
            ref[t] += float(r["w"][t, j]) * _torch_expert(x[t:t + 1], wg[e], wu[e], wd[e])[0]
    # the FP64 sums agree to rounding order; the output is their one BF16 rounding
    assert np.allclose(ex, ref.numpy(), rtol=1e-12, atol=1e-15)
    assert np.array_equal(out, bf16_nearest(ref.numpy()))


def test_output_is_one_rounding_of_the_exact_sum():
    """The layer output is the FP64 sum over the slots rounded once to BF16.
    Built so that each expert's down row is exactly 1 (h = 1: silu(64) * 2^-6
    rounds to 1 in FP32, and W_d picks h_0): the output is w_0 + w_1 exactly.
    With w = (1 + 2^-8, 2^-30) that sum lies just above the BF16 tie
    1 + 2^-8, so one rounding gives 1 + 2^-7; rounding to FP32 first would
    land on the tie and give 1.0.  The second token mirrors it below zero,
    the third is an exact tie (ties to even), the fourth needs no rounding."""
    d = F = 16
    E = 2
    x = torch.zeros(4, d, dtype=torch.bfloat16)
    x[:, 0] = 1.0
    wg = torch.zeros(E, F, d, dtype=torch.bfloat16)
    wu = torch.zeros(E, F, d, dtype=torch.bfloat16)
    wd = torch.zeros(E, d, F, dtype=torch.bfloat16)
    wg[:, :, 0] = 64.0
    wu[:, :, 0] = 2.0 ** -6
    wd[:, :, 0] = 1.0
    idx = np.tile(np.array([[0, 1]], np.int32), (4, 1))
    w = np.array([[1 + 2.0 ** -8, 2.0 ** -30], [-(1 + 2.0 ** -8), -(2.0 ** -30)],
                  [1 + 2.0 ** -8, 0.0], [1.5, 0.25]], np.float32)
    out, ex = oracle.experts_bf16(inputs.bf16_bits(x), idx, w, inputs.bf16_bits(wg),
                                  inputs.bf16_bits(wu), inputs.bf16_bits(wd), E, exact=True)
    assert np.array_equal(ex[:, 0], w.astype(np.float64).sum(1))
    assert np.all(out == out[:, :1])
    assert out[0, 0] == 0x3F81            # 1 + 2^-7
    assert out[1, 0] == 0xBF81            # -(1 + 2^-7)
    assert out[2, 0] == 0x3F80            # the tie 1 + 2^-8 goes to the even 1.0
    assert out[3, 0] == 0x3FE0            # 1.75, exact


def test_token_subset_matches_full_run():
    T, d, F, E = 9, 64, 32, 16
    x = _bf16_matrix((T, d))
    wg, wu, wd = _tiny_weights(E, F, d)
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 8, 4, 4)
    args = (inputs.bf16_bits(x), r["idx"], r["w"], inputs.bf16_bits(wg), inputs.bf16_bits(wu),
            inputs.bf16_bits(wd), E)
    full = oracle.experts_bf16(*args)
    sub = oracle.experts_bf16(*args, tokens=np.array([7, 2]))
    assert np.array_equal(sub[[2, 7]], full[[2, 7]])
    assert np.all(sub[[0, 1, 3, 4, 5, 6, 8]] == 0)


def test_nvfp4_weights_equal_bf16_when_exactly_representable():
    """E2M1 (2 significant bits) x E4M3 (4 bits) x a power of two fits BF16's
    8 bits exactly, so with BF16 activations both oracle paths agree bit for bit."""
    T, d, F, E = 6, 64, 32, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    gate, up, down, deq = {}, {}, {}, {}
    for name, (n, kk), dst in (("g", (F, d), gate), ("u", (F, d), up), ("d", (d, F), down)):
        q = RNG.integers(0, 256, (E, n, kk // 2), dtype=np.uint8)
        sf = RNG.integers(0x20, 0x48, (E, n, kk // 16), dtype=np.uint8)   # normal, modest scales
        gs = np.full(E, 2.0 ** -9, np.float32)
        dst.update(q=q, sf=sf, gs=gs)
        codes = np.stack([q & 15, q >> 4], -1).reshape(E, n, kk)
        val = np.vectorize(oracle.e2m1_value)(codes) * np.repeat(
            np.vectorize(oracle.e4m3_value)(sf), 16, axis=2) * 2.0 ** -9
        t = torch.from_numpy(val).to(torch.bfloat16)
        assert torch.equal(t.double(), torch.from_numpy(val))
        deq[name] = inputs.bf16_bits(t)
    a = oracle.experts_nvfp4(inputs.bf16_bits(x), r["idx"], r["w"], gate, up, down, E,
                             act_quant=False)
    b = oracle.experts_bf16(inputs.bf16_bits(x), r["idx"], r["w"], deq["g"], deq["u"], deq["d"], E)
    assert np.array_equal(a, b)


def test_nvfp4_generator_weights_round_trip_grid_values():
    """Weights already on an NVFP4 grid come back unchanged from the
    checkpoint quantiser the generator uses."""
    n, kk = 8, 64
    codes = torch.from_numpy(RNG.integers(0, 16, (n, kk)).astype(np.uint8))
    vals = torch.tensor([oracle.e2m1_value(int(c)) for c in codes.reshape(-1)]).reshape(n, kk)
    vals[:, ::16] = 6.0                   # every block hits the grid's top value
    w = (vals * 2.0 ** -6).float()
    q, sf, gs = inputs.quantize_nvfp4_weight(w)
    dec = np.stack([q.numpy() & 15, q.numpy() >> 4], -1).reshape(n, kk)
    back = np.vectorize(oracle.e2m1_value)(dec) * np.repeat(
        np.vectorize(oracle.e4m3_value)(sf.numpy()), 16, 1) * float(gs)
    assert np.allclose(back, w.double().numpy(), rtol=1e-6, atol=0)


# ------------------------------------------------- sublayer boundary (post-norm,
# depth-scaled residual add, next pre-norm)
def _bf16_value(bits):
    return np.asarray(bits, np.uint16).astype(np.uint32).__lshift__(16).view(np.float32) \
        .astype(np.float64)


def _rand_bf16(shape, scale=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return inputs.bf16_bits((torch.randn(*shape, generator=g) * scale).to(torch.bfloat16))


def _within_half_step(bits, ref):
    """bits (BF16) is a correct rounding of the float64 values ref."""
    v = _bf16_value(bits)
    _, e = np.frexp(np.abs(ref))
    half = np.where(ref == 0, 0.0, np.ldexp(1.0, e - 9))
    return np.all(np.abs(v - ref) <= half * (1 + 1e-12))


def test_bf16_round_double_is_one_correct_rounding():
    """Against exact rational arithmetic: the nearest BF16, ties to even."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(3000) * 7.0)
    # exact ties and values a hair above / below a tie
    for k in range(0x3f80, 0x3f80 + 40):
        lo = float(_bf16_value(np.uint16(k)))
        hi = float(_bf16_value(np.uint16(k + 1)))
        mid = (lo + hi) / 2
        vals += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    for v in vals:
        got = oracle.bf16_round_double(float(v))
        b32 = np.float32(v).view(np.uint32) >> np.uint32(16)
        cands = [int(b32) + j for j in (-1, 0, 1, 2) if 0 <= int(b32) + j < 0x7f80 or v < 0]
        best = min(cands, key=lambda c: (abs(Fraction(float(_bf16_value(np.uint16(c & 0xffff))))
                                             - Fraction(float(v))), c & 1))
        assert got == (best & 0xffff), (v, got, best)


def test_boundary_norms_match_torch_rms_norm():
    """n = 1: the residual add keeps only the post-normed branch (c_h = 0,
    c_x = 1), so h' is RMSNorm(m) and x is RMSNorm(h'): torch's rms_norm in
    FP64, each rounded once."""
    T, d, eps = 6, 512, 1e-6
    m = _rand_bf16((T, d), 3.0, seed=1)
    h = _rand_bf16((T, d), 1.0, seed=2)
    gp = _rand_bf16((d,), 0.3, seed=3)
    gq = _rand_bf16((d,), 0.3, seed=4)
    h_out, x_out = oracle.boundary(m, h, gp, gq, eps, 1)
    rms = torch.nn.functional.rms_norm
    ref_h = rms(torch.from_numpy(_bf16_value(m)), (d,), torch.from_numpy(_bf16_value(gp)),
                eps=eps).numpy()
    assert _within_half_step(h_out, ref_h)
    ref_x = rms(torch.from_numpy(_bf16_value(h_out)), (d,), torch.from_numpy(_bf16_value(gq)),
                eps=np.float32(eps).item()).numpy()
    assert _within_half_step(x_out, ref_x)


def test_boundary_residual_closed_forms():
    T, d, eps = 4, 256, 1e-6
    m = _rand_bf16((T, d), 1.0, seed=5)
    h = _rand_bf16((T, d), 1.0, seed=6)
    ones = inputs.bf16_bits(torch.ones(d, dtype=torch.bfloat16))
    p, _ = oracle.boundary(m, h, ones, ones, eps, 1)          # p = RMSNorm(m)
    # n = 4 with a zero stream: h' = p / 2 exactly (c_x = 1/2)
    h4, _ = oracle.boundary(m, np.zeros_like(h), ones, ones, eps, 4)
    assert np.array_equal(_bf16_value(h4), _bf16_value(p) / 2)
    # a zero branch: h' = round(fp32(sqrt(3/4)) * h)
    hz, _ = oracle.boundary(np.zeros_like(m), h, ones, ones, eps, 4)
    assert _within_half_step(hz, float(np.float32(math.sqrt(0.75))) * _bf16_value(h))


def test_boundary_is_odd():
    T, d = 3, 256
    m = _rand_bf16((T, d), 2.0, seed=7)
    h = _rand_bf16((T, d), 1.0, seed=8)
    g = _rand_bf16((d,), 0.5, seed=9)
    a = oracle.boundary(m, h, g, g, 1e-6, 7)
    b = oracle.boundary(m ^ np.uint16(0x8000), h ^ np.uint16(0x8000), g, g, 1e-6, 7)
    for x, y in zip(a, b):
        assert np.array_equal(x ^ np.uint16(0x8000), y)


def test_depth_scaled_residual_keeps_unit_variance():
    """The point of the depth scaling: unit-variance stream and branch give a
    unit-variance stream at every depth."""
    T, d = 64, 1024
    h = _rand_bf16((T, d), 1.0, seed=10)
    ones = inputs.bf16_bits(torch.ones(d, dtype=torch.bfloat16))
    for n in (2, 10, 104):
        m = _rand_bf16((T, d), 5.0, seed=11 + n)
        h_out, _ = oracle.boundary(m, h, ones, ones, 1e-6, n)
        assert abs(_bf16_value(h_out).var() - 1.0) < 0.03


# ------------------------------------------------ F16 activations (W4A16 path)
def test_f16_round_matches_torch():
    """binary32 values -> binary16 by torch (round to nearest even, with
    subnormals) inside the finite range; beyond it the reading saturates."""
    vals = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * np.float32(50.0),
        RNG.standard_normal(3000).astype(np.float32) * np.float32(1e-6),   # subnormal range
        # ties between neighbouring binary16 values at several exponents
        (np.arange(1024, 1064, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10),
        (np.arange(1, 40, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),
        np.array([0.0, -0.0, 65504.0, -65504.0, 65503.0, 6.1035156e-05], np.float32),
    ])
    got = np.array([oracle.f16_round(float(v)) for v in vals])
    ref = torch.from_numpy(vals).to(torch.float16).double().numpy()
    assert np.array_equal(got, ref)
    for v, want in ((65519.0, 65504.0), (70000.0, 65504.0), (-1e9, -65504.0)):
        assert oracle.f16_round(v) == want


def test_f16_activation_experts_match_dense_torch():
    """NVFP4 weights with F16 activations: the expert layer against a dense
    torch FP64 restatement that rounds x and the SwiGLU product with torch's
    own float16 casts."""
    T, d, F, E = 5, 64, 32, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        q = RNG.integers(0, 256, (E, n, kk // 2), dtype=np.uint8)
        sf = RNG.integers(0x20, 0x48, (E, n, kk // 16), dtype=np.uint8)
        gs = (RNG.uniform(0.5, 2.0, E) * 2.0 ** -8).astype(np.float32)
        proj[name] = dict(q=q, sf=sf, gs=gs)
        codes = np.stack([q & 15, q >> 4], -1).reshape(E, n, kk)
        deq[name] = torch.from_numpy(
            np.vectorize(oracle.e2m1_value)(codes)
            * np.repeat(np.vectorize(oracle.e4m3_value)(sf), 16, axis=2)
            * gs.astype(np.float64)[:, None, None])
    out, ex = oracle.experts_nvfp4(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"],
                                   proj["d"], E, act_quant=oracle.ACT_F16, exact=True)
    x16 = x.to(torch.float16).double()
    ref = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            g = (x16[t] @ deq["g"][e].T).float().double()
            u = (x16[t] @ deq["u"][e].T).float().double()
            h = (g / (1 + torch.exp(-g)) * u).float().to(torch.float16).double()
            ref[t] += float(r["w"][t, j]) * (h @ deq["d"][e].T)
    assert np.allclose(ex, ref.numpy(), rtol=1e-12, atol=1e-12)


def _nvfp4_torch_blocks(v: torch.Tensor) -> torch.Tensor:
    """The NVFP4 activation rule restated with torch: per 16 consecutive
    values, scale = float8_e4m3fn(amax / 6) (FP32 division, torch's
    round-to-nearest-even cast), codes by the independent E2M1 rounding of
    the generator on v / scale (FP32 division), zeros where the scale is 0;
    returns the dequantised values code * scale in float64."""
    vf = v.float().reshape(-1, 16)
    scale = (vf.abs().amax(dim=1) / 6.0).to(torch.float8_e4m3fn).float().unsqueeze(1)
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    codes = inputs._e2m1_codes(vf / safe)
    mag = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)
    val = mag[(codes & 7).long()] * torch.where(codes >= 8, -1.0, 1.0).double()
    val = torch.where(scale > 0, val * scale.double(), torch.zeros_like(val))
    return val.reshape(v.shape)


def test_nvfp4_activation_experts_match_dense_torch():
    """NVFP4 weights and NVFP4 activations (both GEMM inputs quantised per 16
    with global scale 1): the expert layer against a dense torch FP64
    restatement.  x is quantised along d from its BF16 values; the FP32
    SwiGLU product is quantised along F as it is, with no BF16 rounding first.
    Planting either plausible mistake in the oracle's block rule fails this
    test: rounding h to BF16 before quantising it, or taking the scale from
    amax / 4 instead of amax / 6."""
    T, d, F, E = 6, 64, 48, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        q = RNG.integers(0, 256, (E, n, kk // 2), dtype=np.uint8)
        sf = RNG.integers(0x20, 0x48, (E, n, kk // 16), dtype=np.uint8)
        gs = (RNG.uniform(0.5, 2.0, E) * 2.0 ** -6).astype(np.float32)
        proj[name] = dict(q=q, sf=sf, gs=gs)
        codes = np.stack([q & 15, q >> 4], -1).reshape(E, n, kk)
        deq[name] = torch.from_numpy(
            np.vectorize(oracle.e2m1_value)(codes)
            * np.repeat(np.vectorize(oracle.e4m3_value)(sf), 16, axis=2)
            * gs.astype(np.float64)[:, None, None])
    out, ex = oracle.experts_nvfp4(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"],
                                   proj["d"], E, act_quant=oracle.ACT_NVFP4, exact=True)
    xq = _nvfp4_torch_blocks(x.float())
    ref = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            g = (xq[t] @ deq["g"][e].T).float().double()
            u = (xq[t] @ deq["u"][e].T).float().double()
            hq = _nvfp4_torch_blocks((g / (1 + torch.exp(-g)) * u).float())
            ref[t] += float(r["w"][t, j]) * (hq @ deq["d"][e].T)
    assert np.allclose(ex, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, bf16_nearest(ref.numpy()))


def test_swiglu_rows_through_the_expert_layer():
    """One expert, weight 1 and an identity down projection: the expert
    layer's output is h itself (h is BF16, the identity sum is exact), so the
    standalone gate/up oracle must match the layer oracle bit for bit."""
    T, F = 9, 64
    d = F
    x = _bf16_matrix((T, d))
    wg = _bf16_matrix((1, F, d), 0.3)
    wu = _bf16_matrix((1, F, d), 0.3)
    eye = torch.eye(d, dtype=torch.bfloat16).reshape(1, d, F)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    layer = oracle.experts_bf16(inputs.bf16_bits(x), idx, w, inputs.bf16_bits(wg),
                                inputs.bf16_bits(wu), inputs.bf16_bits(eye), 1)
    h = oracle.swiglu_bf16(inputs.bf16_bits(x), inputs.bf16_bits(wg[0]), inputs.bf16_bits(wu[0]))
    assert np.array_equal(layer, h)


# ------------------------------------------------------------ dynamic FP8
def _fp8_torch_rows(x):
    """Per-row FP8 quantisation written with torch's own float8_e4m3fn cast
    (round to nearest even) for the rounding step."""
    xf = x.float()
    amax = xf.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (xf / scale.unsqueeze(1)).to(torch.float8_e4m3fn)
    return q, scale


def test_fp8_row_quantizer_vs_torch():
    n, cols = 40, 96
    mag = np.exp(RNG.uniform(-12, 6, n))[:, None]
    x = torch.from_numpy((RNG.standard_normal((n, cols)) * mag).astype(np.float32))
    x[3] = 0.0                                    # an all-zero row: scale 1, codes 0
    x[4, :] = 1.0
    x[4, 0] = -2.0                                # exact grid values, amax -> -448
    x = x.to(torch.bfloat16)
    q, sc = oracle.fp8_quantize_rows(inputs.bf16_bits(x))
    q_ref, sc_ref = _fp8_torch_rows(x)
    assert np.array_equal(sc, sc_ref.numpy())
    assert np.array_equal(q, q_ref.view(torch.uint8).numpy())
    assert sc[3] == 1.0 and not q[3].any()
    assert q[4, 0] == 0xFE and np.all(q[4, 1:] == 0x76)         # -448 and 224
    # the element of largest magnitude always lands on +-448
    big = np.abs(x.float().numpy()).argmax(axis=1)
    for i in range(n):
        if i != 3:
            assert q[i, big[i]] & 0x7F == 0x7E


def test_fp8_generator_weights_round_trip_grid_values():
    """Rows already on an E4M3 grid (one power-of-two scale per row, each row
    reaching 448) come back unchanged from the checkpoint quantiser."""
    n, kk = 8, 64
    codes = RNG.integers(0, 127, (n, kk)) | (RNG.integers(0, 2, (n, kk)) << 7)
    vals = np.vectorize(oracle.e4m3_value)(codes)
    vals[:, 0] = 448.0
    w = torch.from_numpy(vals * (2.0 ** RNG.integers(-12, -4, n))[:, None]).float()
    q, s = inputs.quantize_fp8_weight(w)
    back = np.vectorize(oracle.e4m3_value)(q.numpy()) * s.double().numpy()[:, None]
    assert np.array_equal(back, w.double().numpy())


def _fp8_weights(E, n, kk, pow2_scales):
    codes = (RNG.integers(0, 127, (E, n, kk)) | (RNG.integers(0, 2, (E, n, kk)) << 7))
    codes = codes.astype(np.uint8)
    if pow2_scales:
        s = (2.0 ** RNG.integers(-12, -6, (E, n))).astype(np.float32)
    else:
        s = (RNG.uniform(0.5, 2.0, (E, n)) * 2.0 ** -10).astype(np.float32)
    deq = np.vectorize(oracle.e4m3_value)(codes) * s.astype(np.float64)[:, :, None]
    return {"q": codes, "s": s}, torch.from_numpy(deq)


def test_fp8_weights_equal_bf16_when_exactly_representable():
    """An E4M3 value (4 significant bits) times a power of two is a BF16
    value, so with BF16 activations the FP8 and BF16 oracle paths agree bit
    for bit: this pins the weight decoding (codes and row scales)."""
    T, d, F, E = 6, 64, 32, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], full = _fp8_weights(E, n, kk, pow2_scales=True)
        t = full.to(torch.bfloat16)
        assert torch.equal(t.double(), full)
        deq[name] = inputs.bf16_bits(t)
    a = oracle.experts_fp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"], proj["d"],
                           E, act_quant=False)
    b = oracle.experts_bf16(inputs.bf16_bits(x), r["idx"], r["w"], deq["g"], deq["u"], deq["d"], E)
    assert np.array_equal(a, b)


def test_fp8_activation_experts_match_dense_torch():
    """FP8 weights and per-row FP8 activations: the expert layer against a
    dense torch FP64 restatement that quantises x and the BF16 h rows with
    torch's float8_e4m3fn cast."""
    T, d, F, E = 5, 64, 32, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], deq[name] = _fp8_weights(E, n, kk, pow2_scales=False)
    out, ex = oracle.experts_fp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"],
                                 proj["d"], E, act_quant=True, exact=True)
    qx, sx = _fp8_torch_rows(x)
    xh = qx.double() * sx.double().unsqueeze(1)
    ref = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            g = (xh[t] @ deq["g"][e].T).float().double()
            u = (xh[t] @ deq["u"][e].T).float().double()
            h = (g / (1 + torch.exp(-g)) * u).float().to(torch.bfloat16)
            qh, sh = _fp8_torch_rows(h.unsqueeze(0))
            hh = qh.double()[0] * float(sh[0])
            ref[t] += float(r["w"][t, j]) * (hh @ deq["d"][e].T)
    assert np.allclose(ex, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, bf16_nearest(ref.numpy()))


# ------------------------------------------------- near-tie routings and h codes
def _tie_heavy_scores(T, E, tol, seed):
    """Logits and a bias that put every token's choice scores c = s + b on a
    grid of spacing 0.3 tol in a narrow band (about an eighth of the levels
    taken), so the group and expert cuts often fall inside short runs of
    scores closer than tol."""
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    s = (1.0 / (1.0 + np.exp(-lg.astype(np.float64)))).astype(np.float32)
    target = 0.5 + rng.integers(0, 8 * E, (T, E)) * (0.3 * tol)
    return lg, s, target


def test_route_alternatives_without_ties_is_the_routing():
    """tol = 0: the oracle's own routing, weights bit for bit."""
    T, E, G, kg, k = 40, 64, 8, 4, 8
    lg = RNG.standard_normal((T, E)).astype(np.float32)
    r = _route(lg, RNG.uniform(-0.05, 0.05, E).astype(np.float32), G, kg, k)
    for t in range(T):
        alts = oracle.route_alternatives(r, t, G, kg, k, 2.5, 0.0)
        assert len(alts) == 1
        assert np.array_equal(alts[0]["idx"], r["idx"][t])
        assert np.array_equal(alts[0]["w"], r["w"][t])


@pytest.mark.parametrize("E,G,kg,k", [(16, 4, 2, 3), (32, 8, 4, 5), (64, 8, 4, 8)])
def test_route_alternatives_cover_perturbed_selections(E, G, kg, k):
    """Perturbing every choice score by less than tol / 5 (through the bias)
    can only reorder scores closer than tol: each routing the selection then
    returns must be among the alternatives listed from the unperturbed
    scores (same expert set, same weights per expert).  The list is the
    oracle's own routing first; it may hold more than perturbations reach
    (a run of scores each closer than tol to the next is taken whole)."""
    tol = 3e-6
    T = 12
    lg, s, target = _tie_heavy_scores(T, E, tol, seed=E + k)
    rng = np.random.default_rng(7)
    moved = []
    for t in range(T):
        bias = (target[t] - s[t]).astype(np.float32)
        r = _route(lg[t:t + 1], bias, G, kg, k)
        alts = oracle.route_alternatives(r, 0, G, kg, k, 2.5, tol)
        sets = [frozenset(a["idx"].tolist()) for a in alts]
        assert len(set(sets)) == len(sets)
        reached = set()
        for _ in range(200):
            pb = (bias + rng.uniform(-tol / 5, tol / 5, E)).astype(np.float32)
            rp = _route(lg[t:t + 1], pb, G, kg, k)
            key = frozenset(rp["idx"][0].tolist())
            assert key in sets, (t, sorted(key))
            a = alts[sets.index(key)]
            wa = dict(zip(a["idx"].tolist(), a["w"].tolist()))
            for e, wv in zip(rp["idx"][0].tolist(), rp["w"][0].tolist()):
                assert abs(wa[e] - wv) <= 1e-6 * abs(wv)
            reached.add(key)
        assert sets[0] == frozenset(r["idx"][0].tolist())
        assert np.array_equal(alts[0]["idx"], r["idx"][0]) and np.array_equal(alts[0]["w"], r["w"][0])
        moved.append(len(reached))
    assert max(moved) > 1                # the tie-heavy scores do move the selection


def test_fp8_near_tie_slack_matches_torch_restatement():
    """The near ties the FP8 oracle reports, restated with torch: per (token,
    expert) row the FP32 h, its BF16 rounding, the next BF16 value on its
    side and their midpoint; an element within rel * |h| of the midpoint
    whose E4M3 code (row scale from the BF16 row) differs between the two
    BF16 values adds |w * (code change) * W_d[., f]| to every output of its
    token; one whose BF16 value or neighbour reaches the row's amax flags the
    token instead.  A large rel gives many ties.  Forcing one tie to the
    neighbour in the dense restatement moves the output by exactly that
    element's share."""
    T, d, F, E = 5, 64, 48, 8
    rel = 2.0 ** -9
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], deq[name] = _fp8_weights(E, n, kk, pow2_scales=False)
    out, ex, slack, flag = oracle.experts_fp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"],
                                              proj["u"], proj["d"], E, act_quant=True,
                                              ties=True, tie_rel=rel)
    qx, sx = _fp8_torch_rows(x)
    xh = qx.double() * sx.double().unsqueeze(1)
    want = torch.zeros(T, d, dtype=torch.float64)
    want_flag = np.zeros(T, bool)
    n_ties = 0
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            wt = float(r["w"][t, j])
            g = (xh[t] @ deq["g"][e].T).float().double()
            u = (xh[t] @ deq["u"][e].T).float().double()
            hf = (g / (1 + torch.exp(-g)) * u).float()
            hb = hf.to(torch.bfloat16)
            bits = hb.view(torch.int16).int() & 0x7FFF
            up = hf.double().abs() > hb.double().abs()
            nbits = torch.where(up, bits + 1, bits - 1) | torch.where(hf < 0, 0x8000, 0)
            nb = nbits.to(torch.int16).view(torch.bfloat16)
            near = ((hf.double() - (hb.double() + nb.double()) / 2).abs()
                    <= rel * hf.double().abs()) & (hf.double() != hb.double())
            amax = hb.float().abs().max()
            scale = amax / 448.0 if amax > 0 else torch.tensor(1.0)
            at_amax = near & ((nb.double().abs() >= float(amax)) |
                              (hb.double().abs() == float(amax)))
            if at_amax.any():
                want_flag[t] = True
            qb = (hb.float() / scale).to(torch.float8_e4m3fn).double() * float(scale)
            qn = (nb.float() / scale).to(torch.float8_e4m3fn).double() * float(scale)
            moves = near & ~at_amax & (qb != qn)
            for f in torch.nonzero(moves).reshape(-1).tolist():
                n_ties += 1
                share = wt * float(qn[f] - qb[f]) * deq["d"][e][:, f]
                want[t] += share.abs()
                if n_ties == 1:        # force this one tie in the dense restatement
                    h_alt = hb.clone()
                    h_alt[f] = nb[f]
                    qh, sh = _fp8_torch_rows(h_alt.unsqueeze(0))
                    qh0, sh0 = _fp8_torch_rows(hb.unsqueeze(0))
                    assert float(sh[0]) == float(sh0[0])
                    moved = wt * ((qh.double()[0] * float(sh[0]) - qh0.double()[0] * float(sh0[0]))
                                  @ deq["d"][e].T)
                    assert torch.allclose(moved, share, rtol=1e-12, atol=1e-18)
    assert n_ties > 0
    assert np.array_equal(flag, want_flag)
    assert np.allclose(slack, want.numpy(), rtol=1e-12, atol=1e-18)


# ------------------------------------------------------------------ MXFP8
def test_e8m0_all_256_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
    ref = ref.double().numpy()
    for c in range(256):
        v = oracle.e8m0_value(c)
        assert (math.isnan(v) and math.isnan(ref[c])) or v == ref[c], (c, v, ref[c])


def _mx_torch(v: torch.Tensor):
    """The MX conversion restated with torch (OCP MX v1.0, E4M3 elements):
    per 32 values X = floor(log2(amax)) - 8 from torch.frexp, clamped to
    [-127, 127] (-127 for an all-zero block); elements by torch's
    float8_e4m3fn cast of v * 2^-X after clamping to +-448.  Returns (codes,
    scale codes, dequantised float64 values)."""
    b = v.float().reshape(-1, 32)
    amax = b.abs().amax(dim=1)
    _, e = torch.frexp(amax)
    x = torch.where(amax > 0, e - 1 - 8, torch.full_like(e, -127)).clamp(-127, 127)
    q = torch.ldexp(b, -x.unsqueeze(1).float()).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    deq = q.double() * torch.ldexp(torch.ones_like(x, dtype=torch.float64), x.double()).unsqueeze(1)
    return q.view(torch.uint8).reshape(-1), (x + 127).to(torch.uint8), deq.reshape(v.shape)


def test_mx_activation_quantizer_vs_torch():
    v = (RNG.standard_normal(32 * 600) * np.repeat(np.exp(RNG.uniform(-20, 12, 600)), 32))
    v = v.astype(np.float32)
    v[:32] = 0.0                                   # all-zero block
    v[32:64] = 1.0
    v[32] = 1.999                                  # 1.999 / 2^-8 = 511.7: saturates at 448
    v[64:96] = np.float32(2.0 ** -140)             # below E8M0's range: X clamps to -127
    q, sc = oracle.mx_quantize(v)
    qr, scr, _ = _mx_torch(torch.from_numpy(v))
    assert np.array_equal(sc, scr.numpy())
    dec = np.array([oracle.e4m3_value(int(c)) for c in q])
    decr = np.array([oracle.e4m3_value(int(c)) for c in qr.numpy()])
    assert np.array_equal(dec, decr)
    assert sc[1] == 127 - 8 and dec[32] == 448.0
    assert sc[2] == 0


def test_mxfp8_generator_weights_round_trip_grid_values():
    """Weights already on an MXFP8 grid (E4M3 values times a power of two per
    32, each block reaching 448) come back unchanged from the generator's
    quantiser."""
    n, kk = 6, 128
    codes = RNG.integers(0, 127, (n, kk)) | (RNG.integers(0, 2, (n, kk)) << 7)
    vals = np.vectorize(oracle.e4m3_value)(codes)
    vals[:, ::32] = 448.0
    scale = 2.0 ** RNG.integers(-20, -5, (n, kk // 32))
    w = torch.from_numpy(vals * np.repeat(scale, 32, axis=1)).float()
    q, s = inputs.quantize_mxfp8_weight(w)
    back = np.vectorize(oracle.e4m3_value)(q.numpy()) * np.repeat(
        np.vectorize(oracle.e8m0_value)(s.numpy()), 32, axis=1)
    assert np.array_equal(back, w.double().numpy())


def _mx_weights(E, n, kk):
    codes = (RNG.integers(0, 127, (E, n, kk)) | (RNG.integers(0, 2, (E, n, kk)) << 7))
    codes = codes.astype(np.uint8)
    sc = RNG.integers(127 - 14, 127 - 8, (E, n, kk // 32)).astype(np.uint8)
    deq = np.vectorize(oracle.e4m3_value)(codes) * np.repeat(
        np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=2)
    return {"q": codes, "s": sc}, torch.from_numpy(deq)


def test_mxfp8_weights_equal_bf16_when_exactly_representable():
    """E4M3 values (4 significant bits) times a power of two are BF16 values,
    so with BF16 activations the MXFP8 and BF16 oracle paths agree bit for
    bit: this pins the weight decoding (codes and per-32 scales)."""
    T, d, F, E = 6, 64, 64, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], full = _mx_weights(E, n, kk)
        t = full.to(torch.bfloat16)
        assert torch.equal(t.double(), full)
        deq[name] = inputs.bf16_bits(t)
    a = oracle.experts_mxfp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"],
                             proj["d"], E, act_quant=False)
    b = oracle.experts_bf16(inputs.bf16_bits(x), r["idx"], r["w"], deq["g"], deq["u"], deq["d"], E)
    assert np.array_equal(a, b)


def test_mxfp8_activation_experts_match_dense_torch():
    """MXFP8 weights and MX activations: the expert layer against a dense
    torch FP64 restatement that quantises x (from BF16) and the FP32 SwiGLU
    product (no BF16 rounding first) with _mx_torch.  Planting a BF16
    rounding of h, or E4M3's largest exponent 7 instead of 8, fails it."""
    T, d, F, E = 5, 64, 64, 8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], deq[name] = _mx_weights(E, n, kk)
    out, ex = oracle.experts_mxfp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"], proj["u"],
                                   proj["d"], E, act_quant=True, exact=True)
    xq = _mx_torch(x.float().reshape(-1))[2].reshape(T, d)
    ref = torch.zeros(T, d, dtype=torch.float64)
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            g = (xq[t] @ deq["g"][e].T).float().double()
            u = (xq[t] @ deq["u"][e].T).float().double()
            hq = _mx_torch((g / (1 + torch.exp(-g)) * u).float())[2]
            ref[t] += float(r["w"][t, j]) * (hq @ deq["d"][e].T)
    assert np.allclose(ex, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, bf16_nearest(ref.numpy()))


def test_mxfp8_near_tie_slack_matches_torch_restatement():
    """The MX h near ties restated with torch: an element whose scaled FP32
    value lies within rel of the midpoint between its E4M3 value and the next
    one on its side adds |w * (value change) * W_d[., f]| to its token's
    outputs; a block whose amax lies within rel of a power of two flags the
    token."""
    T, d, F, E = 5, 64, 64, 8
    rel = 2.0 ** -8
    x = _bf16_matrix((T, d))
    r = _route(RNG.standard_normal((T, E)), np.zeros(E), 4, 2, 3)
    proj, deq = {}, {}
    for name, (n, kk) in (("g", (F, d)), ("u", (F, d)), ("d", (d, F))):
        proj[name], deq[name] = _mx_weights(E, n, kk)
    out, ex, slack, flag = oracle.experts_mxfp8(inputs.bf16_bits(x), r["idx"], r["w"], proj["g"],
                                                proj["u"], proj["d"], E, act_quant=True,
                                                ties=True, tie_rel=rel)
    mags = torch.tensor([oracle.e4m3_value(c) for c in range(127)], dtype=torch.float64)
    xq = _mx_torch(x.float().reshape(-1))[2].reshape(T, d)
    want = torch.zeros(T, d, dtype=torch.float64)
    want_flag = np.zeros(T, bool)
    n_ties = 0
    for t in range(T):
        for j in range(3):
            e = int(r["idx"][t, j])
            g = (xq[t] @ deq["g"][e].T).float().double()
            u = (xq[t] @ deq["u"][e].T).float().double()
            hf = (g / (1 + torch.exp(-g)) * u).float()
            codes, sc, _ = _mx_torch(hf)
            for b in range(F // 32):
                blk = hf[32 * b:32 * (b + 1)].double()
                amax = float(blk.abs().max())
                m, _ = math.frexp(amax)
                if amax > 0 and (m - 0.5 <= rel * m or 1.0 - m <= rel * m):
                    want_flag[t] = True
                xs = 2.0 ** (int(sc[b]) - 127)
                for i in range(32):
                    f = 32 * b + i
                    rr = abs(float(blk[i])) / xs
                    c = int(codes[f]) & 0x7F
                    vc = float(mags[c])
                    if rr == 0 or rr >= 448 or rr == vc:
                        continue
                    nb = c + 1 if rr > vc else c - 1
                    if not 0 <= nb <= 126:
                        continue
                    vn = float(mags[nb])
                    if abs(rr - (vc + vn) / 2) <= rel * rr:
                        n_ties += 1
                        sgn = -1.0 if float(blk[i]) < 0 else 1.0
                        want[t] += (float(r["w"][t, j]) * sgn * (vn - vc) * xs
                                    * deq["d"][e][:, f]).abs()
    assert n_ties > 0
    assert np.array_equal(flag, want_flag)
    assert np.allclose(slack, want.numpy(), rtol=1e-12, atol=1e-18)
