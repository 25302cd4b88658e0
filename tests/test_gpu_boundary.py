"""GPU parity of the layer fused with the decoder's sublayer boundary
(post-norm, depth-scaled residual add, next pre-norm in the combine kernel)
against the CPU oracle.  Each step is checked from the GPU's own input to it,
so a difference can only come from FP32-versus-FP64 arithmetic before a BF16
rounding: one BF16 step of a rounded value, and rarely.  The residual add
h' = bf16(a + b) of two rounded operands can cancel, so there the bound is one
step of each operand plus one of h': |dh'| <= 2^-7 (|a| + |b|) + step(h')."""
import numpy as np
import pytest
import torch

import oracle
import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _bits(t):
    return inputs.bf16_bits(t)


def _value(bits):
    return bits.astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def _step(bits):
    """One BF16 step at each value (8 significant bits)."""
    v = np.abs(_value(bits))
    _, e = np.frexp(v)
    return np.where(v == 0, 2.0 ** -133, np.ldexp(1.0, e - 8))


def _steps_apart(a, b):
    """BF16 steps between two bit patterns of the same sign (ordered ints)."""
    ia = a.astype(np.int32)
    ib = b.astype(np.int32)
    ia = np.where(ia & 0x8000, 0x8000 - ia, ia)
    ib = np.where(ib & 0x8000, 0x8000 - ib, ib)
    return np.abs(ia - ib)


def _weights(t, fmt):
    names = ("w_gate", "w_up", "w_down")
    if fmt == "bf16":
        return [t[n] for n in names]
    if fmt == "fp8":
        return [pkg.Fp8Weight.of(t[n]) for n in names]
    if fmt == "mxfp8":
        return [pkg.Mxfp8Weight.of(t[n]) for n in names]
    return [pkg.Fp4Weight.of(t[n]) for n in names]


def _plain(cfg, t, fmt, wts):
    args = (cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts)
    return {"bf16": pkg.forward, "fp8": pkg.forward_fp8, "nvfp4": pkg.forward_nvfp4,
            "a16": pkg.forward_nvfp4_a16, "mxfp8": pkg.forward_mxfp8}[fmt](*args)


def _check(cfg, t, n, seed, fmt="bf16"):
    """The boundary call's m is the plain layer call's, bit for bit (the same
    expert kernels and combine order, whatever the expert format); h' and the
    next input are checked from the GPU's m against the oracle."""
    T, d = t["hidden"].shape
    g = torch.Generator(device="cuda").manual_seed(seed)
    h0 = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    gp = (1 + 0.1 * torch.randn(d, generator=g, device="cuda")).to(torch.bfloat16)
    gq = (1 + 0.1 * torch.randn(d, generator=g, device="cuda")).to(torch.bfloat16)
    res = h0.clone()
    wts = _weights(t, fmt)
    out, nx = pkg.forward_boundary(cfg, t["hidden"], t["router_w"], t["corr_bias"], *wts, res, gp,
                                   gq, EPS, n, a16=fmt == "a16")
    ref_out = _plain(cfg, t, fmt, wts)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))   # the same combine
    # new residual from the GPU's m and the old stream
    h_ref, _ = oracle.boundary(_bits(out), _bits(h0), _bits(gp), _bits(gq), EPS, n)
    p_ref, _ = oracle.boundary(_bits(out), _bits(h0), _bits(gp), _bits(gq), EPS, 1)
    c_h, c_x = oracle.residual_coefficients(n)
    scale = np.abs(float(c_h) * _value(_bits(h0))) + np.abs(float(c_x) * _value(p_ref))
    err = np.abs(_value(_bits(res)) - _value(h_ref))
    assert np.all(err <= 2.0 ** -7 * scale + _step(h_ref)), float((err / scale).max())
    dh = _steps_apart(_bits(res), h_ref)
    # next input from the GPU's new residual (n = 1 keeps only the normed branch)
    x_ref, _ = oracle.boundary(_bits(res), _bits(h0), _bits(gq), _bits(gq), EPS, 1)
    dx = _steps_apart(_bits(nx), x_ref)
    assert dx.max() <= 1, dx.max()
    assert (dh > 0).mean() < 0.01 and (dx > 0).mean() < 0.01, ((dh > 0).mean(), (dx > 0).mean())
    return res, nx


@pytest.mark.parametrize("T,n", [(64, 1), (64, 2), (37, 57), (300, 104)])
def test_boundary_matches_oracle(T, n):
    """T = 300 takes the unfused routing and the 256-token expert tiles."""
    cfg = inputs.CONFIGS["tiny"].replace(T=T, seed=90 + T)
    t = inputs.generate(cfg, "cuda")
    _check(cfg, t, n, seed=T + n)


def test_boundary_is_deterministic():
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cuda")
    a = _check(cfg, t, 9, seed=1)
    b = _check(cfg, t, 9, seed=1)
    assert all(torch.equal(x.view(torch.int16), y.view(torch.int16)) for x, y in zip(a, b))


def test_boundary_beam_decode():
    cfg = inputs.CONFIGS["decode"]
    t = inputs.generate(cfg, "cuda")
    _check(cfg, t, 40, seed=3)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "a16", "mxfp8"])
@pytest.mark.parametrize("T,n", [(20, 2), (70, 33)])
def test_boundary_after_quantised_experts(fmt, T, n):
    """The NVFP4, W4A16, FP8 and MXFP8 layers end in the same FP32 expert rows and
    the same combine kernel: T = 20 takes the 16-row token blocks, T = 70
    the 256-row ones (T * topk > 4 * E)."""
    d = 256 if fmt in ("nvfp4", "a16", "mxfp8") else 128
    cfg = inputs.MoEConfig(name=f"bnd_{fmt}", T=T, d=d, d_ff=d, seed=40 + T,
                           weight_fmt="nvfp4" if fmt == "a16" else fmt, n_experts=32, n_groups=4,
                           topk_groups=2, topk=4, routed_scale=2.5)
    t = inputs.generate(cfg, "cuda")
    _check(cfg, t, n, seed=T + n, fmt=fmt)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_boundary_quantised_beam_shapes(fmt):
    """Beam expert shapes with the decode batches of the two quantised
    checkpoint formats."""
    cfg = inputs.CONFIGS[fmt]
    t = inputs.generate(cfg, "cuda")
    _check(cfg, t, 12, seed=5, fmt=fmt)


def test_boundary_rejects_bad_arguments():
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cuda", T=4)
    res = torch.zeros(4, cfg.d, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(cfg.d, dtype=torch.bfloat16, device="cuda")
    for n, eps in ((0, EPS), (3, -1.0)):
        with pytest.raises(pkg.BeamError) as e:
            pkg.forward_boundary(cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"],
                                 t["w_up"], t["w_down"], res, g, g, eps, n)
        assert e.value.code == 1
