"""Seeded synthetic inputs for the Beam MoE layer.

This module only draws numbers: it holds none of the layer's arithmetic.  Both
the CUDA path (tests, bench) and the CPU oracle consume what it produces.

Shapes follow the Beam layer as the pages describe it (vLLM post, section "MoE
and residual stream": hidden 5120, 256 experts in 8 groups, best 4 groups,
top 8, d_ff 2560, scale 2.5; HF release post, section "专家混合": 32 experts per
group).  Distributions: hidden ~ N(0, 1) in BF16; router W_r ~ N(0, 1/d) in
FP32 stored [E, d]; correction bias ~ U(-0.05, 0.05) in FP32; expert weights
~ N(0, 0.02^2) in BF16 stored W_gate/W_up [E, F, d] and W_down [E, d, F]
(NVFP4, FP8 and MXFP8 expert weights are those draws quantised once, here:
they are the checkpoint both sides read).
Draw order: hidden, router_w, corr_bias, [skewed experts], w_gate, w_up,
w_down, one torch.Generator seeded per configuration.  The small configuration
is drawn on the CPU generator (so any machine reproduces it); the Beam-sized
ones on the device's generator, expert by expert.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    n_experts: int
    n_groups: int
    topk_groups: int
    topk: int
    d_ff: int
    routed_scale: float = 2.5
    seed: int = 0
    weight_fmt: str = "bf16"          # "bf16", "nvfp4", "fp8" or "mxfp8"
    skew_experts: int = 0             # experts that get +skew_bias
    skew_bias: float = 0.0
    cpu_generator: bool = False       # draw on the CPU generator
    description: str = ""

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


_BEAM = dict(d=5120, n_experts=256, n_groups=8, topk_groups=4, topk=8, d_ff=2560,
             routed_scale=2.5)

CONFIGS = {
    "tiny": MoEConfig(name="tiny", T=64, d=512, n_experts=64, n_groups=8, topk_groups=4,
                      topk=8, d_ff=256, seed=0, cpu_generator=True,
                      description="tiny MoE layer T=64 d=512 E=64 (8x8) top-4 groups "
                                  "top-8 d_ff=256"),
    "decode": MoEConfig(name="decode", T=32, seed=1, **_BEAM,
                        description="Beam MoE layer decode batch T=32 d=5120 E=256 "
                                    "(8x32) top-4 groups top-8 d_ff=2560 BF16 experts"),
    "prefill": MoEConfig(name="prefill", T=8192, seed=2, **_BEAM,
                         description="Beam MoE layer prefill chunk T=8192, Beam shapes, "
                                     "BF16 experts"),
    "skewed": MoEConfig(name="skewed", T=4096, seed=3, skew_experts=16, skew_bias=2.0,
                        **_BEAM,
                        description="Beam MoE layer skewed routing T=4096, bias +2.0 on "
                                    "16 random experts"),
    # profiling case: the Beam expert shapes with 32 experts (2.5 GB held on
    # the device, more than 1 GB of gate/up weights streamed per call)
    "profile_small": MoEConfig(name="profile_small", T=8, d=5120, n_experts=32, n_groups=8,
                               topk_groups=4, topk=8, d_ff=2560, seed=5,
                               description="Beam expert shapes, 32 experts (8x4), T=8 "
                                           "(profiling case)"),
    # profiling case for the compute-bound regime: 32 experts, 256 rows each
    # on average (the Beam prefill's rows per expert), 2.5 GB on the device
    "profile_prefill": MoEConfig(name="profile_prefill", T=1024, d=5120, n_experts=32,
                                 n_groups=8, topk_groups=4, topk=8, d_ff=2560, seed=6,
                                 description="Beam expert shapes, 32 experts (8x4), T=1024 "
                                             "(profiling case, prefill regime)"),
    # profiling case for the NVFP4 kernels: 32 experts, decode-sized batch
    "profile_fp4": MoEConfig(name="profile_fp4", T=16, d=5120, n_experts=32, n_groups=8,
                             topk_groups=4, topk=8, d_ff=2560, seed=8, weight_fmt="nvfp4",
                             description="Beam expert shapes, 32 NVFP4 experts (8x4), T=16 "
                                         "(profiling case)"),
    "nvfp4": MoEConfig(name="nvfp4", T=128, seed=4, weight_fmt="nvfp4", **_BEAM,
                       description="Beam MoE layer NVFP4 experts T=128 (E2M1 + E4M3 per "
                                   "16 along K + FP32 per-tensor scale)"),
    "fp8": MoEConfig(name="fp8", T=32, seed=9, weight_fmt="fp8", **_BEAM,
                     description="Beam MoE layer decode batch T=32, dynamic FP8 experts "
                                 "(E4M3 weights with one FP32 scale per output row; "
                                 "activations quantised per row at run time)"),
    "fp8_prefill": MoEConfig(name="fp8_prefill", T=8192, seed=10, weight_fmt="fp8", **_BEAM,
                             description="Beam MoE layer prefill chunk T=8192, dynamic FP8 "
                                         "experts"),
    # profiling case for the FP8 kernels in the prefill regime: 32 experts,
    # 256 rows each on average
    "profile_fp8_prefill": MoEConfig(name="profile_fp8_prefill", T=1024, d=5120, n_experts=32,
                                     n_groups=8, topk_groups=4, topk=8, d_ff=2560, seed=12,
                                     weight_fmt="fp8",
                                     description="Beam expert shapes, 32 FP8 experts (8x4), "
                                                 "T=1024 (profiling case, prefill regime)"),
    "mxfp8": MoEConfig(name="mxfp8", T=32, seed=13, weight_fmt="mxfp8", **_BEAM,
                       description="Beam MoE layer decode batch T=32, MXFP8 experts (E4M3 "
                                   "weights and activations, one E8M0 scale per 32 along K)"),
    # profiling case for the MXFP8 kernels: 32 experts, decode-sized batch
    "profile_mxfp8": MoEConfig(name="profile_mxfp8", T=8, d=5120, n_experts=32, n_groups=8,
                               topk_groups=4, topk=8, d_ff=2560, seed=15, weight_fmt="mxfp8",
                               description="Beam expert shapes, 32 MXFP8 experts (8x4), T=8 "
                                           "(profiling case)"),
    # profiling case for the FP8 kernels: 32 experts, decode-sized batch
    "profile_fp8": MoEConfig(name="profile_fp8", T=8, d=5120, n_experts=32, n_groups=8,
                             topk_groups=4, topk=8, d_ff=2560, seed=11, weight_fmt="fp8",
                             description="Beam expert shapes, 32 FP8 experts (8x4), T=8 "
                                         "(profiling case)"),
}


def _gen(cfg: MoEConfig, device) -> tuple[torch.Generator, torch.device]:
    dev = torch.device("cpu") if cfg.cpu_generator else torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(cfg.seed)
    return g, dev


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round to the nearest E2M1 value, ties to the even code, saturating at 6;
    returns 4-bit codes (bit 3 = sign).  Checkpoint-format preparation."""
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=v.device)
    a = v.abs().clamp(max=6.0)
    mid = (grid[1:] + grid[:-1]) / 2
    lo = torch.bucketize(a, mid, right=False)          # a <= mid -> lower bucket
    # exact midpoints: bucketize(right=False) puts them in the lower code;
    # move to the upper code when the upper one is even.
    at_mid = torch.isin(a, mid)
    upper_even = ((lo + 1) % 2 == 0)
    code = torch.where(at_mid & upper_even, lo + 1, lo)
    sign = (v < 0) | ((v == 0) & torch.signbit(v))
    return (code + 8 * sign.to(code.dtype)).to(torch.uint8)


def quantize_nvfp4_weight(w: torch.Tensor):
    """One expert projection [N, K] (float32) -> (packed codes uint8 [N, K/2],
    E4M3 block scales uint8 [N, K/16], FP32 global scale).  The global scale
    maps the tensor's amax onto 6 * 448; each block of 16 along K gets the E4M3
    scale of its own amax.  Two codes per byte, low nibble = even column."""
    N, K = w.shape
    amax = w.abs().max().float()
    gs = (amax / (6.0 * 448.0)).clamp(min=1e-30)
    blk = w.reshape(N, K // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    sf8 = (bmax / (6.0 * gs)).clamp(max=448.0).to(torch.float8_e4m3fn)
    sf_val = sf8.float()
    denom = (sf_val * gs).unsqueeze(-1)
    scaled = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)),
                         torch.zeros_like(blk))
    codes = _e2m1_codes(scaled).reshape(N, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return packed, sf8.view(torch.uint8).contiguous(), gs.reshape(1)


def quantize_fp8_weight(w: torch.Tensor):
    """One expert projection [N, K] (float32) -> (E4M3 codes uint8 [N, K], FP32
    scale per row [N]).  Each output row (channel) maps its amax onto 448, the
    largest finite E4M3 value; codes round to nearest, ties to even (torch's
    float8_e4m3fn cast).  Checkpoint-format preparation (per-channel FP8
    weights of the dynamic FP8 scheme)."""
    amax = w.abs().amax(dim=1).float()
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (w / scale.unsqueeze(1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def quantize_mxfp8_weight(w: torch.Tensor):
    """One expert projection [N, K] (float32) -> (E4M3 codes uint8 [N, K], E8M0
    scale codes uint8 [N, K/32]).  Each block of 32 along K shares the scale
    2^X with X = floor(log2(amax)) - 8 (8 being E4M3's largest exponent), the
    OCP MX conversion; codes round to nearest, ties to even, saturating at
    448.  Checkpoint-format preparation."""
    N, K = w.shape
    blk = w.float().reshape(N, K // 32, 32)
    amax = blk.abs().amax(dim=-1)
    _, e = torch.frexp(amax)                      # amax = m 2^e, m in [0.5, 1)
    x = torch.where(amax > 0, e - 1 - 8, torch.full_like(e, -127)).clamp(-127, 127)
    scaled = torch.ldexp(blk, -x.unsqueeze(-1).float())
    q = scaled.clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(N, K).contiguous(), (x + 127).to(torch.uint8).contiguous()


def generate(cfg: MoEConfig, device="cuda", T: int | None = None,
             weights: bool = True) -> dict:
    """Draw one configuration's tensors on ``device``.

    Returns hidden [T,d] bf16, router_w [E,d] f32, corr_bias [E] f32 and, with
    ``weights``, w_gate/w_up [E,F,d] and w_down [E,d,F] in BF16 or, for the
    NVFP4 format, dicts {'q','sf','gs'} per projection, for the FP8 format
    dicts {'q' uint8 [E,N,K], 's' float32 [E,N]}, for the MXFP8 format dicts
    {'q' uint8 [E,N,K], 's' uint8 E8M0 codes [E,N,K/32]}.
    """
    T = cfg.T if T is None else T
    g, gdev = _gen(cfg, device)
    out_dev = torch.device(device)
    d, E, F = cfg.d, cfg.n_experts, cfg.d_ff
    hidden = torch.randn(T, d, generator=g, device=gdev).to(torch.bfloat16)
    router_w = torch.randn(E, d, generator=g, device=gdev) * (1.0 / d) ** 0.5
    bias = (torch.rand(E, generator=g, device=gdev) * 0.1 - 0.05)
    skew = None
    if cfg.skew_experts:
        skew = torch.randperm(E, generator=g, device=gdev)[: cfg.skew_experts]
        bias[skew] += cfg.skew_bias
    res = {"hidden": hidden.to(out_dev), "router_w": router_w.float().to(out_dev),
           "corr_bias": bias.float().to(out_dev), "skewed": None if skew is None else skew.cpu()}
    if not weights:
        return res
    shapes = {"w_gate": (F, d), "w_up": (F, d), "w_down": (d, F)}
    for name, (n, k) in shapes.items():
        if cfg.weight_fmt == "bf16":
            t = torch.empty(E, n, k, dtype=torch.bfloat16, device=out_dev)
            for e in range(E):
                t[e] = (torch.randn(n, k, generator=g, device=gdev) * 0.02).to(torch.bfloat16)
            res[name] = t
        elif cfg.weight_fmt == "nvfp4":
            q = torch.empty(E, n, k // 2, dtype=torch.uint8, device=out_dev)
            sf = torch.empty(E, n, k // 16, dtype=torch.uint8, device=out_dev)
            gs = torch.empty(E, dtype=torch.float32, device=out_dev)
            for e in range(E):
                wq, wsf, wgs = quantize_nvfp4_weight(
                    torch.randn(n, k, generator=g, device=gdev) * 0.02)
                q[e], sf[e], gs[e:e + 1] = wq, wsf, wgs
            res[name] = {"q": q, "sf": sf, "gs": gs}
        elif cfg.weight_fmt == "mxfp8":
            q = torch.empty(E, n, k, dtype=torch.uint8, device=out_dev)
            sc = torch.empty(E, n, k // 32, dtype=torch.uint8, device=out_dev)
            for e in range(E):
                q[e], sc[e] = quantize_mxfp8_weight(
                    torch.randn(n, k, generator=g, device=gdev) * 0.02)
            res[name] = {"q": q, "s": sc}
        elif cfg.weight_fmt == "fp8":
            q = torch.empty(E, n, k, dtype=torch.uint8, device=out_dev)
            sc = torch.empty(E, n, dtype=torch.float32, device=out_dev)
            for e in range(E):
                q[e], sc[e] = quantize_fp8_weight(
                    torch.randn(n, k, generator=g, device=gdev) * 0.02)
            res[name] = {"q": q, "s": sc}
        else:
            raise ValueError(cfg.weight_fmt)
    return res


def bf16_bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
