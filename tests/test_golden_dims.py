"""The Beam-sized workloads use the layer dimensions the pages state
(tests/golden/beam_layer_dims.txt, one cited line per value)."""
import os

import numpy as np

import oracle
from group_limited_routed_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    vals = {}
    with open(os.path.join(HERE, "golden", "beam_layer_dims.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, val, src = (p.strip() for p in line.split("|", 2))
            assert src, key
            vals[key] = float(val)
    return vals


def test_beam_configs_use_the_stated_dims():
    g = _golden()
    for name in ("decode", "prefill", "skewed", "nvfp4"):
        c = inputs.CONFIGS[name]
        assert c.d == g["hidden"] == g["router_in"]
        assert c.n_experts == g["routed_experts"] == g["router_out"]
        assert c.n_groups == g["groups"]
        assert c.n_experts // c.n_groups == g["experts_per_group"]
        assert c.topk_groups == g["kept_groups"]
        assert c.topk == g["topk"]
        assert c.d_ff == g["d_ff"]
        assert c.routed_scale == g["routed_scale"]
    # SwiGLU expert = gate + up + down = 3 * d * d_ff parameters, about 39M
    assert round(3 * g["hidden"] * g["d_ff"] / 1e6) == g["expert_params_millions"]


def test_tiny_layer_end_to_end_oracle():
    """The whole layer on the tiny workload: finite, nonzero, the routing
    invariants hold, and no shared expert (a token whose weights are all
    zeroed gives an all-zero output)."""
    cfg = inputs.CONFIGS["tiny"]
    t = inputs.generate(cfg, "cpu")
    out, r, _ = oracle.forward_bf16(inputs.bf16_bits(t["hidden"]), t["router_w"].numpy(),
                                    t["corr_bias"].numpy(), inputs.bf16_bits(t["w_gate"]),
                                    inputs.bf16_bits(t["w_up"]), inputs.bf16_bits(t["w_down"]),
                                    cfg.n_groups, cfg.topk_groups, cfg.topk, cfg.routed_scale)
    o = oracle.bf16_to_f64(out)
    assert np.all(np.isfinite(o)) and np.sqrt((o ** 2).mean()) > 1e-3
    w0 = r["w"].copy()
    w0[5] = 0.0
    out0 = oracle.experts_bf16(inputs.bf16_bits(t["hidden"]), r["idx"], w0,
                               inputs.bf16_bits(t["w_gate"]), inputs.bf16_bits(t["w_up"]),
                               inputs.bf16_bits(t["w_down"]), cfg.n_experts)
    assert np.all(oracle.bf16_to_f64(out0[5]) == 0)
    assert np.array_equal(out0[:5], out[:5])
