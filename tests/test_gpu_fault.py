"""Failure detection without a GPU fault: a test knob makes the first CTA of
the gate/up GEMM skip its first operand load, so that stage never fills and
the MMA warp's bounded wait runs out.  The kernel must latch
BEAM_ERR_TIMEOUT, let its other copies land, free TMEM and return; the
context stays usable and the next call is correct."""
import numpy as np
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

from _parity import check_out, gpu_routing, oracle_out, oracle_route, output_routing

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [16, 64])   # 16-row (row gather) and 128-row token blocks
def test_bounded_wait_reports_timeout_and_the_context_recovers(T):
    cfg = inputs.CONFIGS["tiny"].replace(T=T, seed=90 + T)
    t = inputs.generate(cfg, "cuda")
    ws = pkg.Workspace(cfg, cfg.T)
    args = (cfg, t["hidden"], t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"], t["w_down"])
    pkg.set_debug(wait_limit_us=20000, withhold_first_load=True)
    try:
        pkg.forward(*args, ws=ws)
        assert pkg.check_status(ws) == 5          # BEAM_ERR_TIMEOUT, latched
    finally:
        pkg.set_debug(0, False)
    assert pkg.check_status(ws) == 0              # cleared by the read
    out = pkg.forward(*args, ws=ws)
    assert pkg.check_status(ws) == 0
    lg, r = oracle_route(cfg, t)
    check_out(out, oracle_out(cfg, t, *output_routing(cfg, r, gpu_routing(ws, cfg, cfg.T))))
