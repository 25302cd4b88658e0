"""beam_moe_forward_noalloc: the layer for callers that cannot allocate device
memory (its intermediate buffers live in a fixed device array inside the
library instead of a caller workspace).  It must give the same output as
beam_moe_forward on the same inputs, call after call, and refuse batches
whose intermediates would not fit.  Called through the C ABI directly.

This file runs last (pytest collects tests/ in file-name order) so that a
stop-at-first-failure run has already run every other test; it also passes
on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from group_limited_routed_gb300 import api, inputs
from group_limited_routed_gb300.config import CConfig

from _parity import check_out, oracle_out, oracle_route, output_routing

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p


def _noalloc():
    lib = api.lib()
    fn = lib.beam_moe_forward_noalloc
    fn.argtypes = [ctypes.POINTER(CConfig), _P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(cfg, t, hidden, out):
    c = CConfig.of(cfg)
    return _noalloc()(ctypes.byref(c), hidden.data_ptr(), t["router_w"].data_ptr(),
                      t["corr_bias"].data_ptr(), t["w_gate"].data_ptr(), t["w_up"].data_ptr(),
                      t["w_down"].data_ptr(), out.data_ptr(), hidden.shape[0],
                      torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_noalloc_matches_forward_on_two_calls_in_a_row(name):
    cfg = inputs.CONFIGS[name]
    t = inputs.generate(cfg, "cuda")
    # two different batches, one call after the other through the shared array
    batches = [t["hidden"], torch.flip(t["hidden"], dims=[0])[: max(1, cfg.T // 2)].contiguous()]
    outs = []
    for x in batches:
        o = torch.empty(x.shape[0], cfg.d, dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(cfg, t, x, o) == 0
        outs.append(o)
    torch.cuda.synchronize()
    for x, o in zip(batches, outs):
        ref = api.forward(cfg, x, t["router_w"], t["corr_bias"], t["w_gate"], t["w_up"],
                          t["w_down"])
        torch.cuda.synchronize()
        # same kernels on the same inputs: identical, hence within any tolerance
        assert torch.equal(o, ref)
    # and within the parity tolerance of the oracle (first batch)
    sub = cfg.replace(T=batches[0].shape[0])
    tt = dict(t, hidden=batches[0])
    lg, r = oracle_route(sub, tt)
    rows = np.arange(min(sub.T, 8))
    gidx = api.route(sub, batches[0], t["router_w"], t["corr_bias"])[0].cpu().numpy()
    check_out(outs[0], oracle_out(sub, tt, *output_routing(sub, r, gidx, rows), tokens=rows),
              rows=rows)


def test_noalloc_refuses_batches_beyond_its_array():
    cfg = inputs.CONFIGS["decode"]
    t = inputs.generate(cfg, "cuda", T=2, weights=False)
    T_big = 4096
    x = torch.zeros(T_big, cfg.d, dtype=torch.bfloat16, device="cuda")
    o = torch.full((T_big, cfg.d), 3.0, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    c = CConfig.of(cfg)
    rc = _noalloc()(ctypes.byref(c), x.data_ptr(), t["router_w"].data_ptr(),
                    t["corr_bias"].data_ptr(), w.data_ptr(), w.data_ptr(), w.data_ptr(),
                    o.data_ptr(), T_big, torch.cuda.current_stream().cuda_stream)
    assert rc == 3                                  # BEAM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)                      # nothing was launched
