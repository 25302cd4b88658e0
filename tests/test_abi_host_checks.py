"""Host-side argument checks of the C ABI, without a GPU: every entry point
rejects an invalid layer shape, a negative token count or an unknown format
before it touches the device, and a zero-token call is a no-op."""
import ctypes

import pytest

from group_limited_routed_gb300 import api
from group_limited_routed_gb300.inputs import CONFIGS

INVALID, OK = 1, 0
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    from group_limited_routed_gb300 import build
    return ctypes.CDLL(build.build())


def _cfg(**kw):
    return ctypes.byref(api.CConfig.of(CONFIGS["decode"].replace(**kw)))


def _forward_like(fn, cfg, T):
    fn.restype = ctypes.c_int
    return fn(cfg, None, None, None, None, None, None, None, ctypes.c_int64(T), None,
              ctypes.c_size_t(0), None)


@pytest.mark.parametrize("shape", [dict(n_groups=7), dict(d=500), dict(d_ff=100),
                                   dict(n_experts=512), dict(topk=40), dict(topk_groups=9),
                                   dict(routed_scale=0.0)])
def test_invalid_shapes_are_rejected_before_any_launch(lib, shape):
    cfg = _cfg(**shape)
    for name in ("beam_moe_forward", "beam_moe_forward_routed"):
        assert _forward_like(getattr(lib, name), cfg, 4) == INVALID, (name, shape)
    for name in ("beam_moe_forward_nvfp4", "beam_moe_forward_nvfp4_a16", "beam_moe_forward_fp8"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        assert fn(cfg, None, None, None, None, None, None, None, ctypes.c_int64(4), None,
                  ctypes.c_size_t(0), None) == INVALID, (name, shape)
    lib.beam_moe_workspace_size.restype = ctypes.c_size_t
    assert lib.beam_moe_workspace_size(cfg, ctypes.c_int64(4), 0) == 0


def test_negative_token_count_and_zero_tokens(lib):
    cfg = _cfg()
    assert _forward_like(lib.beam_moe_forward, cfg, -1) == INVALID
    # T = 0: valid shape, nothing to do, no pointer is looked at
    assert _forward_like(lib.beam_moe_forward, cfg, 0) == OK
    assert _forward_like(lib.beam_moe_forward_routed, cfg, 0) == OK


def test_nvfp4_paths_need_256_aligned_dimensions(lib):
    cfg = _cfg(d=5120 + 128)          # valid BF16 shape, not an NVFP4 one
    for name in ("beam_moe_forward_nvfp4", "beam_moe_forward_nvfp4_a16"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        assert fn(cfg, None, None, None, None, None, None, None, ctypes.c_int64(4), None,
                  ctypes.c_size_t(0), None) == INVALID
    lib.beam_moe_workspace_size.restype = ctypes.c_size_t
    assert lib.beam_moe_workspace_size(cfg, ctypes.c_int64(4), 0) > 0
    assert lib.beam_moe_workspace_size(cfg, ctypes.c_int64(4), 9) == 0   # unknown format


def test_boundary_and_expert_parallel_checks(lib):
    cfg = _cfg()
    lib.beam_moe_forward_boundary.restype = ctypes.c_int
    assert lib.beam_moe_forward_boundary(_cfg(d=500), None, None, None, None, None, None, None,
                                         ctypes.c_int64(4), None, None, ctypes.c_size_t(0),
                                         None) == INVALID
    lib.beam_moe_ep_experts.restype = ctypes.c_int
    for n_ranks, rank in ((3, 0), (8, 8), (8, -1), (0, 0)):
        assert lib.beam_moe_ep_experts(cfg, n_ranks, rank, None, None, None, None, None, None,
                                       None, ctypes.c_int64(4), None, ctypes.c_size_t(0),
                                       None) == INVALID, (n_ranks, rank)
    # a rank that received nothing launches nothing
    assert lib.beam_moe_ep_experts(cfg, 8, 3, None, None, None, None, None, None, None,
                                   ctypes.c_int64(0), None, ctypes.c_size_t(0), None) == OK
    for name in ("beam_moe_ep_experts_nvfp4", "beam_moe_ep_experts_fp8"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        for n_ranks, rank in ((3, 0), (8, 8), (8, -1)):
            assert fn(cfg, n_ranks, rank, None, None, None, None, None, None, None,
                      ctypes.c_int64(4), None, ctypes.c_size_t(0), None) == INVALID, (name, rank)
        assert fn(cfg, 8, 3, None, None, None, None, None, None, None, ctypes.c_int64(0), None,
                  ctypes.c_size_t(0), None) == OK
    lib.beam_moe_kernels_per_forward.restype = ctypes.c_int32
    assert lib.beam_moe_kernels_per_forward(_cfg(n_groups=7), ctypes.c_int64(32), 0, 0) == 0


def test_fp8_entry_points(lib):
    fwd = lib.beam_moe_forward_fp8
    fwd.restype = ctypes.c_int
    assert fwd(_cfg(), None, None, None, None, None, None, None, ctypes.c_int64(0), None,
               ctypes.c_size_t(0), None) == OK                        # nothing to do
    assert fwd(_cfg(), None, None, None, None, None, None, None, ctypes.c_int64(-3), None,
               ctypes.c_size_t(0), None) == INVALID
    q = lib.beam_moe_fp8_quantize_rows
    q.restype = ctypes.c_int
    q.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P]
    assert q(None, 0, 128, None, None, None) == OK                     # no rows, no launch
    assert q(None, -1, 128, None, None, None) == INVALID
    assert q(None, 4, 100, None, None, None) == INVALID                 # cols % 8 != 0
    assert q(None, 4, 128, None, None, None) == INVALID                 # null pointers
    lib.beam_moe_workspace_size.restype = ctypes.c_size_t
    assert lib.beam_moe_workspace_size(_cfg(), ctypes.c_int64(32), 3) > 0


def test_quantised_boundary_entry_points(lib):
    """The boundary description is checked before the zero-token return; a
    NULL description is the plain layer call."""
    bad_n = api._Boundary(None, None, None, None, 1e-6, 0)
    bad_eps = api._Boundary(None, None, None, None, -1.0, 2)
    good = api._Boundary(None, None, None, None, 1e-6, 2)
    for name in ("beam_moe_forward_nvfp4_boundary", "beam_moe_forward_nvfp4_a16_boundary",
                 "beam_moe_forward_fp8_boundary"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int

        def call(b, T, **kw):
            return fn(_cfg(**kw), None, None, None, None, None, None, None, ctypes.c_int64(T),
                      None if b is None else ctypes.byref(b), None, ctypes.c_size_t(0), None)

        assert call(None, 0) == OK, name
        assert call(good, 0) == OK, name
        assert call(bad_n, 0) == INVALID, name
        assert call(bad_eps, 0) == INVALID, name
        assert call(good, -1) == INVALID, name
        assert call(good, 4, n_groups=7) == INVALID, name
        assert call(good, 4) == INVALID, name                  # null pointers
    fn = lib.beam_moe_forward_nvfp4_boundary
    assert fn(_cfg(d=5120 + 128), None, None, None, None, None, None, None, ctypes.c_int64(4),
              ctypes.byref(good), None, ctypes.c_size_t(0), None) == INVALID
