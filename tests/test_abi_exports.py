"""The C-ABI library builds for sm_103a, loads without a GPU and exports
every entry point include/beam_moe.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "beam_moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from group_limited_routed_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_layer_entry_points():
    names = _declared()
    for n in ("beam_moe_route", "beam_moe_forward", "beam_moe_forward_routed",
              "beam_moe_workspace_size", "beam_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_python_binding_names_match_exports(lib):
    from group_limited_routed_gb300 import api
    assert set(api.EXPORTS) <= set(_declared())


def test_host_only_queries(lib):
    from group_limited_routed_gb300 import api
    from group_limited_routed_gb300.inputs import CONFIGS
    beam = CONFIGS["decode"]
    n = api.workspace_size(beam, 8192)
    lay = api.layout(beam, 8192)
    assert lay["total"] == n and n % 256 == 0
    offs = sorted(v for k, v in lay.items() if k != "total")
    assert offs[0] == 0 and all(o % 256 == 0 for o in offs)
    # routing+permute as one launch, gate/up (gathering), down, combine
    assert api.kernels_per_forward(beam, 32) == 4
    # plane split, tensor router, select, permute, gather, gate/up, down, combine
    assert api.kernels_per_forward(beam, 8192) == 8
    assert api.kernels_per_forward(beam, 32, routed=True) == 4       # permute .. combine
    assert api.kernels_per_forward(beam, 8192, routed=True) == 5
    assert api.kernels_per_forward(beam, 128, weight_fmt=api.NVFP4) == 5
    assert api.kernels_per_forward(beam, 4096, weight_fmt=api.NVFP4) == 8
    assert api.kernels_per_forward(beam, 32, weight_fmt=api.NVFP4, routed=True) == 0
    # FP8: routing+permute, x quantisation, gate/up, h quantisation, down, combine
    assert api.kernels_per_forward(beam, 32, weight_fmt=api.FP8) == 6
    # ... plus plane split, tensor router, select and the gather of the token codes
    assert api.kernels_per_forward(beam, 8192, weight_fmt=api.FP8) == 10
    f8 = api.layout(beam, 32, weight_fmt=api.FP8)
    assert f8["x_fp8"] > 0 and f8["h_scale"] > f8["h_fp8"] > f8["x_scale"] > f8["x_fp8"]
    assert f8["total"] == api.workspace_size(beam, 32, weight_fmt=api.FP8)
    with pytest.raises(api.BeamError):
        api.workspace_size(beam.replace(n_groups=7), 32)
    lib.beam_status_string.restype = ctypes.c_char_p
    assert lib.beam_status_string(5) == b"device-side wait timed out"


def test_ep_workspace_query(lib):
    from group_limited_routed_gb300 import api
    from group_limited_routed_gb300.inputs import CONFIGS
    beam = CONFIGS["decode"]
    c = api.CConfig.of(beam)
    size = lib.beam_moe_ep_workspace_size
    size.restype = ctypes.c_size_t
    size.argtypes = [ctypes.POINTER(api.CConfig), ctypes.c_int32, ctypes.c_int64,
                     ctypes.c_int32]
    assert size(ctypes.byref(c), 8, 256, 0) % 256 == 0 and size(ctypes.byref(c), 8, 256, 0) > 0
    assert size(ctypes.byref(c), 8, 1024, 0) >= size(ctypes.byref(c), 8, 256, 0)
    assert size(ctypes.byref(c), 8, 256, 1) > 0       # NVFP4 experts
    assert size(ctypes.byref(c), 3, 256, 0) == 0      # 3 does not divide 256 experts
    assert size(ctypes.byref(c), 512, 256, 0) == 0    # more ranks than experts
    assert size(ctypes.byref(c), 8, 256, 2) == 0      # no W4A16 expert-parallel path
    assert size(ctypes.byref(c), 8, 256, 3) > 0       # FP8 experts


def _calls_of(tree, name):
    import ast
    return [n for n in ast.walk(tree) if isinstance(n, ast.Call) and
            isinstance(n.func, ast.Name) and n.func.id == name]


def test_every_binding_checks_the_status_of_the_function_it_calls():
    """Each `_check(status, name)` in the binding names the library function
    whose status it checks, and that function is declared and exported (a
    wrapper only reaches the library on a GPU, so this is its CPU check)."""
    import ast
    from group_limited_routed_gb300 import api
    tree = ast.parse(open(api.__file__).read())
    declared = set(_declared())
    checks = _calls_of(tree, "_check")
    assert len(checks) >= 15
    for c in checks:
        assert len(c.args) == 2 and not c.keywords, ast.unparse(c)[:80]
        call, name = c.args
        assert isinstance(call, ast.Call), ast.unparse(c)[:80]
        if isinstance(name, ast.Constant):
            f = call.func
            assert isinstance(f, ast.Attribute) and f.attr == name.value, ast.unparse(c)[:80]
            assert name.value in declared and name.value in api.EXPORTS, name.value
    assert set(api.EXPORTS) <= declared
