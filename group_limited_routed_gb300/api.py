"""Thin Python binding of libbeam_moe.so (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels; this module only
checks tensor dtypes/devices, hands raw device pointers and the current torch
stream to the C ABI, and raises ``BeamError`` on a non-OK status.  There is no
fallback: without the compiled library every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .config import BeamMoEConfig, CConfig

_HERE = os.path.dirname(os.path.abspath(__file__))
# BEAM_MOE_DEVICE_CHECKS=1 loads the debug build with device-side bounds
# checks (group_limited_routed_gb300.build.build(checked=True)) instead
_LIB_PATH = os.path.join(_HERE, "_build_checked" if os.environ.get("BEAM_MOE_DEVICE_CHECKS") == "1"
                         else "_build", "libbeam_moe.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
          4: "CUDA error", 5: "device-side wait timed out", 6: "device-side check failed"}

EXPORTS = ("beam_moe_workspace_size", "beam_moe_workspace_layout", "beam_moe_route",
           "beam_moe_select", "beam_moe_forward", "beam_moe_forward_routed",
           "beam_moe_forward_noalloc", "beam_moe_forward_nvfp4", "beam_moe_nvfp4_pack_scales",
           "beam_moe_check_status", "beam_moe_set_stage_events", "beam_moe_set_debug",
           "beam_moe_kernels_per_forward", "beam_status_string", "beam_moe_ep_dispatch",
           "beam_moe_ep_workspace_size", "beam_moe_ep_experts", "beam_moe_ep_combine",
           "beam_moe_forward_boundary", "beam_moe_forward_nvfp4_a16",
           "beam_moe_ep_experts_nvfp4", "beam_moe_forward_fp8", "beam_moe_fp8_quantize_rows",
           "beam_moe_ep_experts_fp8", "beam_moe_forward_nvfp4_boundary",
           "beam_moe_forward_nvfp4_a16_boundary", "beam_moe_forward_fp8_boundary",
           "beam_moe_forward_mxfp8", "beam_moe_forward_mxfp8_boundary")


class BeamError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "logits", "topk_idx", "topk_w", "counts", "offsets", "perm_src", "pair_row",
        "perm_w", "x_perm", "h", "x_fp4", "x_sf", "h_fp4", "h_sf", "y", "x_fp8", "x_scale",
        "h_fp8", "h_scale", "total")]


class _Boundary(ctypes.Structure):
    _fields_ = [("residual", ctypes.c_void_p), ("post_norm_w", ctypes.c_void_p),
                ("next_norm_w", ctypes.c_void_p), ("next_input", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("residual_index", ctypes.c_int32)]


class _Fp4Weight(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


class _Fp8Weight(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class _Mxfp8Weight(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load libbeam_moe.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with group_limited_routed_gb300.build.build() "
                "(there is no non-CUDA fallback)")
        L = ctypes.CDLL(_LIB_PATH)
        cfgp = ctypes.POINTER(CConfig)
        L.beam_moe_workspace_size.argtypes = [cfgp, _I64, ctypes.c_int32]
        L.beam_moe_workspace_size.restype = _SZ
        L.beam_moe_workspace_layout.argtypes = [cfgp, _I64, ctypes.c_int32, ctypes.POINTER(_Layout)]
        L.beam_moe_workspace_layout.restype = _ST
        L.beam_moe_route.argtypes = [cfgp, _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]
        L.beam_moe_route.restype = _ST
        L.beam_moe_select.argtypes = [cfgp, _P, _P, _I64, _P, _P, _P, _SZ, _P]
        L.beam_moe_select.restype = _ST
        L.beam_moe_forward.argtypes = [cfgp, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _SZ, _P]
        L.beam_moe_forward.restype = _ST
        L.beam_moe_forward_routed.argtypes = [cfgp, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _SZ, _P]
        L.beam_moe_forward_routed.restype = _ST
        L.beam_moe_forward_noalloc.argtypes = [cfgp, _P, _P, _P, _P, _P, _P, _P, _I64, _P]
        L.beam_moe_forward_noalloc.restype = _ST
        fp4p = ctypes.POINTER(_Fp4Weight)
        L.beam_moe_forward_nvfp4.argtypes = [cfgp, _P, _P, _P, fp4p, fp4p, fp4p, _P, _I64, _P,
                                             _SZ, _P]
        L.beam_moe_forward_nvfp4.restype = _ST
        L.beam_moe_forward_nvfp4_a16.argtypes = [cfgp, _P, _P, _P, fp4p, fp4p, fp4p, _P, _I64,
                                                 _P, _SZ, _P]
        L.beam_moe_forward_nvfp4_a16.restype = _ST
        fp8p = ctypes.POINTER(_Fp8Weight)
        L.beam_moe_forward_fp8.argtypes = [cfgp, _P, _P, _P, fp8p, fp8p, fp8p, _P, _I64, _P,
                                           _SZ, _P]
        L.beam_moe_forward_fp8.restype = _ST
        mxp = ctypes.POINTER(_Mxfp8Weight)
        L.beam_moe_forward_mxfp8.argtypes = [cfgp, _P, _P, _P, mxp, mxp, mxp, _P, _I64, _P,
                                             _SZ, _P]
        L.beam_moe_forward_mxfp8.restype = _ST
        L.beam_moe_fp8_quantize_rows.argtypes = [_P, _I64, ctypes.c_int32, _P, _P, _P]
        L.beam_moe_ep_experts_fp8.argtypes = [cfgp, ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                              fp8p, fp8p, fp8p, _P, _I64, _P, _SZ, _P]
        L.beam_moe_ep_experts_fp8.restype = _ST
        L.beam_moe_fp8_quantize_rows.restype = _ST
        L.beam_moe_nvfp4_pack_scales.argtypes = [_P, _I64, _I64, _P, _P]
        L.beam_moe_nvfp4_pack_scales.restype = _ST
        L.beam_moe_check_status.argtypes = [_P, _P]
        L.beam_moe_check_status.restype = _ST
        L.beam_moe_set_stage_events.argtypes = [ctypes.POINTER(_P), ctypes.c_int32]
        L.beam_moe_set_stage_events.restype = _ST
        L.beam_moe_set_debug.argtypes = [ctypes.c_uint32, ctypes.c_int32]
        L.beam_moe_set_debug.restype = _ST
        L.beam_moe_kernels_per_forward.argtypes = [cfgp, _I64, ctypes.c_int32, ctypes.c_int32]
        L.beam_moe_kernels_per_forward.restype = ctypes.c_int32
        L.beam_moe_forward_boundary.argtypes = [cfgp, _P, _P, _P, _P, _P, _P, _P, _I64,
                                                ctypes.POINTER(_Boundary), _P, _SZ, _P]
        L.beam_moe_forward_boundary.restype = _ST
        for name, wp in (("beam_moe_forward_nvfp4_boundary", fp4p),
                         ("beam_moe_forward_nvfp4_a16_boundary", fp4p),
                         ("beam_moe_forward_fp8_boundary", fp8p),
                         ("beam_moe_forward_mxfp8_boundary", mxp)):
            f = getattr(L, name)
            f.argtypes = [cfgp, _P, _P, _P, wp, wp, wp, _P, _I64, ctypes.POINTER(_Boundary), _P,
                          _SZ, _P]
            f.restype = _ST
        L.beam_moe_ep_dispatch.argtypes = [cfgp, _P, _P, _P, _I64, ctypes.c_int32, _P, _P, _P, _P,
                                           _P, _SZ, _P]
        L.beam_moe_ep_dispatch.restype = _ST
        L.beam_moe_ep_workspace_size.argtypes = [cfgp, ctypes.c_int32, _I64, ctypes.c_int32]
        L.beam_moe_ep_workspace_size.restype = _SZ
        L.beam_moe_ep_experts.argtypes = [cfgp, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P,
                                          _P, _P, _I64, _P, _SZ, _P]
        L.beam_moe_ep_experts.restype = _ST
        L.beam_moe_ep_experts_nvfp4.argtypes = [cfgp, ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                                fp4p, fp4p, fp4p, _P, _I64, _P, _SZ, _P]
        L.beam_moe_ep_experts_nvfp4.restype = _ST
        L.beam_moe_ep_combine.argtypes = [cfgp, _P, _I64, _P, _P, _SZ, _P]
        L.beam_moe_ep_combine.restype = _ST
        L.beam_status_string.argtypes = [_ST]
        L.beam_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def _cfg(cfg) -> CConfig:
    return CConfig.of(cfg)


def _check(code: int, where: str):
    if code != 0:
        raise BeamError(code, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def workspace_size(cfg, T_max: int, weight_fmt: int = 0) -> int:
    c = _cfg(cfg)
    n = lib().beam_moe_workspace_size(ctypes.byref(c), int(T_max), int(weight_fmt))
    if n == 0:
        raise BeamError(1, "beam_moe_workspace_size")
    return int(n)


def layout(cfg, T_max: int, weight_fmt: int = 0) -> dict:
    c = _cfg(cfg)
    out = _Layout()
    _check(lib().beam_moe_workspace_layout(ctypes.byref(c), int(T_max), int(weight_fmt),
                                           ctypes.byref(out)), "beam_moe_workspace_layout")
    return {n: int(getattr(out, n)) for n, _ in _Layout._fields_}


class Workspace:
    """Caller-owned device workspace sized for up to T_max tokens."""

    def __init__(self, cfg, T_max: int, device=None, weight_fmt: int = 0):
        self.cfg = cfg
        self.T_max = int(T_max)
        self.nbytes = workspace_size(cfg, T_max, weight_fmt)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8,
                               device=device if device is not None else torch.device("cuda"))
        self.layout = layout(cfg, T_max, weight_fmt)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def view(self, name: str, dtype, shape) -> torch.Tensor:
        """A tensor view of one intermediate buffer (see beam_moe_ws_layout_t)."""
        off = self.layout[name]
        n = 1
        for s in shape:
            n *= int(s)
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return self.buf[off:off + nbytes].view(dtype).view(*shape)


def _ws(cfg, T, ws, device):
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), device)
    return ws


def route(cfg, hidden, router_w, corr_bias, ws: Workspace | None = None, want_logits=False,
          stream=None):
    """Router + group-limited selection -> (idx [T,k] int32, w [T,k] f32[, logits])."""
    T = hidden.shape[0]
    ws = _ws(cfg, T, ws, hidden.device)
    idx = torch.empty(T, cfg.topk, dtype=torch.int32, device=hidden.device)
    w = torch.empty(T, cfg.topk, dtype=torch.float32, device=hidden.device)
    logits = torch.empty(T, cfg.n_experts, dtype=torch.float32, device=hidden.device) \
        if want_logits else None
    c = _cfg(cfg)
    _check(lib().beam_moe_route(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                _dev(router_w, torch.float32, "router_w"),
                                _dev(corr_bias, torch.float32, "corr_bias"), T, idx.data_ptr(),
                                w.data_ptr(), None if logits is None else logits.data_ptr(),
                                ws.ptr, ws.nbytes, _stream(stream)), "beam_moe_route")
    return (idx, w, logits) if want_logits else (idx, w)


def select(cfg, logits, corr_bias, ws: Workspace | None = None, stream=None):
    """Selection alone on given FP32 logits -> (idx, w)."""
    T = logits.shape[0]
    ws = _ws(cfg, T, ws, logits.device)
    idx = torch.empty(T, cfg.topk, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, cfg.topk, dtype=torch.float32, device=logits.device)
    c = _cfg(cfg)
    _check(lib().beam_moe_select(ctypes.byref(c), _dev(logits, torch.float32, "logits"),
                                 _dev(corr_bias, torch.float32, "corr_bias"), T, idx.data_ptr(),
                                 w.data_ptr(), ws.ptr, ws.nbytes, _stream(stream)),
           "beam_moe_select")
    return idx, w


def forward(cfg, hidden, router_w, corr_bias, w_gate, w_up, w_down, out=None,
            ws: Workspace | None = None, stream=None):
    """The whole layer.  ``hidden`` may be a (pinned) host tensor: it is then
    copied to the weights' device and the output copied back to the host."""
    host_in = not hidden.is_cuda
    dev = w_gate.device
    x = hidden.to(dev, non_blocking=True) if host_in else hidden
    T = x.shape[0]
    ws = _ws(cfg, T, ws, dev)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=dev) if (out is None or host_in) else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward(ctypes.byref(c), _dev(x, torch.bfloat16, "hidden"),
                                  _dev(router_w, torch.float32, "router_w"),
                                  _dev(corr_bias, torch.float32, "corr_bias"),
                                  _dev(w_gate, torch.bfloat16, "w_gate"),
                                  _dev(w_up, torch.bfloat16, "w_up"),
                                  _dev(w_down, torch.bfloat16, "w_down"), o.data_ptr(), T,
                                  ws.ptr, ws.nbytes, _stream(stream)), "beam_moe_forward")
    if host_in:
        if out is None:
            out = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        out.copy_(o, non_blocking=True)
        return out
    return o


def forward_boundary(cfg, hidden, router_w, corr_bias, w_gate, w_up, w_down, residual,
                     post_norm_w, next_norm_w, eps: float, n: int, out=None, next_input=None,
                     ws: Workspace | None = None, stream=None, a16: bool = False):
    """The layer followed by the decoder's sublayer boundary (post-norm, n-th
    depth-scaled residual add, next pre-norm) in its combine kernel.  Returns
    (out, next_input); ``residual`` is overwritten with the new stream.

    The expert format follows the weights: BF16 tensors, ``Fp4Weight`` (NVFP4
    activations, or F16 ones with ``a16=True``), ``Fp8Weight`` or
    ``Mxfp8Weight``."""
    T = hidden.shape[0]
    dev = hidden.device
    if isinstance(w_gate, Fp4Weight):
        fmt, name = (NVFP4_A16, "beam_moe_forward_nvfp4_a16_boundary") if a16 else \
            (NVFP4, "beam_moe_forward_nvfp4_boundary")
        wts = tuple(ctypes.byref(x._c) for x in (w_gate, w_up, w_down))
    elif isinstance(w_gate, Fp8Weight):
        fmt, name = FP8, "beam_moe_forward_fp8_boundary"
        wts = tuple(ctypes.byref(x._c) for x in (w_gate, w_up, w_down))
    elif isinstance(w_gate, Mxfp8Weight):
        fmt, name = MXFP8, "beam_moe_forward_mxfp8_boundary"
        wts = tuple(ctypes.byref(x._c) for x in (w_gate, w_up, w_down))
    else:
        fmt, name = BF16, "beam_moe_forward_boundary"
        wts = (_dev(w_gate, torch.bfloat16, "w_gate"), _dev(w_up, torch.bfloat16, "w_up"),
               _dev(w_down, torch.bfloat16, "w_down"))
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), dev, weight_fmt=fmt)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=dev) if out is None else out
    nx = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=dev) if next_input is None \
        else next_input
    b = _Boundary(_dev(residual, torch.bfloat16, "residual"),
                  _dev(post_norm_w, torch.bfloat16, "post_norm_w"),
                  _dev(next_norm_w, torch.bfloat16, "next_norm_w"),
                  _dev(nx, torch.bfloat16, "next_input"), float(eps), int(n))
    c = _cfg(cfg)
    _check(getattr(lib(), name)(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                _dev(router_w, torch.float32, "router_w"),
                                _dev(corr_bias, torch.float32, "corr_bias"), *wts, o.data_ptr(),
                                T, ctypes.byref(b), ws.ptr, ws.nbytes, _stream(stream)), name)
    return o, nx


def forward_routed(cfg, hidden, topk_idx, topk_w, w_gate, w_up, w_down, out=None,
                   ws: Workspace | None = None, stream=None):
    """Experts + combine with a given routing (routing replay)."""
    T = hidden.shape[0]
    ws = _ws(cfg, T, ws, hidden.device)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_routed(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                         _dev(topk_idx, torch.int32, "topk_idx"),
                                         _dev(topk_w, torch.float32, "topk_w"),
                                         _dev(w_gate, torch.bfloat16, "w_gate"),
                                         _dev(w_up, torch.bfloat16, "w_up"),
                                         _dev(w_down, torch.bfloat16, "w_down"), o.data_ptr(), T,
                                         ws.ptr, ws.nbytes, _stream(stream)),
           "beam_moe_forward_routed")
    return o


def forward_noalloc(cfg, hidden, router_w, corr_bias, w_gate, w_up, w_down, out=None,
                    stream=None):
    """The whole layer without a workspace: for callers that cannot allocate
    device memory (the library's fixed 32 MiB device array holds the
    intermediates; small batches only, see beam_moe.h).  Calls overlapping on
    the GPU race on that array."""
    T = hidden.shape[0]
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_noalloc(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                          _dev(router_w, torch.float32, "router_w"),
                                          _dev(corr_bias, torch.float32, "corr_bias"),
                                          _dev(w_gate, torch.bfloat16, "w_gate"),
                                          _dev(w_up, torch.bfloat16, "w_up"),
                                          _dev(w_down, torch.bfloat16, "w_down"), o.data_ptr(),
                                          T, _stream(stream)), "beam_moe_forward_noalloc")
    return o


BF16 = 0
NVFP4 = 1
NVFP4_A16 = 2


def pack_scales(sf: torch.Tensor, stream=None) -> torch.Tensor:
    """Block scales [..., rows, S] (uint8, row-major: E4M3 for NVFP4, E8M0 for
    MXFP8) -> the blocked order the tensor cores take
    (beam_moe_nvfp4_pack_scales); same shape and dtype."""
    src = sf.contiguous()
    S = src.shape[-1]
    rows = src.numel() // S
    dst = torch.empty_like(src)
    _check(lib().beam_moe_nvfp4_pack_scales(_dev(src, torch.uint8, "sf"), rows, S,
                                            dst.data_ptr(), _stream(stream)),
           "beam_moe_nvfp4_pack_scales")
    return dst


class Fp4Weight:
    """One NVFP4 projection: codes q [E, N, K/2], blocked scales, global scales [E]."""

    def __init__(self, q: torch.Tensor, sf_rowmajor: torch.Tensor, gs: torch.Tensor,
                 stream=None):
        self.q = q.contiguous()
        self.sf = pack_scales(sf_rowmajor, stream)
        self.gs = gs.contiguous().float()
        self._c = _Fp4Weight(_dev(self.q, torch.uint8, "q"), self.sf.data_ptr(),
                             _dev(self.gs, torch.float32, "global_scale"))

    @classmethod
    def of(cls, d: dict, stream=None) -> "Fp4Weight":
        return cls(d["q"], d["sf"], d["gs"], stream)


def forward_nvfp4(cfg, hidden, router_w, corr_bias, gate: Fp4Weight, up: Fp4Weight,
                  down: Fp4Weight, out=None, ws: Workspace | None = None, stream=None):
    """The whole layer with NVFP4 experts (activations quantised to NVFP4)."""
    T = hidden.shape[0]
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), hidden.device, weight_fmt=NVFP4)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_nvfp4(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                        _dev(router_w, torch.float32, "router_w"),
                                        _dev(corr_bias, torch.float32, "corr_bias"),
                                        ctypes.byref(gate._c), ctypes.byref(up._c),
                                        ctypes.byref(down._c), o.data_ptr(), T, ws.ptr, ws.nbytes,
                                        _stream(stream)), "beam_moe_forward_nvfp4")
    return o


def forward_nvfp4_a16(cfg, hidden, router_w, corr_bias, gate: Fp4Weight, up: Fp4Weight,
                      down: Fp4Weight, out=None, ws: Workspace | None = None, stream=None):
    """The whole layer with NVFP4 expert weights and 16-bit (F16) activations."""
    T = hidden.shape[0]
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), hidden.device, weight_fmt=NVFP4_A16)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_nvfp4_a16(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                            _dev(router_w, torch.float32, "router_w"),
                                            _dev(corr_bias, torch.float32, "corr_bias"),
                                            ctypes.byref(gate._c), ctypes.byref(up._c),
                                            ctypes.byref(down._c), o.data_ptr(), T, ws.ptr,
                                            ws.nbytes, _stream(stream)),
           "beam_moe_forward_nvfp4_a16")
    return o


FP8 = 3


class Fp8Weight:
    """One dynamic-FP8 projection: E4M3 codes q [E, N, K] (uint8) and one
    FP32 scale per output row [E, N]."""

    def __init__(self, q: torch.Tensor, scale: torch.Tensor):
        self.q = q.contiguous()
        self.scale = scale.contiguous()
        self._c = _Fp8Weight(_dev(self.q, torch.uint8, "q"),
                             _dev(self.scale, torch.float32, "scale"))

    @classmethod
    def of(cls, d: dict) -> "Fp8Weight":
        return cls(d["q"], d["s"])


def forward_fp8(cfg, hidden, router_w, corr_bias, gate: Fp8Weight, up: Fp8Weight,
                down: Fp8Weight, out=None, ws: Workspace | None = None, stream=None):
    """The whole layer with dynamic FP8 experts (E4M3 weights with per-row
    scales; token rows and h quantised per row at run time)."""
    T = hidden.shape[0]
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), hidden.device, weight_fmt=FP8)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_fp8(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                      _dev(router_w, torch.float32, "router_w"),
                                      _dev(corr_bias, torch.float32, "corr_bias"),
                                      ctypes.byref(gate._c), ctypes.byref(up._c),
                                      ctypes.byref(down._c), o.data_ptr(), T, ws.ptr, ws.nbytes,
                                      _stream(stream)), "beam_moe_forward_fp8")
    return o


MXFP8 = 4


class Mxfp8Weight:
    """One MXFP8 projection: E4M3 codes q [E, N, K] (uint8) and E8M0 scales,
    one per 32 along K, given row-major [E, N, K/32] and kept in the blocked
    order the tensor cores take (beam_moe_nvfp4_pack_scales)."""

    def __init__(self, q: torch.Tensor, sf_rowmajor: torch.Tensor, stream=None):
        self.q = q.contiguous()
        self.sf = pack_scales(sf_rowmajor, stream)
        self._c = _Mxfp8Weight(_dev(self.q, torch.uint8, "q"), self.sf.data_ptr())

    @classmethod
    def of(cls, d: dict, stream=None) -> "Mxfp8Weight":
        return cls(d["q"], d["s"], stream)


def forward_mxfp8(cfg, hidden, router_w, corr_bias, gate: Mxfp8Weight, up: Mxfp8Weight,
                  down: Mxfp8Weight, out=None, ws: Workspace | None = None, stream=None):
    """The whole layer with MXFP8 experts (activations quantised to MX blocks)."""
    T = hidden.shape[0]
    if ws is None:
        ws = Workspace(cfg, max(int(T), 1), hidden.device, weight_fmt=MXFP8)
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=hidden.device) if out is None else out
    c = _cfg(cfg)
    _check(lib().beam_moe_forward_mxfp8(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                        _dev(router_w, torch.float32, "router_w"),
                                        _dev(corr_bias, torch.float32, "corr_bias"),
                                        ctypes.byref(gate._c), ctypes.byref(up._c),
                                        ctypes.byref(down._c), o.data_ptr(), T, ws.ptr, ws.nbytes,
                                        _stream(stream)), "beam_moe_forward_mxfp8")
    return o


def fp8_quantize_rows(x: torch.Tensor, stream=None):
    """BF16 rows [n, cols] -> (E4M3 codes uint8 [n, cols], FP32 scales [n]),
    the FP8 path's activation rule (beam_moe_fp8_quantize_rows)."""
    n, cols = x.shape
    q = torch.empty(n, cols, dtype=torch.uint8, device=x.device)
    sc = torch.empty(n, dtype=torch.float32, device=x.device)
    _check(lib().beam_moe_fp8_quantize_rows(_dev(x, torch.bfloat16, "x"), n, cols, q.data_ptr(),
                                            sc.data_ptr(), _stream(stream)),
           "beam_moe_fp8_quantize_rows")
    return q, sc


def check_status(ws: Workspace, stream=None) -> int:
    """Synchronise and return (and clear) the latched device status code."""
    return int(lib().beam_moe_check_status(ws.ptr, _stream(stream)))


def set_stage_events(events) -> None:
    """Record 8 torch.cuda.Event objects at the step boundaries of later calls
    (None switches it off)."""
    if events is None:
        _check(lib().beam_moe_set_stage_events(None, 0), "beam_moe_set_stage_events")
        return
    arr = (_P * len(events))(*[e.cuda_event for e in events])
    _check(lib().beam_moe_set_stage_events(arr, len(events)), "beam_moe_set_stage_events")


def set_debug(wait_limit_us: int = 0, withhold_first_load: bool = False) -> None:
    _check(lib().beam_moe_set_debug(int(wait_limit_us), int(bool(withhold_first_load))),
           "beam_moe_set_debug")


def kernels_per_forward(cfg, T: int, weight_fmt: int = 0, routed: bool = False) -> int:
    c = _cfg(cfg)
    return int(lib().beam_moe_kernels_per_forward(ctypes.byref(c), int(T), int(weight_fmt),
                                                  int(bool(routed))))


# ------------------------------------------------------------ expert parallelism
def ep_dispatch(cfg, hidden, router_w, corr_bias, n_ranks: int, ws: Workspace | None = None,
                stream=None):
    """Route this rank's tokens and pack one row per (token, slot) pair in
    owner order -> (send_x [T*k, d] bf16, send_expert [T*k] int32,
    send_w [T*k] f32, send_counts [n_ranks] int32, ws).  Keep ``ws`` for
    :func:`ep_combine`."""
    T = hidden.shape[0]
    dev = hidden.device
    ws = _ws(cfg, T, ws, dev)
    TK = T * cfg.topk
    send_x = torch.empty(TK, cfg.d, dtype=torch.bfloat16, device=dev)
    send_e = torch.empty(TK, dtype=torch.int32, device=dev)
    send_w = torch.empty(TK, dtype=torch.float32, device=dev)
    counts = torch.empty(n_ranks, dtype=torch.int32, device=dev)
    c = _cfg(cfg)
    _check(lib().beam_moe_ep_dispatch(ctypes.byref(c), _dev(hidden, torch.bfloat16, "hidden"),
                                      _dev(router_w, torch.float32, "router_w"),
                                      _dev(corr_bias, torch.float32, "corr_bias"), T,
                                      int(n_ranks), send_x.data_ptr(), send_e.data_ptr(),
                                      send_w.data_ptr(), counts.data_ptr(), ws.ptr, ws.nbytes,
                                      _stream(stream)), "beam_moe_ep_dispatch")
    return send_x, send_e, send_w, counts, ws


class EpWorkspace:
    """Device workspace of :func:`ep_experts` for up to M_max received rows."""

    def __init__(self, cfg, n_ranks: int, M_max: int, device=None, weight_fmt: int = 0):
        c = _cfg(cfg)
        self.nbytes = int(lib().beam_moe_ep_workspace_size(ctypes.byref(c), int(n_ranks),
                                                           int(M_max), int(weight_fmt)))
        self.weight_fmt = int(weight_fmt)
        if self.nbytes == 0:
            raise BeamError(1, "beam_moe_ep_workspace_size")
        self.M_max = int(M_max)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8,
                               device=device if device is not None else torch.device("cuda"))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def ep_experts(cfg, n_ranks: int, rank: int, x_recv, expert_recv, w_recv, w_gate, w_up, w_down,
               ws: EpWorkspace | None = None, out=None, stream=None):
    """This rank's experts on its received rows -> y_recv [M, d] f32 (weighted)."""
    M = x_recv.shape[0]
    dev = x_recv.device
    if ws is None or ws.M_max < M:
        ws = EpWorkspace(cfg, n_ranks, max(M, 1), dev)
    y = torch.empty(M, cfg.d, dtype=torch.float32, device=dev) if out is None else out
    if M == 0:
        return y
    c = _cfg(cfg)
    _check(lib().beam_moe_ep_experts(ctypes.byref(c), int(n_ranks), int(rank),
                                     _dev(x_recv, torch.bfloat16, "x_recv"),
                                     _dev(expert_recv, torch.int32, "expert_recv"),
                                     _dev(w_recv, torch.float32, "w_recv"),
                                     _dev(w_gate, torch.bfloat16, "w_gate"),
                                     _dev(w_up, torch.bfloat16, "w_up"),
                                     _dev(w_down, torch.bfloat16, "w_down"),
                                     _dev(y, torch.float32, "y_recv"), M, ws.ptr, ws.nbytes,
                                     _stream(stream)), "beam_moe_ep_experts")
    return y


def ep_experts_nvfp4(cfg, n_ranks: int, rank: int, x_recv, expert_recv, w_recv, gate: Fp4Weight,
                     up: Fp4Weight, down: Fp4Weight, ws: EpWorkspace | None = None, out=None,
                     stream=None):
    """This rank's NVFP4 experts on its received rows -> y_recv [M, d] f32."""
    M = x_recv.shape[0]
    dev = x_recv.device
    if ws is None or ws.M_max < M or ws.weight_fmt != NVFP4:
        ws = EpWorkspace(cfg, n_ranks, max(M, 1), dev, weight_fmt=NVFP4)
    y = torch.empty(M, cfg.d, dtype=torch.float32, device=dev) if out is None else out
    if M == 0:
        return y
    c = _cfg(cfg)
    _check(lib().beam_moe_ep_experts_nvfp4(ctypes.byref(c), int(n_ranks), int(rank),
                                           _dev(x_recv, torch.bfloat16, "x_recv"),
                                           _dev(expert_recv, torch.int32, "expert_recv"),
                                           _dev(w_recv, torch.float32, "w_recv"),
                                           ctypes.byref(gate._c), ctypes.byref(up._c),
                                           ctypes.byref(down._c),
                                           _dev(y, torch.float32, "y_recv"), M, ws.ptr,
                                           ws.nbytes, _stream(stream)),
           "beam_moe_ep_experts_nvfp4")
    return y


def ep_experts_fp8(cfg, n_ranks: int, rank: int, x_recv, expert_recv, w_recv, gate: Fp8Weight,
                   up: Fp8Weight, down: Fp8Weight, ws: EpWorkspace | None = None, out=None,
                   stream=None):
    """This rank's dynamic-FP8 experts on its received rows -> y_recv [M, d] f32."""
    M = x_recv.shape[0]
    dev = x_recv.device
    if ws is None or ws.M_max < M or ws.weight_fmt != FP8:
        ws = EpWorkspace(cfg, n_ranks, max(M, 1), dev, weight_fmt=FP8)
    y = torch.empty(M, cfg.d, dtype=torch.float32, device=dev) if out is None else out
    if M == 0:
        return y
    c = _cfg(cfg)
    _check(lib().beam_moe_ep_experts_fp8(ctypes.byref(c), int(n_ranks), int(rank),
                                         _dev(x_recv, torch.bfloat16, "x_recv"),
                                         _dev(expert_recv, torch.int32, "expert_recv"),
                                         _dev(w_recv, torch.float32, "w_recv"),
                                         ctypes.byref(gate._c), ctypes.byref(up._c),
                                         ctypes.byref(down._c),
                                         _dev(y, torch.float32, "y_recv"), M, ws.ptr,
                                         ws.nbytes, _stream(stream)),
           "beam_moe_ep_experts_fp8")
    return y


def ep_combine(cfg, y_back, T: int, ws: Workspace, out=None, stream=None):
    """The owner's combine of the returned rows -> out [T, d] bf16."""
    dev = ws.buf.device
    o = torch.empty(T, cfg.d, dtype=torch.bfloat16, device=dev) if out is None else out
    if T == 0:
        return o
    c = _cfg(cfg)
    _check(lib().beam_moe_ep_combine(ctypes.byref(c), _dev(y_back, torch.float32, "y_back"), T,
                                     o.data_ptr(), ws.ptr, ws.nbytes, _stream(stream)),
           "beam_moe_ep_combine")
    return o
