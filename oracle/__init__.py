"""CPU oracle for the Beam MoE layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct C implementation (``beam_oracle.c``) of what
the CUDA path computes, loaded through ``ctypes``.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs may
import it.  The product package never imports it and shares no code with it;
the two meet only through the seeded input generator and plain arrays.

BF16 arrays cross this boundary as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import itertools
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "beam_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libbeam_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_router_logits.argtypes = [_P, _P, _I64, _I32, _I32, _P]
        lib.oracle_route.argtypes = [_P, _P, _I64, _I32, _I32, _I32, _I32, ctypes.c_float,
                                     _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_experts_bf16.argtypes = [_P, _I64, _I32, _I32, _I32, _I32, _P, _P,
                                            _P, _P, _P, _P, _I64, _P, _P]
        lib.oracle_experts_nvfp4.argtypes = [_P, _I64, _I32, _I32, _I32, _I32, _P, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _I32, _P, _I64, _P, _P]
        for name in ("oracle_e2m1_value", "oracle_e4m3_value"):
            getattr(lib, name).argtypes = [ctypes.c_uint8]
            getattr(lib, name).restype = ctypes.c_double
        for name in ("oracle_e2m1_encode", "oracle_e4m3_encode"):
            getattr(lib, name).argtypes = [ctypes.c_float]
            getattr(lib, name).restype = ctypes.c_uint8
        lib.oracle_bf16_round.argtypes = [ctypes.c_float]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_swiglu_bf16.argtypes = [_P, _I64, _I32, _I32, _P, _P, _P]
        lib.oracle_f16_round.argtypes = [ctypes.c_double]
        lib.oracle_f16_round.restype = ctypes.c_double
        lib.oracle_bf16_round_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_round_double.restype = ctypes.c_uint16
        lib.oracle_boundary.argtypes = [_P, _P, _P, _P, _I64, _I32, ctypes.c_double,
                                        ctypes.c_float, ctypes.c_float, _P, _P]
        lib.oracle_nvfp4_quantize.argtypes = [_P, _I64, _P, _P]
        lib.oracle_experts_fp8.argtypes = [_P, _I64, _I32, _I32, _I32, _I32, _P, _P,
                                           _P, _P, _P, _P, _P, _P,
                                           _I32, _P, _I64, _P, _P]
        lib.oracle_experts_fp8_ties.argtypes = [_P, _I64, _I32, _I32, _I32, _I32, _P, _P,
                                                _P, _P, _P, _P, _P, _P,
                                                ctypes.c_double, _P, _I64, _P, _P, _P, _P]
        lib.oracle_fp8_quantize_rows.argtypes = [_P, _I64, _I32, _P, _P]
        lib.oracle_experts_mxfp8.argtypes = [_P, _I64, _I32, _I32, _I32, _I32, _P, _P,
                                             _P, _P, _P, _P, _P, _P, _I32, ctypes.c_double,
                                             _P, _I64, _P, _P, _P, _P]
        lib.oracle_mx_quantize.argtypes = [_P, _I64, _P, _P]
        lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_value.restype = ctypes.c_double
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


# --------------------------------------------------------------------------
# scalars
# --------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(code))


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(code))


def e8m0_value(code: int) -> float:
    return float(_load().oracle_e8m0_value(code))


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(v))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(v))


def bf16_round(v: float) -> int:
    return int(_load().oracle_bf16_round(v))


def swiglu_bf16(x_bf16, wg, wu) -> np.ndarray:
    """One expert's h = bf16(silu(x W_g^T) * (x W_u^T)) for rows x [n, d];
    wg / wu [F, d]; BF16 bit patterns in and out."""
    x = _c(x_bf16, np.uint16)
    wg = _c(wg, np.uint16)
    wu = _c(wu, np.uint16)
    n, d = x.shape
    F = wg.shape[0]
    assert wg.shape == (F, d) and wu.shape == (F, d)
    h = np.zeros((n, F), np.uint16)
    rc = _load().oracle_swiglu_bf16(_ptr(x), n, d, F, _ptr(wg), _ptr(wu), _ptr(h))
    if rc:
        raise ValueError(f"oracle_swiglu_bf16 failed ({rc})")
    return h


def f16_round(v: float) -> float:
    """Nearest binary16 value (ties to even, subnormals, saturating at 65504)."""
    return float(_load().oracle_f16_round(v))


def bf16_round_double(v: float) -> int:
    """Nearest BF16 of a double (one rounding, ties to even)."""
    return int(_load().oracle_bf16_round_double(v))


def residual_coefficients(n: int) -> tuple[np.float32, np.float32]:
    """(c_h, c_x) of the n-th depth-scaled residual add: FP32 roundings of
    sqrt((n-1)/n) and 1/sqrt(n) ("vLLM 实现 Reflection Beam 501B MoE 模型 Day 0
    支持", section "MoE and residual stream")."""
    if n < 1:
        raise ValueError("the residual adds are numbered from 1")
    return np.float32(np.sqrt((n - 1) / n)), np.float32(1.0 / np.sqrt(n))


def boundary(m_bf16, h_bf16, g_post, g_pre, eps: float, n: int):
    """The sublayer boundary after the MoE branch (post-norm, n-th depth-scaled
    residual add, next pre-norm); BF16 bit patterns in and out ->
    (new residual h' [T, d], next input x [T, d])."""
    m = _c(m_bf16, np.uint16)
    h = _c(h_bf16, np.uint16)
    gp = _c(g_post, np.uint16).reshape(-1)
    gq = _c(g_pre, np.uint16).reshape(-1)
    T, d = m.shape
    assert h.shape == (T, d) and gp.size == d and gq.size == d
    c_h, c_x = residual_coefficients(n)
    h_out = np.zeros((T, d), np.uint16)
    x_out = np.zeros((T, d), np.uint16)
    rc = _load().oracle_boundary(_ptr(m), _ptr(h), _ptr(gp), _ptr(gq), T, d,
                                 float(np.float32(eps)), float(c_h), float(c_x), _ptr(h_out),
                                 _ptr(x_out))
    if rc:
        raise ValueError(f"oracle_boundary failed ({rc})")
    return h_out, x_out


def nvfp4_quantize(v: np.ndarray):
    """Activation quantiser: returns (packed codes uint8 [n/2], scales uint8 [n/16])."""
    v = _c(v, np.float32).reshape(-1)
    q = np.zeros(v.size // 2, np.uint8)
    sf = np.zeros(v.size // 16, np.uint8)
    rc = _load().oracle_nvfp4_quantize(_ptr(v), v.size, _ptr(q), _ptr(sf))
    if rc:
        raise ValueError("length must be a multiple of 16")
    return q, sf


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
def router_logits(x_bf16: np.ndarray, wr: np.ndarray) -> np.ndarray:
    """FP32 logits [T, E] of BF16 hidden rows x [T, d] against W_r [E, d]."""
    x = _c(x_bf16, np.uint16)
    wr = _c(wr, np.float32)
    T, d = x.shape
    E = wr.shape[0]
    assert wr.shape[1] == d
    out = np.zeros((T, E), np.float32)
    rc = _load().oracle_router_logits(_ptr(x), _ptr(wr), T, d, E, _ptr(out))
    if rc:
        raise ValueError(f"oracle_router_logits failed ({rc})")
    return out


def route(logits: np.ndarray, bias: np.ndarray, n_groups: int, topk_groups: int,
          topk: int, routed_scale: float) -> dict:
    """Group-limited selection.  Returns idx [T,k] int32, w [T,k] f32, the
    scores s and c [T,E], the kept-group mask [T,G] and the two margins."""
    lg = _c(logits, np.float32)
    b = _c(bias, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, topk), np.int32)
    w = np.zeros((T, topk), np.float32)
    s = np.zeros((T, E), np.float32)
    c = np.zeros((T, E), np.float32)
    keep = np.zeros((T, n_groups), np.uint8)
    em = np.zeros(T, np.float64)
    gm = np.zeros(T, np.float64)
    rc = _load().oracle_route(_ptr(lg), _ptr(b), T, E, n_groups, topk_groups, topk,
                              float(routed_scale), _ptr(idx), _ptr(w), _ptr(s), _ptr(c),
                              _ptr(keep), _ptr(em), _ptr(gm))
    if rc:
        raise ValueError(f"oracle_route failed ({rc})")
    return {"idx": idx, "w": w, "s": s, "c": c, "keep": keep.astype(bool),
            "expert_margin": em, "group_margin": gm}


def _tie_choices(order, score, n_take, tol):
    """The ways to take the first n_take entries of `order` (sorted best
    first by `score`) when scores closer than tol are read as tied: the
    entries before the tie run that straddles the cut are always taken, and
    any n_take minus that many of the run's members complete the choice."""
    n = len(order)
    if n_take >= n or score[order[n_take - 1]] - score[order[n_take]] >= tol:
        return [tuple(order[:n_take])]
    a = n_take - 1
    while a > 0 and score[order[a - 1]] - score[order[a]] < tol:
        a -= 1
    b = n_take
    while b + 1 < n and score[order[b]] - score[order[b + 1]] < tol:
        b += 1
    run = order[a:b + 1]
    return [tuple(order[:a]) + tuple(pick)
            for pick in itertools.combinations(run, n_take - a)]


def route_alternatives(r: dict, t: int, n_groups: int, topk_groups: int, topk: int,
                       routed_scale: float, tol: float, limit: int = 4096) -> list[dict]:
    """Every routing of token t that the selection would give if the choice
    scores it ranks (the group scores, then the experts' c) that lie closer
    than tol were tied, from this oracle's own scores r["s"], r["c"] (the
    output of route()).  Each entry: 'idx' (the experts, slot order by c
    descending, expert ascending) and 'w' (FP32 weights 2.5 * s / sum s of
    that set).  The first entry is the oracle's own choice when nothing is
    near a tie.  Used to accept a near-tie token routed to another valid set
    and to compute its output from that set."""
    s = np.asarray(r["s"][t], np.float32)
    c = np.asarray(r["c"][t], np.float32)
    E = c.size
    S = E // n_groups
    gs = np.zeros(n_groups, np.float32)
    for g in range(n_groups):
        top = sorted(range(g * S, (g + 1) * S), key=lambda e: (-float(c[e]), e))[:2]
        gs[g] = np.float32(c[top[0]]) + np.float32(c[top[1]])
    g_order = sorted(range(n_groups), key=lambda g: (-float(gs[g]), g))
    out, seen = [], set()
    for groups in _tie_choices(g_order, gs.astype(np.float64), topk_groups, tol):
        cand = sorted((e for g in groups for e in range(g * S, (g + 1) * S)),
                      key=lambda e: (-float(c[e]), e))
        for chosen in _tie_choices(cand, c.astype(np.float64), topk, tol):
            key = frozenset(chosen)
            if key in seen:
                continue
            seen.add(key)
            idx = np.array(sorted(chosen, key=lambda e: (-float(c[e]), e)), np.int32)
            ssum = 0.0
            for e in idx:
                ssum += float(s[e])
            w = np.array([np.float32(routed_scale * float(s[e]) / ssum) for e in idx],
                         np.float32)
            out.append({"idx": idx, "w": w})
            if len(out) > limit:
                raise ValueError(f"token {t}: more than {limit} near-tie routings")
    return out


def _expert_ptrs(ws, E: int):
    """Per-expert pointer table from a 3-D array or a list/dict of 2-D arrays
    (None / missing entries for experts nobody uses)."""
    arr = (ctypes.c_void_p * E)()
    keep = []
    if isinstance(ws, np.ndarray):
        ws = np.ascontiguousarray(ws)
        keep.append(ws)
        for e in range(E):
            arr[e] = ws[e].ctypes.data
        return arr, keep
    items = ws.items() if isinstance(ws, dict) else enumerate(ws)
    for e, a in items:
        if a is None:
            continue
        a = np.ascontiguousarray(a)
        keep.append(a)
        arr[e] = a.ctypes.data
    return arr, keep


def experts_bf16(x_bf16, idx, w, wg, wu, wd, n_experts: int, tokens=None,
                 out: np.ndarray | None = None, exact: bool = False):
    """Weighted SwiGLU experts + combine for BF16 weights; returns BF16 [T, d]
    (and, with ``exact``, also the float64 output before its final rounding).
    wg/wu: per expert [F, d] uint16; wd: per expert [d, F] uint16."""
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    pg, kg_ = _expert_ptrs(wg, n_experts)
    pu, ku_ = _expert_ptrs(wu, n_experts)
    pd, kd_ = _expert_ptrs(wd, n_experts)
    F = _infer_F(wg, d)
    if out is None:
        out = np.zeros((T, d), np.uint16)
    ex = np.zeros((T, d), np.float64) if exact else None
    tok = None if tokens is None else _c(tokens, np.int64)
    rc = _load().oracle_experts_bf16(_ptr(x), T, d, F, k, n_experts, _ptr(idx), _ptr(w),
                                     ctypes.cast(pg, _P), ctypes.cast(pu, _P),
                                     ctypes.cast(pd, _P), _ptr(tok),
                                     0 if tok is None else tok.size, _ptr(out), _ptr(ex))
    if rc:
        raise ValueError(f"oracle_experts_bf16 failed ({rc})")
    return (out, ex) if exact else out


ACT_BF16, ACT_NVFP4, ACT_F16 = 0, 1, 2


def experts_nvfp4(x_bf16, idx, w, gate, up, down, n_experts: int, act_quant=True,
                  tokens=None, out: np.ndarray | None = None, exact: bool = False):
    """NVFP4 experts.  gate/up/down are dicts with per-expert 'q' (packed
    codes [N, K/2]), 'sf' (E4M3 codes [N, K/16]) and 'gs' (float32 [E]).
    act_quant: True / ACT_NVFP4 quantises both GEMM inputs to NVFP4, False /
    ACT_BF16 keeps BF16 activations, ACT_F16 takes them in F16."""
    mode = int(act_quant) if not isinstance(act_quant, bool) else int(act_quant)
    if mode not in (ACT_BF16, ACT_NVFP4, ACT_F16):
        raise ValueError(f"unknown activation mode {act_quant}")
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    keep = []
    tabs = []
    for p in (gate, up, down):
        q, kq = _expert_ptrs(p["q"], n_experts)
        sf, ks = _expert_ptrs(p["sf"], n_experts)
        gs = _c(p["gs"], np.float32)
        keep += kq + ks + [gs]
        tabs += [ctypes.cast(q, _P), ctypes.cast(sf, _P), _ptr(gs)]
    F = _infer_F(gate["q"], d // 2)
    if out is None:
        out = np.zeros((T, d), np.uint16)
    ex = np.zeros((T, d), np.float64) if exact else None
    tok = None if tokens is None else _c(tokens, np.int64)
    rc = _load().oracle_experts_nvfp4(_ptr(x), T, d, F, k, n_experts, _ptr(idx), _ptr(w),
                                      *tabs, mode, _ptr(tok),
                                      0 if tok is None else tok.size, _ptr(out), _ptr(ex))
    if rc:
        raise ValueError(f"oracle_experts_nvfp4 failed ({rc})")
    return (out, ex) if exact else out


ACT_FP8 = 3


FP8_TIE_REL = 2.0 ** -16


def experts_fp8(x_bf16, idx, w, gate, up, down, n_experts: int, act_quant=True,
                tokens=None, out: np.ndarray | None = None, exact: bool = False,
                ties: bool = False, tie_rel: float = FP8_TIE_REL):
    """Dynamic FP8 experts.  gate/up/down are dicts with per-expert 'q' (E4M3
    codes [N, K]) and 's' (FP32 scale per output row [N]).  act_quant: True /
    ACT_FP8 quantises both GEMM inputs per row to E4M3 (x per token, h per
    (token, expert) row after its BF16 rounding); False / ACT_BF16 keeps BF16
    activations.

    With ``ties`` (FP8 activations only) it also returns the near ties of the
    h quantisation: elements whose FP32 value lies within ``tie_rel`` of a
    BF16 rounding midpoint, where a computation that differs from this one by
    less than that may take the other BF16 value and so another E4M3 code.
    Returns (out, exact, slack [T, d], scale_tie [T] bool): slack bounds how far
    each output moves under any such choices; scale_tie marks tokens whose
    row scale itself could move."""
    mode = int(act_quant)
    if mode not in (ACT_BF16, 1, ACT_FP8):
        raise ValueError(f"unknown activation mode {act_quant}")
    if ties and not mode:
        raise ValueError("near ties exist only with FP8 activations")
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    keep = []
    tabs = []
    for p in (gate, up, down):
        q, kq = _expert_ptrs(p["q"], n_experts)
        sc, ks = _expert_ptrs(p["s"], n_experts)
        keep += kq + ks
        tabs += [ctypes.cast(q, _P), ctypes.cast(sc, _P)]
    F = _infer_F(gate["q"], d)
    if out is None:
        out = np.zeros((T, d), np.uint16)
    ex = np.zeros((T, d), np.float64) if exact else None
    tok = None if tokens is None else _c(tokens, np.int64)
    if ties:
        ex = np.zeros((T, d), np.float64) if ex is None else ex
        slack = np.zeros((T, d), np.float64)
        flag = np.zeros(T, np.uint8)
        rc = _load().oracle_experts_fp8_ties(_ptr(x), T, d, F, k, n_experts, _ptr(idx), _ptr(w),
                                             *tabs, float(tie_rel), _ptr(tok),
                                             0 if tok is None else tok.size, _ptr(out), _ptr(ex),
                                             _ptr(slack), _ptr(flag))
        if rc:
            raise ValueError(f"oracle_experts_fp8_ties failed ({rc})")
        return out, ex, slack, flag.astype(bool)
    rc = _load().oracle_experts_fp8(_ptr(x), T, d, F, k, n_experts, _ptr(idx), _ptr(w),
                                    *tabs, 1 if mode else 0, _ptr(tok),
                                    0 if tok is None else tok.size, _ptr(out), _ptr(ex))
    if rc:
        raise ValueError(f"oracle_experts_fp8 failed ({rc})")
    return (out, ex) if exact else out


def experts_mxfp8(x_bf16, idx, w, gate, up, down, n_experts: int, act_quant=True,
                  tokens=None, out: np.ndarray | None = None, exact: bool = False,
                  ties: bool = False, tie_rel: float = FP8_TIE_REL):
    """MXFP8 experts.  gate/up/down are dicts with per-expert 'q' (E4M3 codes
    [N, K]) and 's' (E8M0 scale codes [N, K/32]).  act_quant: True quantises
    both GEMM inputs to MX blocks of 32 (x along d, the FP32 SwiGLU product
    along F); False keeps BF16 activations.  With ``ties`` (quantised
    activations only) also returns the near ties of the h quantisation, as
    experts_fp8 does: (out, exact, slack [T, d], scale_tie [T] bool)."""
    if ties and not act_quant:
        raise ValueError("near ties exist only with quantised activations")
    x = _c(x_bf16, np.uint16)
    T, d = x.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    keep = []
    tabs = []
    for p in (gate, up, down):
        q, kq = _expert_ptrs(p["q"], n_experts)
        sc, ks = _expert_ptrs(p["s"], n_experts)
        keep += kq + ks
        tabs += [ctypes.cast(q, _P), ctypes.cast(sc, _P)]
    F = _infer_F(gate["q"], d)
    if out is None:
        out = np.zeros((T, d), np.uint16)
    ex = np.zeros((T, d), np.float64) if (exact or ties) else None
    slack = np.zeros((T, d), np.float64) if ties else None
    flag = np.zeros(T, np.uint8) if ties else None
    tok = None if tokens is None else _c(tokens, np.int64)
    rc = _load().oracle_experts_mxfp8(_ptr(x), T, d, F, k, n_experts, _ptr(idx), _ptr(w), *tabs,
                                      1 if act_quant else 0, float(tie_rel), _ptr(tok),
                                      0 if tok is None else tok.size, _ptr(out), _ptr(ex),
                                      _ptr(slack), _ptr(flag))
    if rc:
        raise ValueError(f"oracle_experts_mxfp8 failed ({rc})")
    if ties:
        return out, ex, slack, flag.astype(bool)
    return (out, ex) if exact else out


def mx_quantize(v: np.ndarray):
    """The MX activation rule (E4M3 elements, one E8M0 scale per 32): returns
    (codes uint8 [n], scale codes uint8 [n/32])."""
    v = _c(v, np.float32).reshape(-1)
    q = np.zeros(v.size, np.uint8)
    sc = np.zeros(v.size // 32, np.uint8)
    if _load().oracle_mx_quantize(_ptr(v), v.size, _ptr(q), _ptr(sc)):
        raise ValueError("length must be a multiple of 32")
    return q, sc


def fp8_quantize_rows(x_bf16):
    """The FP8 path's activation rule on BF16 rows [n, cols]: returns (E4M3
    codes uint8 [n, cols], FP32 scale per row [n])."""
    x = _c(x_bf16, np.uint16)
    n, cols = x.shape
    q = np.zeros((n, cols), np.uint8)
    sc = np.zeros(n, np.float32)
    rc = _load().oracle_fp8_quantize_rows(_ptr(x), n, cols, _ptr(q), _ptr(sc))
    if rc:
        raise ValueError(f"oracle_fp8_quantize_rows failed ({rc})")
    return q, sc


def _infer_F(ws, inner: int) -> int:
    if isinstance(ws, np.ndarray):
        return int(ws.shape[1])
    items = ws.values() if isinstance(ws, dict) else ws
    for a in items:
        if a is not None:
            return int(np.asarray(a).shape[0])
    raise ValueError("no expert weights given")


def forward_bf16(x_bf16, wr, bias, wg, wu, wd, n_groups, topk_groups, topk,
                 routed_scale, tokens=None):
    """Whole layer: router -> selection -> experts -> combine.
    Returns (out uint16 [T,d], routing dict, logits)."""
    logits = router_logits(x_bf16, wr)
    r = route(logits, bias, n_groups, topk_groups, topk, routed_scale)
    out = experts_bf16(x_bf16, r["idx"], r["w"], wg, wu, wd, logits.shape[1], tokens=tokens)
    return out, r, logits


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    a = np.asarray(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
