"""Test infrastructure only: the fp64 CPU oracle of the NVFP4 MoE layer.

This package wraps ``oracle.c`` (a plain, slow, fp64 restatement of the layer
described on the pages) through ``ctypes``.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it; the
product path (``nvfp4_moe_decode_gb300``) never does, and the two share no
code.  Each function cites the passage it follows in ``oracle.c``.

Functions whose result has no independent pin are marked "parity unpinned";
at present every exported function has at least one pin in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(mutant: int = 0, out_path: Optional[str] = None, openmp: bool = True) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP when available).

    ``mutant`` > 0 plants one of the deliberate mistakes guarded by
    ``ORACLE_MUTANT`` in oracle.c; it is used only by the mutation tests.
    """
    out = out_path or _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", out, _SRC, "-lm"]
    if mutant:
        base.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    if openmp:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
            return out
        except subprocess.CalledProcessError:
            pass
    subprocess.run(base, check=True, capture_output=True)
    return out


def _declare(lib):
    c_int, c_float, c_double = ctypes.c_int, ctypes.c_float, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_e2m1_value.argtypes = [c_int]
    lib.oracle_e2m1_value.restype = c_double
    lib.oracle_e4m3_value.argtypes = [c_int]
    lib.oracle_e4m3_value.restype = c_double
    lib.oracle_bf16_value.argtypes = [c_int]
    lib.oracle_bf16_value.restype = c_double
    lib.oracle_dequant_nvfp4.argtypes = [vp, vp, c_float, c_int, c_int, vp]
    lib.oracle_dequant_nvfp4.restype = None
    lib.oracle_dequant_bf16.argtypes = [vp, c_int, c_int, vp]
    lib.oracle_dequant_bf16.restype = None
    lib.oracle_dense_gemv_nvfp4.argtypes = [vp, vp, c_float, c_int, c_int, vp, c_int, vp]
    lib.oracle_dense_gemv_nvfp4.restype = None
    lib.oracle_router_logits.argtypes = [vp, vp, c_int, c_int, c_int, vp]
    lib.oracle_router_logits.restype = None
    lib.oracle_select_topk.argtypes = [vp, c_int, c_int, c_int, vp, vp]
    lib.oracle_select_topk.restype = c_int
    lib.oracle_expert_ffn.argtypes = [vp, vp, vp, c_int, c_int, vp]
    lib.oracle_expert_ffn.restype = None
    lib.oracle_moe_forward.argtypes = (
        [vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp]
        + [c_int, c_int, vp, vp, c_float, vp, vp, c_float, vp, vp, vp, vp])
    lib.oracle_moe_forward.restype = c_int
    lib.oracle_select_topk_sink.argtypes = [vp, c_int, c_int, c_int, c_int, vp, vp, vp]
    lib.oracle_select_topk_sink.restype = c_int
    lib.oracle_moe_forward_sinks.argtypes = (
        [vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp]
        + [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp])
    lib.oracle_moe_forward_sinks.restype = c_int
    lib.oracle_round_bf16.argtypes = [c_double]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_prenorm.argtypes = [vp, vp, c_int, c_int, c_double, vp, vp]
    lib.oracle_prenorm.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = c_int
    lib.oracle_set_num_threads.argtypes = [c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.uint16, np.int16), a.dtype
    return a.view(np.uint16)


def e2m1_value(code: int, lib=None) -> float:
    return (lib or load()).oracle_e2m1_value(int(code))


def e4m3_value(code: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_value(int(code))


def bf16_value(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_value(int(bits))


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, tscale: float, lib=None) -> np.ndarray:
    """Canonical NVFP4 [N, K/2] codes + [N, K/16] e4m3 scales -> fp64 [N, K]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    assert scales.shape == (N, K // 16)
    W = np.empty((N, K), dtype=np.float64)
    (lib or load()).oracle_dequant_nvfp4(_ptr(codes), _ptr(scales), float(tscale), N, K, _ptr(W))
    return W


def dequant_bf16(w: np.ndarray, lib=None) -> np.ndarray:
    w = _u16(w)
    N, K = w.shape
    W = np.empty((N, K), dtype=np.float64)
    (lib or load()).oracle_dequant_bf16(_ptr(w), N, K, _ptr(W))
    return W


def dense_gemv_nvfp4(codes: np.ndarray, scales: np.ndarray, tscale: float, x: np.ndarray,
                     lib=None) -> np.ndarray:
    """y [T, N] fp64 = W x for canonical NVFP4 W [N, K] and bf16 bits x [T, K]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    x = _u16(x)
    N, K = codes.shape[0], codes.shape[1] * 2
    T = x.shape[0]
    assert scales.shape == (N, K // 16) and x.shape == (T, K)
    y = np.empty((T, N), dtype=np.float64)
    (lib or load()).oracle_dense_gemv_nvfp4(_ptr(codes), _ptr(scales), float(tscale), N, K, _ptr(x), T,
                                            _ptr(y))
    return y


def router_logits(x: np.ndarray, wr: np.ndarray, lib=None) -> np.ndarray:
    x, wr = _u16(x), _u16(wr)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    (lib or load()).oracle_router_logits(_ptr(x), _ptr(wr), T, H, E, _ptr(out))
    return out


def select_topk(logits: np.ndarray, top_k: int, lib=None):
    """Top-k (on fp32-rounded logits, lower index wins ties) + renormalised weights."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = logits.shape
    idx = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    rc = (lib or load()).oracle_select_topk(_ptr(logits), T, E, int(top_k), _ptr(idx), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle_select_topk failed ({rc})")
    return idx, w


def expert_ffn(W13: np.ndarray, W2: np.ndarray, xt: np.ndarray, lib=None) -> np.ndarray:
    W13 = np.ascontiguousarray(W13, dtype=np.float64)
    W2 = np.ascontiguousarray(W2, dtype=np.float64)
    xt = np.ascontiguousarray(xt, dtype=np.float64)
    H = W2.shape[0]
    I = W2.shape[1]
    assert W13.shape == (2 * I, H) and xt.shape == (H,)
    y = np.empty(H, dtype=np.float64)
    (lib or load()).oracle_expert_ffn(_ptr(W13), _ptr(W2), _ptr(xt), H, I, _ptr(y))
    return y


class ExpertWeights:
    """Host arrays of one expert.  NVFP4: canonical codes/scales + tensor scales;
    BF16: uint16 bit patterns of row-major weights."""

    def __init__(self, wtype: int, w13a, w13b, ts13, w2a, w2b, ts2):
        self.wtype = int(wtype)
        self.w13a = np.ascontiguousarray(w13a)
        self.w13b = None if w13b is None else np.ascontiguousarray(w13b)
        self.ts13 = float(ts13)
        self.w2a = np.ascontiguousarray(w2a)
        self.w2b = None if w2b is None else np.ascontiguousarray(w2b)
        self.ts2 = float(ts2)


def moe_forward(x: np.ndarray, wr: np.ndarray, experts: Sequence[Optional[ExpertWeights]],
                top_k: int, inter: int, shared: Optional[ExpertWeights] = None, lib=None):
    """The full layer in fp64.  ``experts`` has one entry per routed expert;
    an entry may be None when no token selects it (the oracle reports -2 if
    one is selected).  Returns (out fp64 [T,H], idx [T,k], w [T,k], logits)."""
    x, wr = _u16(x), _u16(wr)
    T, H = x.shape
    E = wr.shape[0]
    wtypes = {e.wtype for e in experts if e is not None}
    assert len(wtypes) <= 1, "one weight type per routed bank"
    wtype = wtypes.pop() if wtypes else 0
    keep = []  # keep arrays alive during the call

    def parr(getter):
        arr = (ctypes.c_void_p * E)()
        for i, ex in enumerate(experts):
            a = None if ex is None else getter(ex)
            if a is not None:
                keep.append(a)
                arr[i] = a.ctypes.data
            else:
                arr[i] = None
        return arr

    a13 = parr(lambda e: e.w13a)
    b13 = parr(lambda e: e.w13b)
    a2 = parr(lambda e: e.w2a)
    b2 = parr(lambda e: e.w2b)
    ts13 = np.array([1.0 if e is None else e.ts13 for e in experts], dtype=np.float32)
    ts2 = np.array([1.0 if e is None else e.ts2 for e in experts], dtype=np.float32)
    out = np.empty((T, H), dtype=np.float64)
    idx = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    s = shared
    nz = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = (lib or load()).oracle_moe_forward(
        _ptr(x), _ptr(wr), T, H, E, int(inter), int(top_k), wtype,
        ctypes.cast(a13, ctypes.c_void_p), ctypes.cast(b13, ctypes.c_void_p), _ptr(ts13),
        ctypes.cast(a2, ctypes.c_void_p), ctypes.cast(b2, ctypes.c_void_p), _ptr(ts2),
        1 if s is not None else 0, s.wtype if s is not None else 0,
        nz(s.w13a) if s else None, nz(s.w13b) if s else None, s.ts13 if s else 1.0,
        nz(s.w2a) if s else None, nz(s.w2b) if s else None, s.ts2 if s else 1.0,
        _ptr(out), _ptr(idx), _ptr(w), _ptr(logits))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward failed ({rc})")
    return out, idx, w, logits


def select_topk_sink(logits: np.ndarray, n_routed: int, top_k: int, lib=None):
    """Expert-sink routing: logits [T, E+S] (the last S columns the sinks).
    Returns (idx [T,k], w [T,k], sw [T,S])."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, R = logits.shape
    E, S = int(n_routed), R - int(n_routed)
    idx = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    sw = np.empty((T, S), dtype=np.float64)
    rc = (lib or load()).oracle_select_topk_sink(_ptr(logits), T, E, S, int(top_k), _ptr(idx), _ptr(w), _ptr(sw))
    if rc != 0:
        raise ValueError(f"oracle_select_topk_sink failed ({rc})")
    return idx, w, sw


def _bank_arrays(experts):
    n = len(experts)

    def parr(getter):
        arr = (ctypes.c_void_p * max(n, 1))()
        for i, ex in enumerate(experts):
            a = None if ex is None else getter(ex)
            arr[i] = None if a is None else a.ctypes.data
        return arr

    ts13 = np.array([1.0 if e is None else e.ts13 for e in experts] or [1.0], dtype=np.float32)
    ts2 = np.array([1.0 if e is None else e.ts2 for e in experts] or [1.0], dtype=np.float32)
    return (parr(lambda e: e.w13a), parr(lambda e: e.w13b), ts13, parr(lambda e: e.w2a),
            parr(lambda e: e.w2b), ts2)


def moe_forward_sinks(x: np.ndarray, wr: np.ndarray, experts: Sequence[Optional[ExpertWeights]], top_k: int,
                      inter: int, shared: Sequence[ExpertWeights], sink: bool, lib=None):
    """The layer with len(shared) shared experts (their own weight type) and,
    with ``sink``, expert-sink routing (wr has E + S rows).  Returns (out fp64
    [T,H], idx [T,k], w [T,k], sw [T,S], logits [T, E (+S)])."""
    x, wr = _u16(x), _u16(wr)
    T, H = x.shape
    E = len(experts)
    S = len(shared)
    R = wr.shape[0]
    assert R == E + (S if sink else 0)
    wtypes = {e.wtype for e in experts if e is not None}
    assert len(wtypes) <= 1, "one weight type per routed bank"
    wtype = wtypes.pop() if wtypes else 0
    stypes = {e.wtype for e in shared}
    assert len(stypes) <= 1, "one weight type per shared bank"
    swtype = stypes.pop() if stypes else 0
    ra, rb, rts13, r2a, r2b, rts2 = _bank_arrays(experts)
    sa, sb, sts13, s2a, s2b, sts2 = _bank_arrays(shared)
    out = np.empty((T, H), dtype=np.float64)
    idx = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    sw = np.empty((T, max(S, 1)), dtype=np.float64)
    logits = np.empty((T, R), dtype=np.float64)
    c = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
    rc = (lib or load()).oracle_moe_forward_sinks(
        _ptr(x), _ptr(wr), T, H, E, int(inter), int(top_k), wtype, c(ra), c(rb), _ptr(rts13), c(r2a), c(r2b),
        _ptr(rts2), S, 1 if sink else 0, swtype, c(sa), c(sb), _ptr(sts13), c(s2a), c(s2b), _ptr(sts2),
        _ptr(out), _ptr(idx), _ptr(w), _ptr(sw), _ptr(logits))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward_sinks failed ({rc})")
    return out, idx, w, sw[:, :S], logits


def round_bf16(v: float, lib=None) -> int:
    """Nearest bf16 (ties to even) of an fp64 value, as 16-bit pattern."""
    return int((lib or load()).oracle_round_bf16(float(v)))


def prenorm(x: np.ndarray, delta: Optional[np.ndarray], eps: float, lib=None):
    """Pre-norm residual step: (v, xn) bf16 bit patterns [T, H] with
    v = bf16(x + delta) and xn = bf16(v / sqrt(mean(v^2) + eps))."""
    x = _u16(x)
    T, H = x.shape
    d = None
    if delta is not None:
        d = _u16(delta)
        assert d.shape == x.shape
    v = np.empty((T, H), dtype=np.uint16)
    xn = np.empty((T, H), dtype=np.uint16)
    (lib or load()).oracle_prenorm(_ptr(x), None if d is None else _ptr(d), T, H, float(eps), _ptr(v), _ptr(xn))
    return v, xn


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    (lib or load()).oracle_set_num_threads(int(n))
