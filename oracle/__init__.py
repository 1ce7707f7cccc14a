"""ctypes front end of the f64 CPU oracle (smoe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg; the product package never imports it, and
it imports nothing from the product package.

Every function takes numpy arrays that live on the host and returns f64
numpy arrays.  The arithmetic is in the C file; this module only moves
arrays in and out.  Definitions follow the S-MoE page "Metal Compute
Kernels" (sections "Fused FFN Kernels -- One Simdgroup Per Output Row",
"Coalesced Dense Matvec -- the Same Contract for bf16" and "Token-Batch
Fused FFN"); the C file lists the readings taken where that page is silent.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_L = ctypes.c_long


def lib():
    """Builds (if needed) and loads liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        h = ctypes.CDLL(path)
        h.oracle_set_threads.argtypes = [ctypes.c_int]
        h.oracle_set_threads.restype = ctypes.c_int
        h.oracle_get_threads.restype = ctypes.c_int
        h.oracle_code_at.argtypes = [_u8p, ctypes.c_int, _L]
        h.oracle_unpack.argtypes = [_u8p, ctypes.c_int, _L, _u8p]
        h.oracle_dequant.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double]
        h.oracle_dequant.restype = ctypes.c_double
        h.oracle_silu.argtypes = [ctypes.c_double]
        h.oracle_silu.restype = ctypes.c_double
        h.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        h.oracle_bf16_value.restype = ctypes.c_double
        h.oracle_qgemv.argtypes = [ctypes.c_int, _u8p, _f32p, _L, _L, _L, _f64p, _L, _L,
                                   _f64p, _f64p]
        h.oracle_gate_up.argtypes = [ctypes.c_int, _u8p, _f32p, _u8p, _f32p, _L, _L, _L,
                                     _f64p, _L, _L, _f64p, _f64p, _f64p, _f64p, _f64p]
        h.oracle_ffn.argtypes = [ctypes.c_int, _u8p, _f32p, _u8p, _f32p, _u8p, _f32p, _L,
                                 _L, _L, _f64p, _f64p, _f64p, _f64p]
        h.oracle_ffn_batch.argtypes = [ctypes.c_int, _u8p, _f32p, _u8p, _f32p, _u8p, _f32p,
                                       _L, _L, _L, _L, _f64p, _L, _L, _f64p, _f64p, _f64p]
        h.oracle_matvec_bf16.argtypes = [_u16p, _L, _L, _f64p, _L, _L, _f64p, _f64p]
        _lp = ctypes.POINTER(ctypes.c_long)
        h.oracle_topk.argtypes = [_f64p, _L, _L, _lp, _f64p]
        h.oracle_route.argtypes = [_u16p, _L, _L, _f64p, _L, _f64p, _f64p, _lp, _f64p]
        h.oracle_combine.argtypes = [_f64p, _f64p, _L, _L, _f64p, _f64p]
        _lib = h
    return _lib


def _c(a, dtype):
    """A C-contiguous array of `dtype` (the caller's array when it already is)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a, ptype):
    return a.ctypes.data_as(ptype) if a is not None else None


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def set_threads(n: int) -> int:
    return lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return lib().oracle_get_threads()


def silu(v: float) -> float:
    return lib().oracle_silu(float(v))


def dequant(code: int, bits: int, scale: float) -> float:
    return lib().oracle_dequant(int(code), int(bits), float(scale))


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(int(bits))


def unpack(packed, bits: int, n: int):
    """The first n codes of a packed byte stream, one uint8 per code."""
    packed = _c(packed, np.uint8).reshape(-1)
    if n * bits > packed.size * 8:
        raise ValueError("unpack: stream too short")
    out = np.empty(n, dtype=np.uint8)
    _check(lib().oracle_unpack(_p(packed, _u8p), bits, n, _p(out, _u8p)), "unpack")
    return out


def qgemv(bits, codes, scales, rows, cols, group, x, row0=0, nrows=None):
    """(y, sum|w*x|) for rows [row0, row0+nrows) of a packed [rows x cols] matrix."""
    nrows = rows - row0 if nrows is None else nrows
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    x = _c(x, np.float64).reshape(-1)
    if codes.size < rows * cols * bits // 8 or scales.size < rows * (cols // group) or x.size < cols:
        raise ValueError("qgemv: arrays smaller than the stated shape")
    y = np.empty(nrows)
    a = np.empty(nrows)
    _check(lib().oracle_qgemv(bits, _p(codes, _u8p), _p(scales, _f32p), rows, cols, group,
                              _p(x, _f64p), row0, nrows, _p(y, _f64p), _p(a, _f64p)),
           "qgemv")
    return y, a


def gate_up(bits, gate_codes, gate_scales, up_codes, up_scales, d_ff, d_model, group, x,
            row0=0, nrows=None):
    """dict(hidden, g, u, g_abs, u_abs) for hidden rows [row0, row0+nrows)."""
    nrows = d_ff - row0 if nrows is None else nrows
    gc, uc = _c(gate_codes, np.uint8), _c(up_codes, np.uint8)
    gs, us = _c(gate_scales, np.float32), _c(up_scales, np.float32)
    x = _c(x, np.float64).reshape(-1)
    out = {k: np.empty(nrows) for k in ("hidden", "g", "u", "g_abs", "u_abs")}
    _check(lib().oracle_gate_up(bits, _p(gc, _u8p), _p(gs, _f32p), _p(uc, _u8p),
                                _p(us, _f32p), d_ff, d_model, group, _p(x, _f64p), row0,
                                nrows, *(_p(out[k], _f64p) for k in
                                         ("hidden", "g", "u", "g_abs", "u_abs"))),
           "gate_up")
    return out


def ffn(bits, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
        d_model, d_ff, group, x):
    """(hidden[d_ff], out[d_model], out_abs[d_model]) for one token."""
    args = [_c(a, t) for a, t in ((gate_codes, np.uint8), (gate_scales, np.float32),
                                  (up_codes, np.uint8), (up_scales, np.float32),
                                  (down_codes, np.uint8), (down_scales, np.float32))]
    x = _c(x, np.float64).reshape(-1)
    hidden, out, out_abs = np.empty(d_ff), np.empty(d_model), np.empty(d_model)
    ptrs = [_p(a, _u8p if a.dtype == np.uint8 else _f32p) for a in args]
    _check(lib().oracle_ffn(bits, *ptrs, d_model, d_ff, group, _p(x, _f64p),
                            _p(hidden, _f64p), _p(out, _f64p), _p(out_abs, _f64p)), "ffn")
    return hidden, out, out_abs


def ffn_batch(bits, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales,
              T, d_model, d_ff, group, X, t0=0, nt=None):
    """(hidden[nt,d_ff], Y[nt,d_model], Y_abs[nt,d_model]) for tokens [t0, t0+nt)."""
    nt = T - t0 if nt is None else nt
    args = [_c(a, t) for a, t in ((gate_codes, np.uint8), (gate_scales, np.float32),
                                  (up_codes, np.uint8), (up_scales, np.float32),
                                  (down_codes, np.uint8), (down_scales, np.float32))]
    X = _c(X, np.float64).reshape(-1)
    if X.size < T * d_model:
        raise ValueError("ffn_batch: X smaller than T*d_model")
    hidden = np.empty((nt, d_ff))
    Y, Ya = np.empty((nt, d_model)), np.empty((nt, d_model))
    ptrs = [_p(a, _u8p if a.dtype == np.uint8 else _f32p) for a in args]
    _check(lib().oracle_ffn_batch(bits, *ptrs, T, d_model, d_ff, group, _p(X, _f64p), t0, nt,
                                  _p(hidden, _f64p), _p(Y, _f64p), _p(Ya, _f64p)),
           "ffn_batch")
    return hidden, Y, Ya


def matvec_bf16(w_bits, rows, cols, x, row0=0, nrows=None):
    """(y, sum|w*x|) for rows [row0, row0+nrows) of a [rows x cols] bf16 matrix."""
    nrows = rows - row0 if nrows is None else nrows
    w = _c(w_bits, np.uint16)
    x = _c(x, np.float64).reshape(-1)
    if w.size < rows * cols or x.size < cols:
        raise ValueError("matvec_bf16: arrays smaller than the stated shape")
    y, a = np.empty(nrows), np.empty(nrows)
    _check(lib().oracle_matvec_bf16(_p(w, _u16p), rows, cols, _p(x, _f64p), row0, nrows,
                                    _p(y, _f64p), _p(a, _f64p)), "matvec_bf16")
    return y, a


def topk(logits, k):
    """(expert indices in selection order, weights) from given logits: the k
    largest, ties to the lower index, NaN below every number; weights are a
    softmax over the selected logits."""
    v = _c(logits, np.float64).reshape(-1)
    idx = np.empty(k, dtype=np.int64)
    w = np.empty(k)
    _check(lib().oracle_topk(_p(v, _f64p), v.size, k, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                             _p(w, _f64p)), "topk")
    return idx, w


def route(g_bits, n_experts, d_model, x, k):
    """Router of a bf16 gate matrix [n_experts x d_model]:
    (logits, sum|g*x| per expert, indices, weights)."""
    g = _c(g_bits, np.uint16)
    x = _c(x, np.float64).reshape(-1)
    if g.size < n_experts * d_model or x.size < d_model:
        raise ValueError("route: arrays smaller than the stated shape")
    logits, a = np.empty(n_experts), np.empty(n_experts)
    idx = np.empty(k, dtype=np.int64)
    w = np.empty(k)
    _check(lib().oracle_route(_p(g, _u16p), n_experts, d_model, _p(x, _f64p), k, _p(logits, _f64p),
                              _p(a, _f64p), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), _p(w, _f64p)),
           "route")
    return logits, a, idx, w


def combine(expert_out, w):
    """(out, sum|w*y| per output) for the k rows of expert_out [k x d_model]."""
    eo = _c(expert_out, np.float64)
    wv = _c(w, np.float64).reshape(-1)
    k = wv.size
    d_model = eo.size // max(k, 1)
    out, a = np.empty(d_model), np.empty(d_model)
    _check(lib().oracle_combine(_p(eo, _f64p), _p(wv, _f64p), k, d_model, _p(out, _f64p), _p(a, _f64p)),
           "combine")
    return out, a


def host_threads() -> int:
    """Host cores this process may run on (sched_getaffinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
