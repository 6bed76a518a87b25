"""CPU oracle for the fused RoPE + causal attention forward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg may import this package; the product path never does.  The
arithmetic lives in ``oracle.c`` (plain C, float64); this file compiles it
with gcc on first use and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, IEEE float64, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            i32p = ctypes.POINTER(ctypes.c_int)
            f64p = ctypes.POINTER(ctypes.c_double)
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p] + [ctypes.c_int] * 6 + [
                ctypes.c_double, ctypes.c_double, ctypes.c_longlong, ctypes.c_int, i32p, i32p, i32p, f64p, f64p]
            lib.oracle_pruned_terms.restype = ctypes.c_longlong
            lib.oracle_pruned_terms.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double]
            lib.oracle_window_widths.restype = None
            lib.oracle_window_widths.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, f64p]
            lib.oracle_rope_rotate.restype = None
            lib.oracle_rope_rotate.argtypes = [u16p] + [ctypes.c_int] * 4 + [ctypes.c_double, f64p]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [f64p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_double] + [f64p] * 3
            lib.oracle_attn_bwd_local.restype = ctypes.c_int
            lib.oracle_attn_bwd_local.argtypes = [f64p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int,
                                                                                   ctypes.c_int] + [f64p] * 3
            lib.oracle_attn_bwd_bs.restype = ctypes.c_int
            lib.oracle_attn_bwd_bs.argtypes = [f64p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int,
                                                                                  i32p, i32p] + [f64p] * 3
            lib.oracle_attn_rows_bs.restype = ctypes.c_int
            lib.oracle_attn_rows_bs.argtypes = [u16p, u16p, u16p] + [ctypes.c_int] * 6 + [
                ctypes.c_double, ctypes.c_int, i32p, i32p, ctypes.c_int, i32p, i32p, i32p, f64p, f64p]
            lib.oracle_attn_rows_local.restype = ctypes.c_int
            lib.oracle_attn_rows_local.argtypes = [u16p, u16p, u16p] + [ctypes.c_int] * 6 + [
                ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p, i32p, f64p, f64p]
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def threads() -> int:
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def attn_rows(q, k, v, rows_b, rows_h, rows_i, *, causal=True, rope_base=None, window_k=None, pos_offset=0):
    """O [n, D] and LSE [n] (float64) for the selected query rows.

    q: uint16 bf16 bits [B, S, Hq, D]; k, v: [B, S, Hkv, D].
    rope_base None/<=0 turns RoPE off; window_k None/<=0/inf turns the window off.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, S, Hkv, D) and v.shape == k.shape
    rb = np.ascontiguousarray(rows_b, dtype=np.int32)
    rh = np.ascontiguousarray(rows_h, dtype=np.int32)
    ri = np.ascontiguousarray(rows_i, dtype=np.int32)
    n = len(ri)
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_attn_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                              B, Hq, Hkv, S, D, int(bool(causal)),
                              float(rope_base) if rope_base else 0.0,
                              float(window_k) if window_k else 0.0, int(pos_offset), n,
                              _ptr(rb, ctypes.c_int), _ptr(rh, ctypes.c_int), _ptr(ri, ctypes.c_int),
                              _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def attn_full(q, k, v, **kw):
    """O [B, S, Hq, D] and LSE [B, Hq, S] (float64) for every query row."""
    B, S, Hq, D = q.shape
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(S), indexing="ij")
    o, lse = attn_rows(q, k, v, bb.ravel(), hh.ravel(), ii.ravel(), **kw)
    return o.reshape(B, Hq, S, D).transpose(0, 2, 1, 3).copy(), lse.reshape(B, Hq, S)


def rope_rotate(x, rope_base: float) -> np.ndarray:
    """Every row of x (uint16 bf16 bits [B, S, H, D]) rotated at its position s, float64 [B, S, H, D]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    B, S, H, D = x.shape
    out = np.empty(x.shape, dtype=np.float64)
    _load().oracle_rope_rotate(_ptr(x, ctypes.c_uint16), B, S, H, D, float(rope_base), _ptr(out, ctypes.c_double))
    return out


def pruned_terms(S: int, D: int, rope_base: float, window_k: float) -> int:
    """Cell-by-cell count of pruned (cell, pair) terms over the causal S x S triangle."""
    return int(_load().oracle_pruned_terms(S, D, float(rope_base), float(window_k)))


def window_widths(D: int, rope_base: float, window_k: float) -> np.ndarray:
    w = np.zeros(D // 2, dtype=np.float64)
    _load().oracle_window_widths(D, float(rope_base), float(window_k) if window_k else 0.0, _ptr(w, ctypes.c_double))
    return w


def bf16_to_f64(x) -> np.ndarray:
    """bf16 bits (uint16) widened exactly to float64."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attn_bwd(q, k, v, dO, *, causal=True, rope_base=None, block_mask=None, block=128, window=0, alibi=False):
    """dQ [B,S,Hq,D], dK, dV [B,S,Hkv,D] (float64) of sum(O * dO) for the attention forward.

    q, k, v, dO: uint16 bf16 bits (widened exactly) or float64 arrays, BSHD.
    block_mask: optional CSR (row_ptr, col_idx) over block x block tiles.
    window / alibi: the local forward's sliding window (|i-j| < window) and ALiBi bias.
    """
    def f64(a):
        return bf16_to_f64(a) if a.dtype == np.uint16 else np.ascontiguousarray(a, dtype=np.float64)
    q, k, v, dO = (f64(a) for a in (q, k, v, dO))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    args = (_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
            _ptr(dO, ctypes.c_double), B, Hq, Hkv, S, D, 1 if causal else 0, float(rope_base) if rope_base else 0.0)
    outs = (_ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double))
    if window or alibi:
        if block_mask is not None:
            raise ValueError("a block mask does not combine with window / alibi here")
        rc = _load().oracle_attn_bwd_local(*args, int(window), 1 if alibi else 0, *outs)
    elif block_mask is None:
        rc = _load().oracle_attn_bwd(*args, *outs)
    else:
        rp = np.ascontiguousarray(block_mask[0], dtype=np.int32)
        ci = np.ascontiguousarray(block_mask[1], dtype=np.int32) if len(block_mask[1]) else np.zeros(1, np.int32)
        rc = _load().oracle_attn_bwd_bs(*args, int(block), _ptr(rp, ctypes.c_int), _ptr(ci, ctypes.c_int), *outs)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dq, dk, dv


def attn_rows_bs(q, k, v, row_ptr, col_idx, rows_b, rows_h, rows_i, *, block=128, causal=False, rope_base=None):
    """Block-sparse attention for the listed rows: (O [n, D], LSE [n]) float64; CSR mask over blocks."""
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k, v))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32) if len(col_idx) else np.zeros(1, np.int32)
    rb, rh, ri = (np.ascontiguousarray(a, dtype=np.int32) for a in (rows_b, rows_h, rows_i))
    n = len(rb)
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().oracle_attn_rows_bs(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                     B, Hq, Hkv, S, D, 1 if causal else 0, float(rope_base) if rope_base else 0.0,
                                     int(block), _ptr(rp, ctypes.c_int), _ptr(ci, ctypes.c_int), n,
                                     _ptr(rb, ctypes.c_int), _ptr(rh, ctypes.c_int), _ptr(ri, ctypes.c_int),
                                     _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def attn_full_bs(q, k, v, row_ptr, col_idx, **kw):
    """Block-sparse O [B, S, Hq, D] and LSE [B, Hq, S] (float64) for every query row."""
    B, S, Hq, D = q.shape
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(S), indexing="ij")
    o, lse = attn_rows_bs(q, k, v, row_ptr, col_idx, bb.ravel(), hh.ravel(), ii.ravel(), **kw)
    return o.reshape(B, Hq, S, D).transpose(0, 2, 1, 3).copy(), lse.reshape(B, Hq, S)


def attn_rows_local(q, k, v, rows_b, rows_h, rows_i, *, causal=True, rope_base=None, window=0, alibi=False):
    """Sliding-window (|i-j| < window) and/or ALiBi attention for the listed rows: (O [n, D], LSE [n])."""
    q, k, v = (np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k, v))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    rb, rh, ri = (np.ascontiguousarray(a, dtype=np.int32) for a in (rows_b, rows_h, rows_i))
    n = len(rb)
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().oracle_attn_rows_local(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                        B, Hq, Hkv, S, D, 1 if causal else 0, float(rope_base) if rope_base else 0.0,
                                        int(window), 1 if alibi else 0, n, _ptr(rb, ctypes.c_int),
                                        _ptr(rh, ctypes.c_int), _ptr(ri, ctypes.c_int), _ptr(o, ctypes.c_double),
                                        _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return o, lse


def attn_full_local(q, k, v, **kw):
    """Sliding-window / ALiBi O [B, S, Hq, D] and LSE [B, Hq, S] (float64) for every query row."""
    B, S, Hq, D = q.shape
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(S), indexing="ij")
    o, lse = attn_rows_local(q, k, v, bb.ravel(), hh.ravel(), ii.ravel(), **kw)
    return o.reshape(B, Hq, S, D).transpose(0, 2, 1, 3).copy(), lse.reshape(B, Hq, S)
