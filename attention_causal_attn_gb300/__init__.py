"""Python binding of libattn.so, the sm_103a fused RoPE + causal attention forward.

Argument marshalling only: every step of the computation runs in the CUDA
library (include/attn.h).  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing or the device is not an sm_103
GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

from ._build import INCLUDE, LIB, build

__all__ = ["attn_fwd", "attn_fwd_host", "attn_decode", "attn_bwd", "attn_fwd_blocksparse", "attn_bwd_blocksparse",
           "attn_fwd_local", "attn_bwd_local", "create_block_mask", "attn_rope_rotate", "attn_fwd_rotated", "attn_mask_schedule", "attn_fwd_schedule", "attn_build_tables", "attn_check", "attn_error_string", "attn_release_cache",
           "AttnError", "build", "load_library", "header_functions", "ATTN_STATUS"]

ATTN_STATUS = {
    "ATTN_OK": 0, "ATTN_ERR_NULL": -1, "ATTN_ERR_SHAPE": -2, "ATTN_ERR_ALIGN": -3,
    "ATTN_ERR_UNSUPPORTED": -4, "ATTN_ERR_CUDA": -5, "ATTN_ERR_TIMEOUT": -6, "ATTN_ERR_OOM": -7,
    "ATTN_ERR_NO_DEVICE": -8, "ATTN_ERR_SCRATCH": -9, "ATTN_ERR_NONFINITE": -10,
}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {attn_error_string(code)} ({code})")
        self.code = code


def load_library(path: str | None = None):
    """Load libattn.so (built by build()); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with attention_causal_attn_gb300.build()")
        lib = ctypes.CDLL(p)
        vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.attn_fwd.restype = i
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, d, d, vp]
        lib.attn_selftest_wait_timeout.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, d, ctypes.c_ulonglong, vp]
        lib.attn_fwd_noalloc.restype = i
        lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, d, d, vp]
        lib.attn_fwd_host.restype = i
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, d, d]
        lib.attn_rope_rotate.restype = i
        lib.attn_rope_rotate.argtypes = [vp, vp, i, i, i, i, d, vp]
        lib.attn_fwd_rotated.restype = i
        lib.attn_fwd_rotated.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_decode.restype = i
        lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, d, d, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd.argtypes = [vp] * 9 + [i] * 6 + [d, vp]
        lib.attn_fwd_blocksparse.restype = i
        lib.attn_fwd_blocksparse.argtypes = [vp] * 5 + [i] * 6 + [d, vp, vp, vp]
        lib.attn_bwd_blocksparse.restype = i
        lib.attn_bwd_blocksparse.argtypes = [vp] * 9 + [i] * 6 + [d, vp, vp, vp]
        lib.attn_fwd_local.restype = i
        lib.attn_fwd_local.argtypes = [vp] * 5 + [i] * 6 + [d, i, i, vp]
        lib.attn_bwd_local.restype = i
        lib.attn_bwd_local.argtypes = [vp] * 9 + [i] * 6 + [d, i, i, vp]
        lib.attn_build_tables.restype = i
        lib.attn_build_tables.argtypes = [i, i, d, d, ctypes.c_longlong, vp, vp, vp]
        lib.attn_mask_schedule.restype = i
        lib.attn_mask_schedule.argtypes = [vp, i, ctypes.c_longlong, i, vp, vp, vp]
        lib.attn_fwd_schedule.restype = i
        lib.attn_fwd_schedule.argtypes = [i, i, i, i, i, i, i, d, vp, vp, vp]
        lib.attn_check.restype = i
        lib.attn_check.argtypes = [vp]
        lib.attn_error_string.restype = ctypes.c_char_p
        lib.attn_error_string.argtypes = [i]
        lib.attn_release_cache.restype = None
        lib.attn_release_cache.argtypes = []
        if path is None:
            _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/*.h."""
    names = []
    for fn in sorted(os.listdir(INCLUDE)):
        if fn.endswith(".h"):
            text = open(os.path.join(INCLUDE, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)
    return names


def attn_error_string(code: int) -> str:
    return load_library().attn_error_string(int(code)).decode()


def _stream_handle(stream, device):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def attn_fwd(q, k, v, o=None, lse=None, *, causal: bool = True, rope_base=None, window_k=None,
             return_lse: bool = True, stream=None):
    """Fused RoPE + causal attention forward on BSHD bf16 CUDA tensors.

    q [B, S, Hq, D], k and v [B, S, Hkv, D].  Returns (o, lse): o [B, S, Hq, D]
    bf16 and lse [B, Hq, S] float32 (None when return_lse is False).  Runs on
    `stream` (default: the current stream of q's device).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor (BSHD)")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, S, Hkv, D] with q's B, S and D")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()
                                and tuple(lse.shape) == (B, Hq, S)):
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, Hq, S]")
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr() if lse is not None else None,
                          B, Hq, Hkv, S, D, int(bool(causal)),
                          float(rope_base) if rope_base else 0.0,
                          float(window_k) if window_k else 0.0,
                          _stream_handle(stream, q.device))
    if rc != 0:
        raise AttnError(rc, "attn_fwd")
    return o, lse


def attn_rope_rotate(x, rope_base: float, out=None, stream=None):
    """RoPE of a whole BSHD bf16 CUDA tensor in one pass; returns the rotated fp16 tensor."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 4 and x.is_contiguous()):
        raise ValueError("x must be a contiguous 4-D bf16 CUDA tensor (BSHD)")
    B, S, H, D = x.shape
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    lib = load_library()
    with torch.cuda.device(x.device):
        rc = lib.attn_rope_rotate(x.data_ptr(), out.data_ptr(), B, S, H, D, float(rope_base),
                                  _stream_handle(stream, x.device))
    if rc != 0:
        raise AttnError(rc, "attn_rope_rotate")
    return out


def attn_fwd_rotated(q_rot, k_rot, v, o=None, lse=None, *, causal: bool = True, return_lse: bool = True,
                     stream=None):
    """The forward on fp16 Q and K rotated by attn_rope_rotate (v bf16); returns (o, lse)."""
    import torch
    for name, t, dt in (("q_rot", q_rot, torch.float16), ("k_rot", k_rot, torch.float16), ("v", v, torch.bfloat16)):
        if not (t.is_cuda and t.dtype == dt and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D {dt} CUDA tensor (BSHD)")
    B, S, Hq, D = q_rot.shape
    Hkv = k_rot.shape[2]
    if o is None:
        o = torch.empty(q_rot.shape, dtype=torch.bfloat16, device=q_rot.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q_rot.device)
    lib = load_library()
    with torch.cuda.device(q_rot.device):
        rc = lib.attn_fwd_rotated(q_rot.data_ptr(), k_rot.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, B, Hq, Hkv, S, D, int(bool(causal)),
                                  _stream_handle(stream, q_rot.device))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_rotated")
    return o, lse


def attn_decode(q, k, v, o=None, lse=None, *, rope_base=None, window_k=None, return_lse: bool = True,
                stream=None):
    """One decode step: q [B, Hq, D] (position S-1) against caches k, v [B, S, Hkv, D]; returns (o, lse)."""
    import torch
    for name, t, nd in (("q", q, 3), ("k", k, 4), ("v", v, 4)):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == nd and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous {nd}-D bf16 CUDA tensor")
    B, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, S, Hkv, D] with q's B and D")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr() if lse is not None else None, B, Hq, Hkv, S, D,
                             float(rope_base) if rope_base else 0.0, float(window_k) if window_k else 0.0,
                             _stream_handle(stream, q.device))
    if rc != 0:
        raise AttnError(rc, "attn_decode")
    return o, lse


def attn_bwd(q, k, v, o, lse, dO, *, causal: bool = True, rope_base=None, stream=None, block_mask=None,
             window: int = 0, alibi: bool = False):
    """Gradients (dq, dk, dv) of the forward for upstream gradient dO; o and lse are the forward's outputs.

    block_mask: the (row_ptr, col_idx) of attn_fwd_blocksparse, or None for the dense forward.
    window / alibi: those of attn_fwd_local (its backward, attn_bwd_local); not with block_mask.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO)):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor (BSHD)")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, S, Hkv, D] with q's B, S and D")
    if tuple(o.shape) != tuple(q.shape) or tuple(dO.shape) != tuple(q.shape):
        raise ValueError("o and dO must have q's shape")
    if not (lse.is_cuda and lse.dtype == torch.float32 and tuple(lse.shape) == (B, Hq, S) and lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, Hq, S]")
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, S, D, 1 if causal else 0, float(rope_base) if rope_base else 0.0)
    if (window or alibi) and block_mask is not None:
        raise ValueError("block_mask does not combine with window / alibi")
    with torch.cuda.device(q.device):
        if window or alibi:
            rc = lib.attn_bwd_local(*args, int(window), 1 if alibi else 0, _stream_handle(stream, q.device))
        elif block_mask is None:
            rc = lib.attn_bwd(*args, _stream_handle(stream, q.device))
        else:
            import numpy as np
            rp = np.ascontiguousarray(block_mask[0], dtype=np.int32)
            ci = np.ascontiguousarray(block_mask[1], dtype=np.int32)
            if rp.shape != ((S + 127) // 128 + 1,):
                raise ValueError("row_ptr must have ceil(S/128) + 1 entries")
            rc = lib.attn_bwd_blocksparse(*args, rp.ctypes.data, ci.ctypes.data if ci.size else None,
                                          _stream_handle(stream, q.device))
    if rc != 0:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_bwd_local(q, k, v, o, lse, dO, *, causal: bool = True, rope_base=None, window: int = 0,
                   alibi: bool = False, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd_local with the same window and alibi; o, lse: its outputs."""
    if window < 0:
        raise ValueError("window must be >= 0")
    if not window and not alibi:
        return attn_bwd(q, k, v, o, lse, dO, causal=causal, rope_base=rope_base, stream=stream)
    return attn_bwd(q, k, v, o, lse, dO, causal=causal, rope_base=rope_base, stream=stream, window=window,
                    alibi=alibi)


def _check_bshd(q, k, v):
    """Shape checks shared by the bindings: BSHD bf16 CUDA tensors; returns (B, S, Hq, D, Hkv)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor (BSHD)")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, S, Hkv, D] with q's B, S and D")
    return B, S, Hq, D, Hkv


def create_block_mask(predicate, S: int, *, block: int = 128):
    """The CSR block mask (row_ptr, col_idx) of predicate(q_block, k_block) -> bool over ceil(S/block)
    blocks per side, evaluated once per block pair (int32 numpy arrays)."""
    import numpy as np
    nb = (S + block - 1) // block
    rows = [[kb for kb in range(nb) if predicate(qb, kb)] for qb in range(nb)]
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum([len(r) for r in rows])
    col_idx = np.array([c for r in rows for c in r], dtype=np.int32)
    return row_ptr, col_idx


def attn_fwd_blocksparse(q, k, v, row_ptr, col_idx, o=None, lse=None, *, causal: bool = False, rope_base=None,
                         return_lse: bool = True, stream=None):
    """The forward over a CSR block mask of 128 x 128 blocks (see create_block_mask); returns (o, lse)."""
    import numpy as np
    import torch
    B, S, Hq, D, Hkv = _check_bshd(q, k, v)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    if rp.shape != ((S + 127) // 128 + 1,):
        raise ValueError("row_ptr must have ceil(S/128) + 1 entries")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr() if lse is not None else None, B, Hq, Hkv, S, D,
                                      1 if causal else 0, float(rope_base) if rope_base else 0.0,
                                      rp.ctypes.data, ci.ctypes.data if ci.size else None,
                                      _stream_handle(stream, q.device))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_blocksparse")
    return o, lse


def attn_fwd_local(q, k, v, o=None, lse=None, *, causal: bool = True, rope_base=None, window: int = 0,
                   alibi: bool = False, return_lse: bool = True, stream=None):
    """The forward with a sliding window (|i - j| < window) and/or the ALiBi bias; returns (o, lse)."""
    import torch
    B, S, Hq, D, Hkv = _check_bshd(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_local(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr() if lse is not None else None, B, Hq, Hkv, S, D, 1 if causal else 0,
                                float(rope_base) if rope_base else 0.0, int(window), 1 if alibi else 0,
                                _stream_handle(stream, q.device))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_local")
    return o, lse


def attn_fwd_host(q, k, v, o=None, lse=None, *, causal: bool = True, rope_base=None, window_k=None,
                  return_lse: bool = True, device=None):
    """The forward on BSHD bf16 CPU tensors (pinned for overlapped copies), on `device` (default: current).

    Returns (o, lse) as CPU tensors; the call returns when both are filled.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.device.type == "cpu" and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CPU tensor (BSHD)")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, S, Hkv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, S, Hkv, D] with q's B, S and D")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, pin_memory=q.is_pinned())
    for name, t, shape, dt in (("o", o, (B, S, Hq, D), torch.bfloat16), ("lse", lse, (B, Hq, S), torch.float32)):
        if t is not None and not (t.device.type == "cpu" and t.dtype == dt and t.is_contiguous()
                                  and tuple(t.shape) == shape):
            raise ValueError(f"{name} must be a contiguous CPU tensor {shape} of {dt}")
    lib = load_library()
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr() if lse is not None else None,
                               B, Hq, Hkv, S, D, int(bool(causal)),
                               float(rope_base) if rope_base else 0.0,
                               float(window_k) if window_k else 0.0)
    if rc != 0:
        raise AttnError(rc, "attn_fwd_host")
    return o, lse


def attn_mask_schedule(row_ptr, bh: int, num_ctas: int):
    """The block-sparse forward's task schedule for a CSR mask: (tasks, offsets), int32; stream s of
    CTA c runs tasks[offsets[2c+s]:offsets[2c+s+1]], task t = query tile * bh + batch-head."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    nrows = len(rp) - 1
    ctas = ctypes.c_int(0)
    lib = load_library()
    rc = lib.attn_mask_schedule(rp.ctypes.data, nrows, int(bh), int(num_ctas), None, None, ctypes.byref(ctas))
    if rc != 0:
        raise AttnError(rc, "attn_mask_schedule")
    tasks = np.zeros(max(nrows * int(bh), 1), dtype=np.int32)
    offsets = np.zeros(2 * ctas.value + 1, dtype=np.int32)
    rc = lib.attn_mask_schedule(rp.ctypes.data, nrows, int(bh), int(num_ctas), tasks.ctypes.data, offsets.ctypes.data,
                                None)
    if rc != 0:
        raise AttnError(rc, "attn_mask_schedule")
    return tasks[: nrows * int(bh)], offsets


def attn_fwd_schedule(B: int, Hq: int, Hkv: int, S: int, D: int, causal: bool, num_ctas: int,
                      kv_window_bytes: float = 64 * 2 ** 20):
    """The forward's tile schedule: (words [units, 2] uint32, offsets [ctas + 1] int32); CTA c runs
    units offsets[c]:offsets[c+1], word x = qtile0 | qtile1 << 16, y = h0 | h1 << 8 | b << 16."""
    lib = load_library()
    ctas = ctypes.c_int(0)
    args = (int(B), int(Hq), int(Hkv), int(S), int(D), int(bool(causal)), int(num_ctas), float(kv_window_bytes))
    rc = lib.attn_fwd_schedule(*args, None, None, ctypes.byref(ctas))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_schedule")
    offsets = np.zeros(ctas.value + 1, dtype=np.int32)
    rc = lib.attn_fwd_schedule(*args, None, offsets.ctypes.data, None)
    if rc != 0:
        raise AttnError(rc, "attn_fwd_schedule")
    words = np.zeros((max(int(offsets[-1]), 1), 2), dtype=np.uint32)
    rc = lib.attn_fwd_schedule(*args, words.ctypes.data, None, None)
    if rc != 0:
        raise AttnError(rc, "attn_fwd_schedule")
    return words[: int(offsets[-1])], offsets


def attn_build_tables(S: int, D: int, rope_base: float, window_k=None, pos_offset: int = 0):
    """Host RoPE tables cos/sin [S, D/2] (float32) and window widths W_r [D/2] (int32)."""
    cos = np.zeros((S, D // 2), dtype=np.float32)
    sin = np.zeros((S, D // 2), dtype=np.float32)
    win = np.zeros(D // 2, dtype=np.int32)
    rc = load_library().attn_build_tables(S, D, float(rope_base), float(window_k) if window_k else 0.0,
                                          int(pos_offset), cos.ctypes.data, sin.ctypes.data, win.ctypes.data)
    if rc != 0:
        raise AttnError(rc, "attn_build_tables")
    return cos, sin, win


def attn_check(stream=None, device=None) -> None:
    """Synchronise the stream and raise if a kernel reported a bounded-wait timeout or a non-finite forward row."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        rc = load_library().attn_check(_stream_handle(stream, dev))
    if rc != 0:
        raise AttnError(rc, "attn_check")


def attn_release_cache() -> None:
    load_library().attn_release_cache()
