"""fp64 CPU oracle for the fused attention + All-to-All path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline /
reference legs may import this package. It shares no code with the CUDA path
(``comm_comp_fusion_gb300``) and never imports it; the CUDA path never imports
this. The arithmetic lives in ``xs_oracle.c`` (plain C, fp64, libm ``exp``);
this file only compiles it and marshals numpy arrays.

Passages followed (X-Stage paper, arXiv 2607.23264v1):
  * section 4.3 -- full, non-causal softmax attention of the DiT setting;
  * section 4.3, Figure 5 (d-e) -- the Ulysses post-attention All-to-All that
    turns the head partition back into the sequence partition;
  * section 5.3 -- "Serial" = attention followed by that All-to-All, which is
    exactly what ``attention_a2a`` returns;
  * section 4.3's contrast with "the causal attention used by typical
    autoregressive LLMs" -- ``causal=True`` restricts query token i to keys
    0..i (the standard autoregressive mask; the pages do not write it out).

Every function here is pinned by ``tests/test_oracle.py`` against brute force,
closed forms, invariants and hand-derived fixtures in ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xs_oracle.c")
_LIB = os.path.join(_HERE, "libxs_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libxs_oracle.so`` next to its source (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        lib.xs_oracle_attention.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ctypes.c_int]
        lib.xs_oracle_attention.restype = ctypes.c_int
        lib.xs_oracle_attention_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp, i64, vp,
                                                 ctypes.c_int]
        lib.xs_oracle_attention_rows.restype = ctypes.c_int
        lib.xs_oracle_attention_a2a.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ctypes.c_int]
        lib.xs_oracle_attention_a2a.restype = ctypes.c_int
        ci = ctypes.c_int
        lib.xs_oracle_attention_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ci, ci]
        lib.xs_oracle_attention_ex.restype = ci
        lib.xs_oracle_attention_rows_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, ci, vp, i64, vp, ci]
        lib.xs_oracle_attention_rows_ex.restype = ci
        lib.xs_oracle_attention_a2a_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, ci, ci]
        lib.xs_oracle_attention_a2a_ex.restype = ci
        lib.xs_oracle_e4m3_decode.argtypes = [vp, vp, i64]
        lib.xs_oracle_e4m3_decode.restype = ci
        lib.xs_oracle_attention_q8.argtypes = [vp, vp, vp, ci, vp, i64, i64, i64, i64, i64, dbl, ci, ci]
        lib.xs_oracle_attention_q8.restype = ci
        lib.xs_oracle_attention_rows_q8.argtypes = [vp, vp, vp, ci, i64, i64, i64, i64, i64, dbl, ci, vp, i64, vp,
                                                    ci]
        lib.xs_oracle_attention_rows_q8.restype = ci
        lib.xs_oracle_a2a.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64]
        lib.xs_oracle_a2a.restype = ctypes.c_int
        lib.xs_oracle_a2a_inverse.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64]
        lib.xs_oracle_a2a_inverse.restype = ctypes.c_int
        lib.xs_oracle_head_offset.argtypes = [i64] * 10
        lib.xs_oracle_head_offset.restype = i64
        lib.xs_oracle_seq_offset.argtypes = [i64] * 9
        lib.xs_oracle_seq_offset.restype = i64
        lib.xs_oracle_default_threads.argtypes = []
        lib.xs_oracle_default_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return a


def _check(rc):
    if rc < 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return rc


def default_threads() -> int:
    return _load().xs_oracle_default_threads()


def attention(q, k, v, B, S, H, D, P, scale, nthreads=0, return_threads=False, causal=False):
    """Head-partitioned fp64 attention output, shape [P][B][S][H/P][D]; with
    causal=True query token i sees keys 0..i only."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    out = np.empty((P, B, S, H // P, D), dtype=np.float64)
    used = _check(_load().xs_oracle_attention_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                                 out.ctypes.data, B, S, H, D, P, float(scale), int(causal),
                                                 nthreads))
    return (out, used) if return_threads else out


def attention_rows(q, k, v, B, S, H, D, P, scale, rows, nthreads=0, return_threads=False, causal=False):
    """fp64 attention for selected head-partitioned rows ((r*B+b)*S+s)*Hl+hl -> [n][D]."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, D), dtype=np.float64)
    used = _check(_load().xs_oracle_attention_rows_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                                      B, S, H, D, P, float(scale), int(causal), rows.ctypes.data,
                                                      rows.size, out.ctypes.data, nthreads))
    return (out, used) if return_threads else out


def attention_a2a(q, k, v, B, S, H, D, P, scale, nthreads=0, causal=False):
    """Attention then the All-to-All, fp64, shape [P][B][S/P][H][D]."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    out = np.empty((P, B, S // P, H, D), dtype=np.float64)
    _check(_load().xs_oracle_attention_a2a_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                              out.ctypes.data, B, S, H, D, P, float(scale), int(causal), nthreads))
    return out


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("E4M3 inputs are bytes (numpy uint8)")
    return a


def e4m3_decode(codes):
    """OFP8 E4M3 bytes -> float64 values (NaN for the NaN codes)."""
    codes = _u8(codes)
    out = np.empty(codes.shape, dtype=np.float64)
    _check(_load().xs_oracle_e4m3_decode(codes.ctypes.data, out.ctypes.data, codes.size))
    return out


def _v_any(v):
    """v as bf16 bit patterns (uint16) or, when given as uint8, E4M3 bytes; -> (array, is_e4m3)."""
    v = np.asarray(v)
    return (_u8(v), 1) if v.dtype == np.uint8 else (_u16(v), 0)


def attention_q8(q8, k8, v, B, S, H, D, P, scale, causal=False, nthreads=0):
    """Head-partitioned fp64 attention with q and k given as E4M3 bytes; v is bf16
    (uint16 bit patterns) or E4M3 (uint8 bytes)."""
    q8, k8 = _u8(q8), _u8(k8)
    v, v8 = _v_any(v)
    out = np.empty((P, B, S, H // P, D), dtype=np.float64)
    _check(_load().xs_oracle_attention_q8(q8.ctypes.data, k8.ctypes.data, v.ctypes.data, v8, out.ctypes.data,
                                          B, S, H, D, P, float(scale), int(causal), nthreads))
    return out


def attention_rows_q8(q8, k8, v, B, S, H, D, P, scale, rows, causal=False, nthreads=0):
    """fp64 attention with E4M3 q and k (v bf16 or E4M3, as for attention_q8) for
    selected head-partitioned rows -> [n][D]."""
    q8, k8 = _u8(q8), _u8(k8)
    v, v8 = _v_any(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, D), dtype=np.float64)
    _check(_load().xs_oracle_attention_rows_q8(q8.ctypes.data, k8.ctypes.data, v.ctypes.data, v8, B, S, H, D, P,
                                               float(scale), int(causal), rows.ctypes.data, rows.size,
                                               out.ctypes.data, nthreads))
    return out


def a2a(x, B, S, H, D, P):
    """Head-partitioned [P][B][S][H/P][D] -> sequence-partitioned [P][B][S/P][H][D], any dtype."""
    x = np.ascontiguousarray(x)
    out = np.empty((P, B, S // P, H, D), dtype=x.dtype)
    _check(_load().xs_oracle_a2a(x.ctypes.data, out.ctypes.data, B, S, H, D, P, x.itemsize))
    return out


def a2a_inverse(y, B, S, H, D, P):
    """Sequence-partitioned [P][B][S/P][H][D] -> head-partitioned [P][B][S][H/P][D]."""
    y = np.ascontiguousarray(y)
    out = np.empty((P, B, S, H // P, D), dtype=y.dtype)
    _check(_load().xs_oracle_a2a_inverse(y.ctypes.data, out.ctypes.data, B, S, H, D, P, y.itemsize))
    return out


def head_offset(r, b, s, hl, d, B, S, H, D, P):
    return _load().xs_oracle_head_offset(r, b, s, hl, d, B, S, H, D, P)


def seq_offset(b, s, h, d, B, S, H, D, P):
    return _load().xs_oracle_seq_offset(b, s, h, d, B, S, H, D, P)
