"""Seeded synthetic inputs (PCG32 -> Box-Muller -> bf16) for tests and the bench.

This module holds none of the attention or All-to-All arithmetic; it only
produces reproducible bf16 tensors, returned as numpy ``uint16`` arrays holding
the bf16 bit patterns. The C source (``pcg_normal.c``) documents the recipe.

Workload recipe used by the tests and the bench: seed = 1000 + workload index,
stream 1 for Q, 2 for K, 3 for V, sigma as the workload states (1 for N(0,1),
sqrt(2) for N(0,2)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pcg_normal.c")
_LIB = os.path.join(_HERE, "libxsgen.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libxsgen.so`` next to its source (plain C, gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.xsgen_pcg32_raw.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_void_p, ctypes.c_int64]
        lib.xsgen_pcg32_raw.restype = None
        lib.xsgen_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        lib.xsgen_normal_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def pcg32_raw(seed: int, stream: int, n: int, skip: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    _load().xsgen_pcg32_raw(seed, stream, skip, out.ctypes.data, n)
    return out


def normal_bf16(seed: int, stream: int, shape, sigma: float = 1.0, nthreads: int = 0) -> np.ndarray:
    """bf16 bit patterns of sigma * N(0,1), C-contiguous, dtype uint16."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    _load().xsgen_normal_bf16(seed, stream, float(sigma), out.ctypes.data, n, nthreads)
    return out.reshape(shape)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for inspection only)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (for building test inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# The synthetic workloads: (B, S, H, D, P, sigma_qk, sigma_v, scale, name).
WORKLOADS = [
    dict(B=1, S=256, H=8, D=64, P=4, sigma_qk=1.0, sigma_v=1.0, scale=1.0 / 8.0,
         name="small: B=1 S=256 H=8 D=64 P=4"),
    dict(B=1, S=4096, H=24, D=128, P=8, sigma_qk=1.0, sigma_v=1.0, scale=128 ** -0.5,
         name="DiT: B=1 S=4096 H=24 D=128 P=8"),
    dict(B=1, S=8192, H=24, D=128, P=8, sigma_qk=1.0, sigma_v=1.0, scale=128 ** -0.5,
         name="B=1 S=8192 H=24 D=128 P=8"),
    dict(B=1, S=32768, H=16, D=128, P=8, sigma_qk=1.0, sigma_v=1.0, scale=128 ** -0.5,
         name="long video DiT: B=1 S=32768 H=16 D=128 P=8"),
    dict(B=2, S=16384, H=40, D=128, P=4, sigma_qk=2.0 ** 0.5, sigma_v=1.0, scale=128 ** -0.5,
         name="peaked: B=2 S=16384 H=40 D=128 P=4, Q,K ~ N(0,2)"),
    # shape variants (measured, not the headline): a sequence length that is
    # not a multiple of the 128-row tile, and head dimension 96
    dict(B=1, S=4032, H=24, D=128, P=8, sigma_qk=1.0, sigma_v=1.0, scale=128 ** -0.5,
         name="ragged DiT: B=1 S=4032 H=24 D=128 P=8"),
    dict(B=1, S=8192, H=32, D=96, P=8, sigma_qk=1.0, sigma_v=1.0, scale=96 ** -0.5,
         name="D=96: B=1 S=8192 H=32 D=96 P=8"),
    dict(B=1, S=8192, H=16, D=256, P=8, sigma_qk=1.0, sigma_v=1.0, scale=256 ** -0.5,
         name="D=256: B=1 S=8192 H=16 D=256 P=8"),
    # head dimension 64 at the flops of the S=8192 workload (H doubled)
    dict(B=1, S=8192, H=48, D=64, P=8, sigma_qk=1.0, sigma_v=1.0, scale=64 ** -0.5,
         name="D=64: B=1 S=8192 H=48 D=64 P=8"),
]


def workload_inputs(idx: int, nthreads: int = 0):
    """(q, k, v) bf16 bit arrays of shape [P][B][S][H/P][D] for workload ``idx``."""
    w = WORKLOADS[idx]
    shape = (w["P"], w["B"], w["S"], w["H"] // w["P"], w["D"])
    seed = 1000 + idx
    q = normal_bf16(seed, 1, shape, w["sigma_qk"], nthreads)
    k = normal_bf16(seed, 2, shape, w["sigma_qk"], nthreads)
    v = normal_bf16(seed, 3, shape, w["sigma_v"], nthreads)
    return q, k, v


def random_inputs(seed: int, P: int, B: int, S: int, H: int, D: int, sigma_qk: float = 1.0,
                  sigma_v: float = 1.0, nthreads: int = 0):
    shape = (P, B, S, H // P, D)
    return (normal_bf16(seed, 1, shape, sigma_qk, nthreads),
            normal_bf16(seed, 2, shape, sigma_qk, nthreads),
            normal_bf16(seed, 3, shape, sigma_v, nthreads))


# ------------------------------------------------------------ FP8 (E4M3) inputs
# OFP8 E4M3 (OCP 8-bit floating point specification): 1 sign bit, 4 exponent
# bits with bias 7, 3 mantissa bits, subnormals at exponent field 0, no
# infinities, S.1111.111 is NaN. Used only to turn the seeded normal draws into
# E4M3 bytes; the oracle decodes bytes with its own implementation.

def _e4m3_positive_values() -> np.ndarray:
    codes = np.arange(0x7F)
    e, m = codes >> 3, codes & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest finite E4M3 value (ties to the even code), saturating
    at +-448; returns the bytes (uint8)."""
    x = np.asarray(x, dtype=np.float64)
    vals = _e4m3_positive_values()
    a = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return (code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)).astype(np.uint8)


def normal_e4m3(seed: int, stream: int, shape, sigma: float = 1.0, nthreads: int = 0) -> np.ndarray:
    """E4M3 bytes of the seeded sigma * N(0,1) draw (its bf16 value rounded to E4M3)."""
    return f32_to_e4m3(bf16_bits_to_f32(normal_bf16(seed, stream, shape, sigma, nthreads)))
