"""Python binding of libxs.so: fused non-causal attention + Ulysses All-to-All scatter.

The names match the C ABI in ``include/xs.h``. This module only marshals
arguments: every step of the path runs in the library's CUDA kernels. There is
no fallback; if ``libxs.so`` is missing, importing the binding raises.

Arguments may be torch tensors (their ``data_ptr()`` is used; the current CUDA
stream of their device is used unless ``stream`` is given) or raw integer
device pointers. Shapes follow the C ABI:

    q, k, v  : head-partitioned     [P][B][S][H/P][D]  bf16
    out      : sequence-partitioned [P][B][S/P][H][D]  bf16   (attn_a2a, a2a_permute)
               head-partitioned     [P][B][S][H/P][D]  bf16   (attn)

``ulysses_attn`` takes q, k, v and out all sequence-partitioned (both
All-to-Alls fused); ``a2a_permute_inverse`` maps sequence- to head-partitioned.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH, build  # noqa: F401  (build is re-exported)

XS_OK = 0
XS_ERR_NULL = 1
XS_ERR_SHAPE = 2
XS_ERR_ALIGN = 3
XS_ERR_UNSUPPORTED = 4
XS_ERR_CUDA = 5
XS_ERR_TIMEOUT = 6
XS_ERR_ALIAS = 7
XS_ERR_WORKSPACE = 8

STATUS_NAMES = {0: "XS_OK", 1: "XS_ERR_NULL", 2: "XS_ERR_SHAPE", 3: "XS_ERR_ALIGN", 4: "XS_ERR_UNSUPPORTED",
                5: "XS_ERR_CUDA", 6: "XS_ERR_TIMEOUT", 7: "XS_ERR_ALIAS", 8: "XS_ERR_WORKSPACE"}

# Every symbol include/*.h declares.
EXPORTS = ("xs_attn_a2a", "xs_attn", "xs_a2a_permute", "xs_a2a_permute_inverse", "xs_ulysses_attn",
           "xs_attn_a2a_ws", "xs_attn_ws", "xs_attn_workspace_size", "xs_attn_a2a_noalloc", "xs_last_error",
           "xs_device_status", "xs_selftest_wait_timeout", "xs_version", "xs_attn_a2a_trace", "xs_attn_trace_layout",
           "xs_attn_causal_a2a", "xs_attn_causal", "xs_attn_a2a_q8", "xs_attn_q8",
           "xs_attn_a2a_qkv8", "xs_attn_qkv8", "xs_attn_a2a_host", "xs_attn_host",
           # include/xs_burst.h
           "xs_burst_rec_bytes", "xs_burst_gap")


class XsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class BurstStats(ctypes.Structure):
    """xs_burst_stats of include/xs_burst.h."""
    _fields_ = [("t_iss_mean_ns", ctypes.c_double), ("t_iss_max_ns", ctypes.c_double),
                ("t_period_ns", ctypes.c_double), ("sm_clock_mhz", ctypes.c_double),
                ("bursts_measured", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libxs.so is not built ({_LIB_PATH}); run comm_comp_fusion_gb300.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.xs_attn_a2a.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.xs_attn_a2a.restype = i
    lib.xs_attn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.xs_attn.restype = i
    lib.xs_a2a_permute.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.xs_a2a_permute.restype = i
    sz = ctypes.c_size_t
    lib.xs_a2a_permute_inverse.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.xs_a2a_permute_inverse.restype = ctypes.c_int
    lib.xs_ulysses_attn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_ulysses_attn.restype = ctypes.c_int
    lib.xs_attn_causal_a2a.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.xs_attn_causal_a2a.restype = i
    lib.xs_attn_causal.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.xs_attn_causal.restype = i
    lib.xs_attn_a2a_trace.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_a2a_trace.restype = i
    lib.xs_attn_trace_layout.argtypes = [i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(sz)]
    lib.xs_attn_trace_layout.restype = i
    lib.xs_burst_rec_bytes.argtypes = [i, i]
    lib.xs_burst_rec_bytes.restype = sz
    lib.xs_burst_gap.argtypes = [vp, sz, vp, sz, i, i, i, ctypes.c_double, i, i, i, i, ctypes.POINTER(BurstStats), vp]
    lib.xs_burst_gap.restype = ctypes.c_int
    lib.xs_attn_a2a_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_a2a_ws.restype = i
    lib.xs_attn_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_ws.restype = i
    lib.xs_attn_a2a_q8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_a2a_q8.restype = i
    lib.xs_attn_q8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_q8.restype = i
    lib.xs_attn_a2a_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_a2a_host.restype = i
    lib.xs_attn_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_host.restype = i
    lib.xs_attn_a2a_qkv8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_a2a_qkv8.restype = i
    lib.xs_attn_qkv8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.xs_attn_qkv8.restype = i
    lib.xs_attn_workspace_size.argtypes = [i, i, i, i, i, ctypes.POINTER(sz)]
    lib.xs_attn_workspace_size.restype = i
    lib.xs_attn_a2a_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.xs_attn_a2a_noalloc.restype = i
    lib.xs_last_error.argtypes = []
    lib.xs_last_error.restype = ctypes.c_char_p
    lib.xs_device_status.argtypes = [vp, i]
    lib.xs_device_status.restype = i
    lib.xs_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.xs_selftest_wait_timeout.restype = i
    lib.xs_version.argtypes = []
    lib.xs_version.restype = i
    return lib


lib = _load()


def last_error() -> str:
    return lib.xs_last_error().decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _hptr(x):
    """Address of a host buffer: a CPU torch tensor, a C-contiguous numpy array or an int."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if not x.flags["C_CONTIGUOUS"]:
        raise ValueError("host buffers must be C-contiguous")
    return x.ctypes.data


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else getattr(stream, "cuda_stream", stream)
    for t in tensors:
        if hasattr(t, "is_cuda") and t.is_cuda:
            import torch
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _check(status: int) -> int:
    if status != XS_OK:
        raise XsError(status, last_error())
    return status


def attn_a2a(q, k, v, out, B, S, H, D, P, scale, stream=None, check=True):
    """Fused attention + All-to-All scatter (``xs_attn_a2a``); returns the status."""
    st = lib.xs_attn_a2a(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale),
                         _stream(stream, q, out))
    return _check(st) if check else st


def attn(q, k, v, out, B, S, H, D, P, scale, stream=None, check=True):
    """Attention only, head-partitioned output (``xs_attn``); returns the status."""
    st = lib.xs_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _stream(stream, q, out))
    return _check(st) if check else st


def _nbytes(ws, ws_bytes):
    if ws_bytes is not None:
        return int(ws_bytes)
    if ws is None or isinstance(ws, int):
        return 0
    return ws.numel() * ws.element_size()


def attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, workspace, workspace_bytes=None, stream=None, check=True):
    """Fused call with the balanced schedule (``xs_attn_a2a_ws``); returns the status."""
    st = lib.xs_attn_a2a_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                            _nbytes(workspace, workspace_bytes), _stream(stream, q, out))
    return _check(st) if check else st


def attn_ws(q, k, v, out, B, S, H, D, P, scale, workspace, workspace_bytes=None, stream=None, check=True):
    """Attention only with the balanced schedule (``xs_attn_ws``); returns the status."""
    st = lib.xs_attn_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                        _nbytes(workspace, workspace_bytes), _stream(stream, q, out))
    return _check(st) if check else st


def attn_a2a_q8(q8, k8, v, out, B, S, H, D, P, scale, workspace=None, workspace_bytes=None, stream=None,
                check=True):
    """Fused call with E4M3 queries and keys (``xs_attn_a2a_q8``): q8, k8 uint8 codes, v bf16;
    ``workspace=None`` selects the whole-item schedule. Returns the status."""
    st = lib.xs_attn_a2a_q8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                            _nbytes(workspace, workspace_bytes), _stream(stream, v, out))
    return _check(st) if check else st


def attn_q8(q8, k8, v, out, B, S, H, D, P, scale, workspace=None, workspace_bytes=None, stream=None, check=True):
    """Attention only with E4M3 queries and keys (``xs_attn_q8``), head-partitioned output."""
    st = lib.xs_attn_q8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                        _nbytes(workspace, workspace_bytes), _stream(stream, v, out))
    return _check(st) if check else st


def attn_a2a_qkv8(q8, k8, v8, out, B, S, H, D, P, scale, workspace=None, workspace_bytes=None, stream=None,
                  check=True):
    """Fused call with E4M3 queries, keys and values (``xs_attn_a2a_qkv8``); bf16 output."""
    st = lib.xs_attn_a2a_qkv8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                              _nbytes(workspace, workspace_bytes), _stream(stream, v8, out))
    return _check(st) if check else st


def attn_qkv8(q8, k8, v8, out, B, S, H, D, P, scale, workspace=None, workspace_bytes=None, stream=None, check=True):
    """Attention only with E4M3 queries, keys and values (``xs_attn_qkv8``), head-partitioned output."""
    st = lib.xs_attn_qkv8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                          _nbytes(workspace, workspace_bytes), _stream(stream, v8, out))
    return _check(st) if check else st


def attn_a2a_host(q_host, k_host, v_host, out_host, q, k, v, out, B, S, H, D, P, scale, workspace=None,
                  workspace_bytes=None, stream=None, check=True):
    """Fused call on host-memory inputs and output (``xs_attn_a2a_host``): copies in,
    compute and copies out pipelined over rank chunks; q, k, v, out are device
    staging buffers. Host buffers are torch CPU tensors (pinned for overlap),
    numpy arrays or raw addresses."""
    st = lib.xs_attn_a2a_host(_hptr(q_host), _hptr(k_host), _hptr(v_host), _hptr(out_host), _ptr(q), _ptr(k),
                              _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                              _nbytes(workspace, workspace_bytes), _stream(stream, q, out))
    return _check(st) if check else st


def attn_host(q_host, k_host, v_host, out_host, q, k, v, out, B, S, H, D, P, scale, workspace=None,
              workspace_bytes=None, stream=None, check=True):
    """Attention only on host-memory inputs and output (``xs_attn_host``), pipelined like
    ``attn_a2a_host``."""
    st = lib.xs_attn_host(_hptr(q_host), _hptr(k_host), _hptr(v_host), _hptr(out_host), _ptr(q), _ptr(k), _ptr(v),
                          _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace), _nbytes(workspace, workspace_bytes),
                          _stream(stream, q, out))
    return _check(st) if check else st


def workspace_size(B, S, H, D, P) -> int:
    """``xs_attn_workspace_size`` for the current device, in bytes."""
    n = ctypes.c_size_t(0)
    _check(lib.xs_attn_workspace_size(B, S, H, D, P, ctypes.byref(n)))
    return n.value


def attn_a2a_noalloc(q, k, v, out, B, S, H, D, P, scale, stream=None, check=True):
    """Balanced fused call on the library's built-in scratch (``xs_attn_a2a_noalloc``),
    for callers that cannot allocate a workspace; returns the status."""
    st = lib.xs_attn_a2a_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale),
                                 _stream(stream, q, out))
    return _check(st) if check else st


def a2a_permute(inp, out, B, S, H, D, P, stream=None, check=True):
    """Standalone All-to-All layout pass (``xs_a2a_permute``); returns the status."""
    st = lib.xs_a2a_permute(_ptr(inp), _ptr(out), B, S, H, D, P, _stream(stream, inp, out))
    return _check(st) if check else st


def a2a_permute_inverse(inp, out, B, S, H, D, P, stream=None, check=True):
    """Standalone pre-attention All-to-All, sequence- to head-partitioned
    (``xs_a2a_permute_inverse``); returns the status."""
    st = lib.xs_a2a_permute_inverse(_ptr(inp), _ptr(out), B, S, H, D, P, _stream(stream, inp, out))
    return _check(st) if check else st


def ulysses_attn(q, k, v, out, B, S, H, D, P, scale, workspace=None, workspace_bytes=None, stream=None, check=True):
    """Attention with both Ulysses All-to-Alls fused (``xs_ulysses_attn``): q, k, v and
    out sequence-partitioned; ``workspace=None`` selects the whole-item schedule."""
    st = lib.xs_ulysses_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(workspace),
                             _nbytes(workspace, workspace_bytes), _stream(stream, q, out))
    return _check(st) if check else st


def attn_causal_a2a(q, k, v, out, B, S, H, D, P, scale, stream=None, check=True):
    """Causal attention with the All-to-All scatter (``xs_attn_causal_a2a``); returns the status."""
    st = lib.xs_attn_causal_a2a(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale),
                                _stream(stream, q, out))
    return _check(st) if check else st


def attn_causal(q, k, v, out, B, S, H, D, P, scale, stream=None, check=True):
    """Causal attention, head-partitioned output (``xs_attn_causal``); returns the status."""
    st = lib.xs_attn_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale),
                            _stream(stream, q, out))
    return _check(st) if check else st


def attn_a2a_trace(q, k, v, out, B, S, H, D, P, scale, trace, trace_bytes=None, stream=None, check=True):
    """Fused call with the epilogue traced (``xs_attn_a2a_trace``); returns the status."""
    st = lib.xs_attn_a2a_trace(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, P, float(scale), _ptr(trace),
                               _nbytes(trace, trace_bytes), _stream(stream, q, out))
    return _check(st) if check else st


def trace_layout(B, S, H, D, P):
    """``xs_attn_trace_layout``: (ctas, items_per_cta, trace bytes) on the current device."""
    c, n, b = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    _check(lib.xs_attn_trace_layout(B, S, H, D, P, ctypes.byref(c), ctypes.byref(n), ctypes.byref(b)))
    return c.value, n.value, b.value


def burst_gap(buf, buf_bytes, rec, rec_bytes, K, B, gap_ns, n_bursts, isolated=False, row_bytes=128,
              row_stride=128, warps=4, stream=None):
    """One Burst-Gap microbenchmark launch (``xs_burst_gap``); synchronises and returns
    a dict with t_iss_mean_ns, t_iss_max_ns, t_period_ns, sm_clock_mhz, bursts_measured."""
    st = BurstStats()
    _check(lib.xs_burst_gap(_ptr(buf), int(buf_bytes), _ptr(rec), int(rec_bytes), K, warps, B, float(gap_ns),
                            n_bursts, 1 if isolated else 0, row_bytes, row_stride, ctypes.byref(st),
                            _stream(stream, buf)))
    return {f: getattr(st, f) for f, _ in BurstStats._fields_}


def burst_rec_bytes(K, n_bursts) -> int:
    return lib.xs_burst_rec_bytes(K, n_bursts)


def device_status(stream=None, clear=True) -> int:
    """``xs_device_status``: synchronises the stream and reports in-kernel wait timeouts."""
    return lib.xs_device_status(_stream(stream), 1 if clear else 0)


def selftest_wait_timeout(timeout_us: int = 1000, stream=None) -> int:
    return lib.xs_selftest_wait_timeout(int(timeout_us), _stream(stream))


def version() -> int:
    return lib.xs_version()
