"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def xs():
    import __graft_entry__
    __graft_entry__.build()
    import comm_comp_fusion_gb300 as m
    return m


def _declared_symbols():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(xs_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_and_binding_agree(xs):
    assert _declared_symbols() == sorted(xs.EXPORTS)


def test_library_exports_every_declared_symbol(xs):
    lib = ctypes.CDLL(xs._LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", xs._LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\S+)", out))
    assert set(_declared_symbols()) <= exported


def test_version(xs):
    assert xs.version() >= 100


# Fake but aligned, non-overlapping "device" addresses: argument checks must
# reject the call before anything dereferences them.
Q, K, V, O = 0x10000000, 0x20000000, 0x30000000, 0x40000000
GOOD = dict(B=1, S=256, H=8, D=64, P=4, scale=0.125)


def _attn(xs, fn, q=Q, k=K, v=V, o=O, **kw):
    a = dict(GOOD, **kw)
    return fn(q, k, v, o, a["B"], a["S"], a["H"], a["D"], a["P"], a["scale"], check=False)


@pytest.mark.parametrize("fn_name", ["attn_a2a", "attn"])
def test_attention_argument_checks(xs, fn_name):
    fn = getattr(xs, fn_name)
    assert _attn(xs, fn, q=0) == xs.XS_ERR_NULL
    assert _attn(xs, fn, o=0) == xs.XS_ERR_NULL
    assert "non-NULL" in xs.last_error()
    assert _attn(xs, fn, H=6, P=4) == xs.XS_ERR_SHAPE          # H % P
    assert _attn(xs, fn, S=131, P=2) == xs.XS_ERR_SHAPE        # S % P
    assert _attn(xs, fn, S=384, P=5, H=10) == xs.XS_ERR_SHAPE  # S % P
    assert _attn(xs, fn, H=0) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, P=0) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, B=-1) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, scale=float("nan")) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, scale=float("inf")) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, scale=0.0) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, scale=-0.125) == xs.XS_ERR_SHAPE
    assert _attn(xs, fn, D=512) == xs.XS_ERR_UNSUPPORTED
    assert "D=512" in xs.last_error()
    assert _attn(xs, fn, D=80) == xs.XS_ERR_UNSUPPORTED
    assert _attn(xs, fn, q=Q + 8) == xs.XS_ERR_ALIGN
    assert _attn(xs, fn, o=O + 2) == xs.XS_ERR_ALIGN
    assert _attn(xs, fn, o=Q + 64) == xs.XS_ERR_ALIAS
    assert _attn(xs, fn, o=V - 16) == xs.XS_ERR_ALIAS
    assert _attn(xs, fn, B=1 << 16, S=1 << 15, H=1 << 8) == xs.XS_ERR_SHAPE  # > 2^31 rows
    # empty calls enqueue nothing and succeed without a GPU
    assert _attn(xs, fn, B=0) == xs.XS_OK
    assert _attn(xs, fn, S=0) == xs.XS_OK


def test_workspace_argument_checks(xs):
    W = 0x50000000
    f = lambda ws=W, nb=1 << 26, **kw: xs.attn_a2a_ws(Q, K, V, O, kw.get("B", 1), kw.get("S", 256), 8, 64, 4, 0.125,
                                                      ws, nb, check=False)
    assert f(ws=None, nb=64) == xs.XS_ERR_WORKSPACE        # NULL with a size
    assert f(ws=W + 16) == xs.XS_ERR_WORKSPACE              # not 256-byte aligned
    assert f(ws=O) == xs.XS_ERR_WORKSPACE                   # overlaps out
    assert f(ws=V - 256, nb=4096) == xs.XS_ERR_WORKSPACE     # overlaps v
    assert f(B=0) == xs.XS_OK                               # empty call
    assert xs.attn_ws(0, K, V, O, 1, 256, 8, 64, 4, 0.1, W, 1 << 20, check=False) == xs.XS_ERR_NULL
    n = ctypes.c_size_t(7)
    assert xs.lib.xs_attn_workspace_size(1, 0, 8, 64, 4, ctypes.byref(n)) == xs.XS_OK and n.value == 0
    assert xs.lib.xs_attn_workspace_size(1, 102, 8, 64, 4, ctypes.byref(n)) == xs.XS_ERR_SHAPE
    assert xs.lib.xs_attn_workspace_size(1, 256, 8, 64, 4, None) == xs.XS_ERR_NULL


def test_ulysses_argument_checks(xs):
    W = 0x50000000
    f = lambda q=Q, o=O, ws=None, nb=0, **kw: xs.ulysses_attn(
        q, K, V, o, kw.get("B", 1), kw.get("S", 256), kw.get("H", 8), kw.get("D", 64), kw.get("P", 4),
        kw.get("scale", 0.125), ws, nb, check=False)
    assert f(q=0) == xs.XS_ERR_NULL
    assert f(H=6) == xs.XS_ERR_SHAPE
    assert f(S=202) == xs.XS_ERR_SHAPE                  # S % P
    assert f(S=100) == xs.XS_ERR_UNSUPPORTED            # Sl = 25 is not a multiple of 8
    assert f(D=512) == xs.XS_ERR_UNSUPPORTED
    assert f(P=16, H=16) == xs.XS_ERR_UNSUPPORTED and "P=16" in xs.last_error()
    assert f(o=Q + 32) == xs.XS_ERR_ALIAS
    assert f(o=O + 8) == xs.XS_ERR_ALIGN
    assert f(ws=None, nb=64) == xs.XS_ERR_WORKSPACE
    assert f(ws=W + 64, nb=1 << 20) == xs.XS_ERR_WORKSPACE
    assert f(B=0) == xs.XS_OK
    assert f(S=0, P=16, H=16) == xs.XS_ERR_UNSUPPORTED   # the rank limit holds for empty calls too


def test_permute_argument_checks(xs):
    f = lambda i=Q, o=O, B=1, S=256, H=8, D=64, P=4: xs.a2a_permute(i, o, B, S, H, D, P, check=False)
    assert f(i=0) == xs.XS_ERR_NULL
    assert f(H=6) == xs.XS_ERR_SHAPE
    assert f(S=6, P=4) == xs.XS_ERR_SHAPE
    assert f(D=32) == xs.XS_ERR_UNSUPPORTED
    assert f(o=O + 4) == xs.XS_ERR_ALIGN
    assert f(o=Q + 16) == xs.XS_ERR_ALIAS
    assert f(B=0) == xs.XS_OK
    assert f(S=4, P=2) != xs.XS_ERR_SHAPE   # no multiple-of-128 rule for the permute
    g = lambda i=Q, o=O, B=1, S=256, H=8, D=64, P=4: xs.a2a_permute_inverse(i, o, B, S, H, D, P, check=False)
    assert g(o=0) == xs.XS_ERR_NULL
    assert g(S=6, P=4) == xs.XS_ERR_SHAPE
    assert g(i=Q + 2) == xs.XS_ERR_ALIGN
    assert g(o=Q - 16) == xs.XS_ERR_ALIAS
    assert g(B=0) == xs.XS_OK


def test_selftest_rejects_bad_limit(xs):
    assert xs.selftest_wait_timeout(0) == xs.XS_ERR_SHAPE
    assert xs.selftest_wait_timeout(5_000_000) == xs.XS_ERR_SHAPE


def test_valid_call_without_gpu_fails_loudly(xs):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _attn(xs, xs.attn_a2a)
    assert st in (xs.XS_ERR_CUDA, xs.XS_ERR_UNSUPPORTED)
    assert xs.last_error()
    with pytest.raises(xs.XsError):
        xs.attn_a2a(Q, K, V, O, 1, 256, 8, 64, 4, 0.125)


def test_q8_argument_checks(xs):
    W = 0x50000000
    f = lambda q=Q, k=K, o=O, ws=None, nb=0, **kw: getattr(xs, kw.pop("fn", "attn_a2a_q8"))(
        q, k, V, o, kw.get("B", 1), kw.get("S", 256), kw.get("H", 8), kw.get("D", 128), kw.get("P", 4),
        kw.get("scale", 0.088), ws, nb, check=False)
    for fn in ("attn_a2a_q8", "attn_q8"):
        assert f(fn=fn, D=64) == xs.XS_ERR_UNSUPPORTED and "D=128" in xs.last_error()
        assert f(fn=fn, D=256) == xs.XS_ERR_UNSUPPORTED
        assert f(fn=fn, q=0) == xs.XS_ERR_NULL
        assert f(fn=fn, k=K + 8) == xs.XS_ERR_ALIGN
        assert f(fn=fn, scale=0.0) == xs.XS_ERR_SHAPE
        assert f(fn=fn, ws=None, nb=64) == xs.XS_ERR_WORKSPACE
        assert f(fn=fn, B=0) == xs.XS_OK
    g = lambda o=O, **kw: xs.attn_a2a_qkv8(Q, K, V, o, 1, 256, 8, kw.get("D", 128), 4, 0.088, None, 0,
                                           check=False)
    assert g(D=64) == xs.XS_ERR_UNSUPPORTED
    assert g(o=V + 262144 - 16) == xs.XS_ERR_ALIAS     # v8 holds one byte per element too
    assert xs.attn_qkv8(Q, K, 0, O, 1, 256, 8, 128, 4, 0.088, check=False) == xs.XS_ERR_NULL
    # q8 and k8 hold one byte per element: B*S*H*D = 262144 bytes here
    assert f(o=Q + 262144 - 16) == xs.XS_ERR_ALIAS
    assert f(o=K + 262144 - 16) == xs.XS_ERR_ALIAS
    assert f(o=V + 524288 - 16) == xs.XS_ERR_ALIAS
    assert f(ws=W, nb=1 << 20, k=W + (1 << 20) - 256) == xs.XS_ERR_WORKSPACE
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        # past the end of q8: only the missing GPU stops the call
        assert f(o=Q + 262144) in (xs.XS_ERR_CUDA, xs.XS_ERR_UNSUPPORTED)
        assert g(o=V + 262144) in (xs.XS_ERR_CUDA, xs.XS_ERR_UNSUPPORTED)


def test_host_buffer_argument_checks(xs):
    HQ, HK, HV, HO = 0x60000000, 0x70000000, 0x80000000, 0x90000000
    f = lambda hq=HQ, ho=HO, q=Q, o=O, **kw: xs.attn_a2a_host(hq, HK, HV, ho, q, K, V, o, kw.get("B", 1),
                                                              kw.get("S", 256), 8, kw.get("D", 64), 4, 0.125,
                                                              check=False)
    assert f(hq=0) == xs.XS_ERR_NULL and "host" in xs.last_error()
    assert f(ho=0) == xs.XS_ERR_NULL
    assert f(q=0) == xs.XS_ERR_NULL
    assert f(hq=Q + 64) == xs.XS_ERR_ALIAS       # host q inside device q
    assert f(ho=HV + 16) == xs.XS_ERR_ALIAS      # host out overlaps host v
    assert f(o=O + 8) == xs.XS_ERR_ALIGN
    assert f(D=80) == xs.XS_ERR_UNSUPPORTED
    assert f(B=0) == xs.XS_OK
    g = lambda hv=HV: xs.attn_host(HQ, HK, hv, HO, Q, K, V, O, 1, 256, 8, 64, 4, 0.125, check=False)
    assert g(hv=0) == xs.XS_ERR_NULL
    assert g(hv=O) == xs.XS_ERR_ALIAS
