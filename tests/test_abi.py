"""The C-ABI library loads and exports every symbol include/mha.h declares,
and rejects bad arguments on the host, before any CUDA call (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

from masked_head_attention_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, DEVICE, TOO_LARGE = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def L():
    path = mbuild.build()
    lib = ctypes.CDLL(path)
    P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.mha_fwd.argtypes = [P, P, P, i, P, P, i, i, i, i, i, f, i, P]
    lib.prenorm_cross_attn_fwd.argtypes = [P, P, P, f, P, P, P, P, i, i, i, i, i, f, i, P]
    lib.mha_strerror.restype = ctypes.c_char_p
    lib.mha_selftest_umma.argtypes = [i, i, P, P, P, P]
    lib.mha_fwd_lse.argtypes = [P, P, P, i, P, P, P, i, i, i, i, i, f, i, P]
    lib.mha_bwd.argtypes = [P, P, P, P, P, P, i, P, P, P, P, i, i, i, i, i, f, i, P,
                            ctypes.c_size_t, P]
    lib.mha_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.mha_bwd_workspace_size.restype = ctypes.c_size_t
    lib.mha_test_set_device_status.argtypes = [i, ctypes.c_uint32]
    lib.mha_fwd_host.argtypes = [P, P, P, i, P, P, i, i, i, i, i, f, i, P, ctypes.c_size_t, P]
    lib.mha_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.mha_fwd_host_workspace_size.restype = ctypes.c_size_t
    return lib


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        names += re.findall(r"^MHA_API\s+[\w\s\*]*?\**\s*(\w+)\s*\(", text, re.M)
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("mha_fwd", "prenorm_cross_attn_fwd", "mha_strerror", "mha_device_status",
                 "mha_bwd", "mha_bwd_workspace_size", "mha_set_bf16_grid",
                 "mha_test_set_device_status", "mha_test_set_wait_limit_ns"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_strerror_covers_every_status(L):
    for code in (OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, DEVICE, TOO_LARGE):
        s = L.mha_strerror(code).decode()
        assert s and s != "unknown status"
    assert L.mha_strerror(12345).decode() == "unknown status"


# Fake, never-dereferenced addresses: every case below is rejected (or is a
# no-op) on the host before the library touches CUDA.
A = ctypes.c_void_p(0x10000)
A2 = ctypes.c_void_p(0x20000)
A3 = ctypes.c_void_p(0x30000)
OUT = ctypes.c_void_p(0x40000)
BAD = ctypes.c_void_p(0x40008)


def fwd(L, q=A, k=A2, v=A3, mask=0, lens=None, out=OUT, B=2, H=2, Lq=8, Lk=8, D=64,
        scale=0.125, dtype=1):
    return L.mha_fwd(q, k, v, mask, lens, out, B, H, Lq, Lk, D, scale, dtype, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), INVALID), (dict(out=None), INVALID), (dict(k=None), INVALID),
    (dict(B=-1), INVALID), (dict(Lk=-3), INVALID), (dict(scale=0.0), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=-1.0), INVALID),
    (dict(mask=4), INVALID), (dict(mask=2, lens=None), INVALID),
    (dict(D=32), UNSUPPORTED), (dict(D=96), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED),
    (dict(out=BAD), MISALIGNED), (dict(q=ctypes.c_void_p(0x10004)), MISALIGNED),
    (dict(B=0), OK), (dict(H=0), OK), (dict(Lq=0), OK),
    (dict(B=70000), INVALID),
])
def test_mha_fwd_host_validation(L, kw, want):
    assert fwd(L, **kw) == want


def pre(L, x=A, g=A2, b=A3, eps=1e-5, k=A, v=A2, lens=None, out=OUT, B=2, H=2, Lq=8, Lk=8,
        D=64, scale=0.125, dtype=1):
    return L.prenorm_cross_attn_fwd(x, g, b, eps, k, v, lens, out, B, H, Lq, Lk, D, scale,
                                    dtype, None)


@pytest.mark.parametrize("kw,want", [
    (dict(x=None), INVALID), (dict(g=None), INVALID), (dict(b=None), INVALID),
    (dict(eps=-1.0), INVALID), (dict(eps=float("inf")), INVALID),
    (dict(dtype=0), UNSUPPORTED), (dict(D=80), UNSUPPORTED),
    (dict(g=ctypes.c_void_p(0x20004)), MISALIGNED), (dict(Lq=0), OK), (dict(B=0), OK),
])
def test_prenorm_host_validation(L, kw, want):
    assert pre(L, **kw) == want


LSE = ctypes.c_void_p(0x50000)
G = ctypes.c_void_p(0x60000)
DQ, DK, DV = ctypes.c_void_p(0x70000), ctypes.c_void_p(0x80000), ctypes.c_void_p(0x90000)


def fwd_lse(L, q=A, k=A2, v=A3, mask=0, lens=None, out=OUT, lse=LSE, B=2, H=2, Lq=8, Lk=8,
            D=64, scale=0.125, dtype=0):
    return L.mha_fwd_lse(q, k, v, mask, lens, out, lse, B, H, Lq, Lk, D, scale, dtype, None)


@pytest.mark.parametrize("kw,want", [
    (dict(lse=None), INVALID), (dict(q=None), INVALID), (dict(mask=8), INVALID),
    (dict(dtype=5), UNSUPPORTED), (dict(D=80), UNSUPPORTED),
    (dict(lse=ctypes.c_void_p(0x50004)), MISALIGNED), (dict(Lq=0), OK), (dict(B=0), OK),
])
def test_fwd_lse_host_validation(L, kw, want):
    assert fwd_lse(L, **kw) == want


WS = ctypes.c_void_p(0xA0000)


def bwd(L, q=A, k=A2, v=A3, o=OUT, g=G, lse=LSE, mask=0, lens=None, dq=DQ, dk=DK, dv=DV,
        B=2, H=2, Lq=8, Lk=8, D=64, scale=0.125, dtype=0, ws=WS, ws_bytes=1 << 20):
    return L.mha_bwd(q, k, v, o, g, lse, mask, lens, dq, dk, dv, B, H, Lq, Lk, D, scale, dtype,
                     ws, ws_bytes, None)


@pytest.mark.parametrize("kw,want", [
    (dict(g=None), INVALID), (dict(lse=None), INVALID), (dict(dq=None), INVALID),
    (dict(dk=None), INVALID), (dict(o=None), INVALID), (dict(mask=2, lens=None), INVALID),
    (dict(scale=0.0), INVALID), (dict(Lq=-1), INVALID),
    (dict(dtype=2), UNSUPPORTED), (dict(D=32), UNSUPPORTED),
    (dict(dv=ctypes.c_void_p(0x90008)), MISALIGNED), (dict(g=ctypes.c_void_p(0x60004)), MISALIGNED),
    (dict(B=0), OK), (dict(H=0), OK), (dict(Lq=0, Lk=0), OK),
    # Lq == 0 still writes dk, dv: the query-side pointers are not needed
    (dict(Lq=0, q=None, o=None, g=None, lse=None, dq=None, dk=None), INVALID),
    # the caller's workspace: present, large enough, aligned
    (dict(ws=None), INVALID), (dict(ws_bytes=2 * 2 * 8 * 4 - 1), INVALID),
    (dict(ws=ctypes.c_void_p(0xA0008)), MISALIGNED),
])
def test_bwd_host_validation(L, kw, want):
    assert bwd(L, **kw) == want


def fwd_host(L, q=A, k=A2, v=A3, mask=0, lens=None, out=OUT, B=2, H=2, Lq=8, Lk=8, D=64,
             scale=0.125, dtype=1, ws=WS, ws_bytes=1 << 30):
    return L.mha_fwd_host(q, k, v, mask, lens, out, B, H, Lq, Lk, D, scale, dtype, ws, ws_bytes,
                          None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), INVALID), (dict(out=None), INVALID), (dict(v=None), INVALID),
    (dict(mask=2, lens=None), INVALID), (dict(mask=4), INVALID), (dict(scale=0.0), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(dtype=3), UNSUPPORTED),
    (dict(ws=None), INVALID), (dict(ws_bytes=1024), INVALID),
    (dict(ws=ctypes.c_void_p(0xA0008)), MISALIGNED),
    (dict(B=0), OK), (dict(Lq=0), OK),
])
def test_fwd_host_copies_validation(L, kw, want):
    """mha_fwd_host (host tensors, pipelined copies) rejects bad arguments
    before it creates a stream or copies anything."""
    assert fwd_host(L, **kw) == want


def test_fwd_host_workspace_size(L):
    """Two slots of one piece (q, k, v, out of the largest divisor of H whose
    piece holds at most 64 MB), each part rounded up to 256 bytes, plus the
    lengths."""
    r = lambda x: (x + 255) // 256 * 256
    # long causal workload shape: 8 MB per head, pieces of 8 heads
    q = 8 * 8192 * 128 * 2
    assert L.mha_fwd_host_workspace_size(2, 32, 8192, 8192, 128, 1) == 2 * 4 * q + r(8)
    # H = 5 (prime), small heads: one piece per batch
    q, k = 5 * 100 * 64 * 4, 5 * 300 * 64 * 4
    assert L.mha_fwd_host_workspace_size(3, 5, 100, 300, 64, 0) == 2 * (2 * r(q) + 2 * r(k)) + r(12)
    # one head larger than a piece: pieces of one head
    q = 65536 * 128 * 4
    assert L.mha_fwd_host_workspace_size(1, 3, 65536, 65536, 128, 0) == 2 * 4 * q + r(4)
    assert L.mha_fwd_host_workspace_size(0, 5, 70, 70, 64, 0) == 0
    assert L.mha_fwd_host_workspace_size(3, 5, 70, 70, 96, 0) == 0
    assert L.mha_fwd_host_workspace_size(3, 5, 70, 70, 64, 4) == 0


def test_bwd_workspace_size(L):
    rows = 3 * 5 * 70
    delta = (4 * rows + 255) // 256 * 256
    assert L.mha_bwd_workspace_size(3, 5, 70, 64, 0) == delta       # fp32
    assert L.mha_bwd_workspace_size(3, 5, 70, 128, 1) == delta      # bf16 on the tensor cores
    assert L.mha_bwd_workspace_size(0, 5, 70, 64, 0) == 0
    assert L.mha_bwd_workspace_size(3, 5, 70, 96, 0) == 0
    L.mha_set_bwd_kernel(1)    # thread-local: this thread only
    try:
        assert L.mha_bwd_workspace_size(3, 5, 70, 128, 1) == delta + 4 * rows * 128
    finally:
        L.mha_set_bwd_kernel(0)
    assert L.mha_bwd_workspace_size(3, 5, 70, 128, 1) == delta


def test_hooks_are_thread_local(L):
    import threading
    rows = 2 * 2 * 8
    delta = (4 * rows + 255) // 256 * 256
    seen = []
    L.mha_set_bwd_kernel(1)
    try:
        t = threading.Thread(target=lambda: seen.append(L.mha_bwd_workspace_size(2, 2, 8, 64, 1)))
        t.start()
        t.join()
        assert seen == [delta]    # the other thread still has the automatic choice
        assert L.mha_bwd_workspace_size(2, 2, 8, 64, 1) == delta + 4 * rows * 64
    finally:
        L.mha_set_bwd_kernel(0)


def test_status_hook_rejects_unknown_unit(L):
    assert L.mha_test_set_device_status(4, 1) == INVALID
    assert L.mha_test_set_device_status(-1, 1) == INVALID


def test_selftest_host_validation(L):
    assert L.mha_selftest_umma(3, 64, A, A2, OUT, None) == INVALID
    assert L.mha_selftest_umma(0, 96, A, A2, OUT, None) == UNSUPPORTED
    assert L.mha_selftest_umma(0, 64, None, A2, OUT, None) == INVALID
    assert L.mha_selftest_umma(0, 64, A, A2, BAD, None) == MISALIGNED


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import masked_head_attention_gb300 as mha
    monkeypatch.setattr(mha, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mha, "_lib", None)
    with pytest.raises(mha.MhaError):
        mha.lib()
