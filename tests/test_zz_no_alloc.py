"""The no-allocation Pre-LN entry point, called through the C ABI.

Some callers cannot let a library allocate device memory (a serving runtime
that owns all GPU memory through its own pools, a latency-critical loop where
an allocation may block or fail).  prenorm_cross_attn_fwd_noalloc serves
them with a fixed device array for the row statistics; these tests check it
returns exactly (bit for bit) what prenorm_cross_attn_fwd returns, and
matches the fp64 oracle, on two calls in a row (the second with a different
shape, so stale contents of the shared array would show), and that a problem
too large for the array is refused before any launch.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, randn

MAX_ROWS = 262144
TOO_LARGE = -6


def _bind():
    L = mha.lib()
    P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = L.prenorm_cross_attn_fwd_noalloc
    fn.argtypes = [P, P, P, f, P, P, P, P, i, i, i, i, i, f, i, P]
    fn.restype = i
    return fn


def _inputs(B, H, Lq, Lk, D, seed):
    N = H * D
    x = (randn((B, Lq, N), seed, 1.3) + 0.2).to(torch.bfloat16).cuda()
    g = (1.0 + 0.1 * randn((N,), seed + 1)).cuda()
    b = (0.1 * randn((N,), seed + 2)).cuda()
    k = randn((B, H, Lk, D), seed + 3, dtype=torch.bfloat16).cuda()
    v = randn((B, H, Lk, D), seed + 4, dtype=torch.bfloat16).cuda()
    lens = torch.randint(1, Lk + 1, (B,), generator=torch.Generator().manual_seed(seed),
                         dtype=torch.int32).cuda()
    return x, g, b, k, v, lens


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_two_calls():
    fn = _bind()
    stream = torch.cuda.current_stream()
    for call, (B, H, Lq, Lk, D) in enumerate([(2, 4, 300, 260, 64), (3, 2, 200, 333, 128)]):
        x, g, b, k, v, lens = _inputs(B, H, Lq, Lk, D, 70 + call)
        scale = 1.0 / D ** 0.5
        ref = mha.prenorm_cross_attn_fwd(x, g, b, 1e-5, k, v, lens, scale=scale)
        out = torch.full_like(ref, float("nan"))
        rc = fn(_p(x), _p(g), _p(b), 1e-5, _p(k), _p(v), _p(lens), _p(out), B, H, Lq, Lk, D,
                scale, 1, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, mha.mha_strerror(rc)
        torch.cuda.synchronize()
        # Same statistics and the same attention kernel: identical bits.
        assert torch.equal(out, ref), "no-alloc call %d differs from the allocating call" % call
        want = oracle.prenorm_cross_attn(x.float().cpu().numpy(), g.cpu().numpy(),
                                         b.cpu().numpy(), 1e-5, k.float().cpu().numpy(),
                                         v.float().cpu().numpy(), lens.cpu().numpy(), scale)
        check_bf16(as_np(out), want, "no-alloc call %d" % call)
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_noalloc_matches_on_a_capped_grid():
    """On one CTA the kernel groups all four heads of a row block into one
    chunk; the no-allocation call (statistics copied from the fixed array)
    still returns the same bits as prenorm_cross_attn_fwd (statistics formed
    inside the attention kernel)."""
    fn = _bind()
    stream = torch.cuda.current_stream()
    B, H, Lq, Lk, D = 3, 4, 300, 260, 64
    x, g, b, k, v, lens = _inputs(B, H, Lq, Lk, D, 90)
    try:
        mha.set_bf16_grid(1)
        ref = mha.prenorm_cross_attn_fwd(x, g, b, 1e-5, k, v, lens, scale=0.125)
        out = torch.full_like(ref, float("nan"))
        rc = fn(_p(x), _p(g), _p(b), 1e-5, _p(k), _p(v), _p(lens), _p(out), B, H, Lq, Lk, D,
                0.125, 1, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, mha.mha_strerror(rc)
        torch.cuda.synchronize()
    finally:
        mha.set_bf16_grid(0)
    assert torch.equal(out, ref)
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_noalloc_refuses_problems_beyond_its_scratch():
    fn = _bind()
    fake = ctypes.c_void_p(0x10000)
    B, Lq = 2, MAX_ROWS // 2 + 1
    rc = fn(fake, fake, fake, 1e-5, fake, fake, None, fake, B, 1, Lq, 8, 64, 0.125, 1, None)
    assert rc == TOO_LARGE
    assert "scratch" in mha.mha_strerror(rc)
