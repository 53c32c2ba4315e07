"""Programmatic dependent launch: a call that reads the previous call's output
(read after write) or overwrites a buffer the previous call is still reading
(write after read) sees the same data as with ordinary launches.  Every kernel
waits on the device for the previous grid before it touches global memory;
these chains would show a missing wait as a changed output (GPU)."""
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, dev, randn


@pytest.fixture
def pdl_off_then_on():
    yield
    mha.set_pdl(1)


def _chain(dtype, D, Lq, Lk, mask):
    """Three calls on one stream: out1 from (q, k, v); out2 from (out1, k, v),
    reading out1 right after it is written; then a third call writes into k,
    which the second call reads.  Returns out1, out2 and the third output."""
    q = dev(randn((2, 4, Lq, D), 301, 1.0, dtype))
    k = dev(randn((2, 4, Lk, D), 302, 1.0, dtype))
    v = dev(randn((2, 4, Lk, D), 303, 1.0, dtype))
    q3 = dev(randn((2, 4, Lq, D), 304, 1.0, dtype))
    k0 = k.clone()
    torch.cuda.synchronize()
    out1 = mha.mha_fwd(q, k, v, mask)
    out2 = mha.mha_fwd(out1, k, v, mask)
    out3 = mha.mha_fwd(q3, q3, q3, mask, out=k) if Lq == Lk else None
    torch.cuda.synchronize()
    return q.cpu(), k0.cpu(), v.cpu(), out1.cpu(), out2.cpu(), None if out3 is None else out3.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,D,Lq,Lk,mask", [
    (torch.bfloat16, 128, 2048, 2048, 1),   # tensor-core forward
    (torch.bfloat16, 128, 4, 4096, 0),      # decode kernel
    (torch.float32, 64, 512, 512, 1),       # 3xTF32 kernel
    (torch.float32, 128, 256, 256, 0),      # CUDA-core fp32 kernel
], ids=["bf16", "decode", "tf32x3", "f32"])
def test_dependent_calls_match_ordinary_launches(dtype, D, Lq, Lk, mask, pdl_off_then_on):
    mha.set_pdl(0)
    ref = _chain(dtype, D, Lq, Lk, mask)
    mha.set_pdl(1)
    got = _chain(dtype, D, Lq, Lk, mask)
    for a, b in zip(ref[3:], got[3:]):
        if a is not None:
            assert torch.equal(a, b)
    assert mha.device_status() == 0
    if dtype == torch.bfloat16:
        # The second call saw the first call's output, and nothing else.
        q, k, v, out1, out2, _ = got
        want2 = oracle.mha_fwd(out1.float().numpy(), k.float().numpy(), v.float().numpy(), mask,
                               None)
        check_bf16(as_np(out2), want2, "second call of the chain")


@pytest.mark.gpu
def test_backward_after_forward_matches_ordinary_launches(pdl_off_then_on):
    """mha_fwd_lse, then mha_bwd reading its output and row log-sum-exp (the
    row pass and the tensor-core backward, two dependent kernels)."""
    B, H, L, D = 1, 4, 512, 128

    def run():
        q = dev(randn((B, H, L, D), 311, 1.0, torch.bfloat16))
        k = dev(randn((B, H, L, D), 312, 1.0, torch.bfloat16))
        v = dev(randn((B, H, L, D), 313, 1.0, torch.bfloat16))
        g = dev(randn((B, H, L, D), 314, 1.0, torch.bfloat16))
        torch.cuda.synchronize()
        o, lse = mha.mha_fwd_lse(q, k, v, 1)
        dq, dk, dv = mha.mha_bwd(q, k, v, o, g, lse, 1)
        torch.cuda.synchronize()
        return [t.cpu() for t in (o, lse, dq, dk, dv)]

    mha.set_pdl(0)
    ref = run()
    mha.set_pdl(1)
    got = run()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_noalloc_prenorm_matches_ordinary_launches(pdl_off_then_on):
    """The no-allocation Pre-LN entry point runs a statistics pass and then the
    attention kernel that reads its output."""
    B, H, L, D = 2, 4, 512, 64
    N = H * D

    def run():
        x = dev(randn((B, L, N), 321, 1.0, torch.bfloat16))
        gamma = dev(randn((N,), 322, 0.1, torch.float32) + 1.0)
        beta = dev(randn((N,), 323, 0.1, torch.float32))
        k = dev(randn((B, H, L, D), 324, 1.0, torch.bfloat16))
        v = dev(randn((B, H, L, D), 325, 1.0, torch.bfloat16))
        torch.cuda.synchronize()
        out = mha.prenorm_cross_attn_fwd_noalloc(x, gamma, beta, 1e-5, k, v, None)
        torch.cuda.synchronize()
        return out.cpu()

    mha.set_pdl(0)
    ref = run()
    mha.set_pdl(1)
    assert torch.equal(ref, run())
    assert mha.device_status() == 0
