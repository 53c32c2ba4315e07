"""mha_fwd_host: host tensors in, host tensor out, the copies of successive
pieces overlapped with the kernels (GPU).  Each piece is one mha_fwd call on
the piece's heads, so outside the decode kernel (whose key split depends on
the number of problems in a launch) the result is bit-identical to mha_fwd on
the whole device tensors."""
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, dev, lens_tensor, randn


def _inputs(B, H, Lq, Lk, D, dtype, seed, pinned=True):
    q = randn((B, H, Lq, D), seed, 1.0, dtype)
    k = randn((B, H, Lk, D), seed + 1, 1.0, dtype)
    v = randn((B, H, Lk, D), seed + 2, 1.0, dtype)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    return q, k, v


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Lq,Lk,D,dtype,mask,lens", [
    (3, 6, 700, 700, 128, torch.bfloat16, 1, None),           # one piece per batch, slots reused
    (2, 16, 8192, 8192, 128, torch.bfloat16, 1, None),        # two pieces of 8 heads per batch
    (3, 5, 300, 1000, 64, torch.bfloat16, 2, [1000, 17, 0]),  # lengths, a batch with none
    (2, 4, 512, 512, 64, torch.float32, 3, [512, 300]),       # 3xTF32 kernel
    (2, 3, 200, 900, 128, torch.float32, 0, None),            # CUDA-core fp32 kernel
], ids=["bf16-causal", "bf16-2-pieces-per-batch", "bf16-lengths", "tf32x3", "f32"])
def test_fwd_host_matches_device_call(B, H, Lq, Lk, D, dtype, mask, lens):
    q, k, v = _inputs(B, H, Lq, Lk, D, dtype, 401)
    lh = lens_tensor(lens)
    got = mha.mha_fwd_host(q, k, v, mask, lh)
    torch.cuda.synchronize()
    want = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lh)).cpu()
    assert torch.equal(got, want)
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_fwd_host_pageable_memory_and_oracle():
    """Pageable host tensors work (their copies are staged by the driver); the
    result agrees with the oracle."""
    B, H, Lq, Lk, D = 2, 4, 300, 300, 64
    q, k, v = _inputs(B, H, Lq, Lk, D, torch.bfloat16, 411, pinned=False)
    out = torch.empty(q.shape, dtype=q.dtype)
    mha.mha_fwd_host(q, k, v, 1, None, out=out)
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 1, None)
    check_bf16(as_np(out), want, "pageable")
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_fwd_host_decode_rows_against_oracle():
    """A few query rows (the decode kernel) per piece."""
    B, H, Lq, Lk, D, lens = 3, 8, 4, 5000, 128, [5000, 2500, 1]
    q, k, v = _inputs(B, H, Lq, Lk, D, torch.bfloat16, 421)
    out = mha.mha_fwd_host(q, k, v, 2, lens_tensor(lens))
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 2, lens)
    check_bf16(as_np(out), want, "decode rows")
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_fwd_host_workspace_reused_by_consecutive_calls():
    """Two calls on one stream with one workspace: the second call's copies
    into the workspace wait for the first call's copies out of it."""
    B, H, Lq, Lk, D = 4, 8, 1024, 1024, 128
    dt = mha.BF16
    ws = torch.empty((mha.mha_fwd_host_workspace_size(B, H, Lq, Lk, D, dt),), dtype=torch.uint8,
                     device="cuda")
    a = _inputs(B, H, Lq, Lk, D, torch.bfloat16, 431)
    b = _inputs(B, H, Lq, Lk, D, torch.bfloat16, 441)
    out_a = mha.mha_fwd_host(*a, 1, None, workspace=ws)
    out_b = mha.mha_fwd_host(*b, 1, None, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_a, mha.mha_fwd(dev(a[0]), dev(a[1]), dev(a[2]), 1).cpu())
    assert torch.equal(out_b, mha.mha_fwd(dev(b[0]), dev(b[1]), dev(b[2]), 1).cpu())
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_fwd_host_no_keys_and_single_head():
    """Lk = 0 gives zeros (k and v may be empty); one batch of one head is a
    single piece."""
    q = randn((2, 3, 50, 64), 451, 1.0, torch.bfloat16).pin_memory()
    e = torch.empty((2, 3, 0, 64), dtype=torch.bfloat16)
    out = mha.mha_fwd_host(q, e, e, 0, None)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(q))
    q, k, v = _inputs(1, 1, 130, 257, 128, torch.float32, 461)
    got = mha.mha_fwd_host(q, k, v, 1, None)
    torch.cuda.synchronize()
    assert torch.equal(got, mha.mha_fwd(dev(q), dev(k), dev(v), 1).cpu())
    assert mha.device_status() == 0
