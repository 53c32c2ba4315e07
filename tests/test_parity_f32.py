"""fp32 path against the fp64 oracle, element by element (GPU): the
tensor-core kernel (3xTF32, D = 64) and both CUDA-core kernels."""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from masked_head_attention_gb300 import synthetic
from parity_util import as_np, check_f32, dev, lens_tensor, randn

# (B, H, Lq, Lk, D, mask, lengths): several tiles, ragged tails, Lq != Lk,
# lengths at 0, 1, the end, beyond the end (clamped) and negative (clamped).
CASES = [
    (1, 1, 1, 1, 64, 0, None),
    (1, 1, 1, 1, 64, 1, None),
    (2, 3, 7, 7, 64, 1, None),
    (2, 2, 130, 130, 64, 1, None),
    (1, 2, 200, 200, 128, 1, None),
    (2, 2, 65, 200, 64, 0, None),
    (3, 2, 100, 37, 64, 1, None),
    (2, 2, 37, 100, 128, 1, None),
    (4, 2, 150, 150, 64, 2, [0, 1, 150, 77]),
    (3, 1, 129, 129, 128, 2, [200, -5, 64]),
    (4, 2, 190, 190, 64, 3, [1, 63, 64, 190]),
    (2, 2, 256, 256, 128, 3, [129, 256]),
    # the short-key kernel's chunk ring: 8 chunks of 32 keys, ragged rows
    (2, 2, 300, 256, 64, 1, None),
    (1, 3, 47, 250, 64, 2, [250, 33, 0]),
    (3, 2, 128, 128, 128, 3, [128, 97, 5]),
]


def _run(B, H, Lq, Lk, D, mask, lens, seed=0):
    q = randn((B, H, Lq, D), seed)
    k = randn((B, H, Lk, D), seed + 1)
    v = randn((B, H, Lk, D), seed + 2)
    lt = lens_tensor(lens)
    out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lt))
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.numpy(), k.numpy(), v.numpy(), mask, lens)
    return as_np(out), want


@pytest.fixture
def f32_kernel(request):
    mha.set_f32_kernel(request.param)
    yield request.param
    mha.set_f32_kernel(0)


@pytest.mark.gpu
@pytest.mark.parametrize("f32_kernel", [0, 1, 2, 3], indirect=True,
                         ids=["auto", "tiled", "short", "tf32x3"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%dm%d" % c[:6])
def test_f32_small(case, f32_kernel):
    got, want = _run(*case)
    err = check_f32(got, want, str(case))
    print(case, f32_kernel, "max abs %.2e" % err)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["c1_causal_f32", "c2_padding_f32"])
def test_f32_full_workload(name):
    w = synthetic.WORKLOADS[name]
    x = synthetic.make(w, seed=0)
    out = mha.mha_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, dev(x["kv_lengths"]),
                      scale=w.scale)
    torch.cuda.synchronize()
    lens = None if x["kv_lengths"] is None else x["kv_lengths"].numpy()
    want = oracle.mha_fwd(x["q"].numpy(), x["k"].numpy(), x["v"].numpy(), w.mask, lens, w.scale)
    err = check_f32(as_np(out), want, name)
    print(name, "max abs %.2e" % err)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("f32_kernel", [1, 2, 3], indirect=True, ids=["tiled", "short", "tf32x3"])
def test_f32_masked_keys_contribute_exactly_zero(f32_kernel):
    B, H, L, D = 2, 2, 160, 64
    q, k, v = randn((B, H, L, D), 5), randn((B, H, L, D), 6), randn((B, H, L, D), 7)
    lens = torch.tensor([70, 160], dtype=torch.int32)
    a = mha.mha_fwd(dev(q), dev(k), dev(v), 3, dev(lens)).cpu()
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 70:] = randn((H, L - 70, D), 8, std=30.0)
    v2[0, :, 70:] = randn((H, L - 70, D), 9, std=30.0)
    for i in (10, 100):        # causal: keys after row i never matter for row i
        k2[1, :, i + 1:i + 2] += 5.0
    b = mha.mha_fwd(dev(q), dev(k2), dev(v2), 3, dev(lens)).cpu()
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1, :, :11], b[1, :, :11])
    assert not torch.equal(a[1, :, 11:101], b[1, :, 11:101])


@pytest.mark.gpu
@pytest.mark.parametrize("f32_kernel", [1, 2, 3], indirect=True, ids=["tiled", "short", "tf32x3"])
def test_f32_zero_keys_gives_zeros(f32_kernel):
    q = randn((2, 2, 9, 64), 1).cuda()
    kv = torch.empty((2, 2, 0, 64), device="cuda")
    out = mha.mha_fwd(q, kv, kv, 0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.gpu
def test_tf32x3_many_items_persistent():
    """More 128-row tiles than SMs, mixed lengths (0 included): every CTA
    walks several items, with and without work, through the same barriers."""
    mha.set_f32_kernel(3)
    try:
        lens = [0, 1, 64, 65, 700, 333, 128, 1000] * 4
        got, want = _run(32, 4, 700, 1000, 64, 3, lens, seed=40)
    finally:
        mha.set_f32_kernel(0)
    err = check_f32(got, want, "many items")
    print("many items max abs %.2e" % err)
    assert mha.device_status() == 0
