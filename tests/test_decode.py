"""Decode path (bf16, at most 8 query rows, keys split over a thread-block
cluster) against the fp64 oracle, and the same calls on the tensor-core
kernel (GPU)."""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, dev, lens_tensor, randn

# (B, H, Lq, Lk, D, mask, lengths): 1..8 rows; keys around the 32-key blocks
# and the split chunks; lengths 0, 1, mid, Lk and beyond (clamped); B*H from
# 1 (8-way split) to 512 (no split).
CASES = [
    (1, 1, 1, 1, 128, 0, None),
    (1, 1, 1, 33, 64, 0, None),
    (1, 2, 1, 4097, 128, 2, [3000]),
    (2, 3, 2, 1000, 64, 2, [0, 999]),
    (1, 4, 3, 300, 128, 1, None),
    (2, 2, 5, 2048, 128, 3, [1, 2048]),
    (3, 2, 8, 777, 64, 2, [777, 5000, 31]),
    (4, 8, 4, 8192, 128, 2, [8192, 4096, 1, 6000]),
    (16, 32, 1, 512, 64, 0, None),
]


@pytest.fixture
def decode_mode(request):
    mha.set_bf16_decode(request.param)
    yield request.param
    mha.set_bf16_decode(0)


@pytest.mark.gpu
@pytest.mark.parametrize("decode_mode", [0, 1], indirect=True, ids=["decode", "tensor"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%dm%d" % c[:6])
def test_decode_parity(case, decode_mode):
    B, H, Lq, Lk, D, mask, lens = case
    q = randn((B, H, Lq, D), 61, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 62, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 63, 1.0, torch.bfloat16)
    out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), mask, lens)
    check_bf16(as_np(out), want, str(case))
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_decode_masked_keys_contribute_exactly_zero():
    """Keys past a batch's length (and, under the causal rule, past the row)
    never matter: changing them leaves the output bit-identical."""
    B, H, Lq, Lk, D = 2, 4, 4, 3000, 128
    q = randn((B, H, Lq, D), 71, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 72, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 73, 1.0, torch.bfloat16)
    lens = torch.tensor([1500, 3000], dtype=torch.int32)
    a = mha.mha_fwd(dev(q), dev(k), dev(v), 2, dev(lens)).cpu()
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 1500:] = randn((H, Lk - 1500, D), 74, 30.0, torch.bfloat16)
    v2[0, :, 1500:] = randn((H, Lk - 1500, D), 75, 30.0, torch.bfloat16)
    b = mha.mha_fwd(dev(q), dev(k2), dev(v2), 2, dev(lens)).cpu()
    assert torch.equal(a, b)


@pytest.mark.gpu
def test_decode_workload_full():
    """The decode workload of the benchmark, every output against the oracle."""
    from masked_head_attention_gb300 import synthetic
    w = synthetic.WORKLOADS["c6_decode_bf16"]
    x = synthetic.make(w, seed=0)
    out = mha.mha_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, dev(x["kv_lengths"]),
                      scale=w.scale)
    torch.cuda.synchronize()
    want = oracle.mha_fwd(x["q"].float().numpy(), x["k"].float().numpy(),
                          x["v"].float().numpy(), w.mask, x["kv_lengths"].numpy(), w.scale)
    r = check_bf16(as_np(out), want, w.name)
    print(w.name, r)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_decode_forced_splits(splits):
    """Every cluster size combines its CTAs' partials correctly (keys split
    in chunks of a multiple of 32, the last chunk ragged or empty)."""
    B, H, Lq, Lk, D, mask, lens = 2, 3, 3, 2100, 128, 2, [2100, 700]
    q = randn((B, H, Lq, D), 81, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 82, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 83, 1.0, torch.bfloat16)
    mha.set_bf16_decode_splits(splits)
    try:
        out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lens_tensor(lens)))
        torch.cuda.synchronize()
    finally:
        mha.set_bf16_decode_splits(0)
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), mask, lens)
    check_bf16(as_np(out), want, "splits=%d" % splits)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Lq,Lk,D", [(40, 3, 2, 300, 128), (300, 1, 1, 64, 64)],
                         ids=["ranked-40-batches", "natural-order-300-batches"])
def test_decode_problem_order(B, H, Lq, Lk, D):
    """With per-batch lengths the problems run longest first (the kernel ranks
    up to 256 batches itself, ties by index); every (b, h) output still lands
    in its own place.  Lengths with many ties, zeros and values past Lk; 300
    batches take the unranked order."""
    rng = np.random.default_rng(91)
    lens = [int(x) for x in rng.choice([0, 1, 17, Lk // 2, Lk, Lk + 5], size=B)]
    q = randn((B, H, Lq, D), 92, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 93, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 94, 1.0, torch.bfloat16)
    out = mha.mha_fwd(dev(q), dev(k), dev(v), 2, dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 2, lens)
    check_bf16(as_np(out), want, "B=%d" % B)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [2, 8])
def test_decode_short_problems_forced_splits(splits):
    """Each problem's visible keys are split on their own; with short lengths
    the later CTAs of a cluster get no key at all and contribute nothing."""
    B, H, Lq, Lk, D, mask, lens = 3, 2, 2, 500, 64, 2, [5, 0, 33]
    q = randn((B, H, Lq, D), 95, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 96, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 97, 1.0, torch.bfloat16)
    mha.set_bf16_decode_splits(splits)
    try:
        out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lens_tensor(lens)))
        torch.cuda.synchronize()
    finally:
        mha.set_bf16_decode_splits(0)
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), mask, lens)
    check_bf16(as_np(out), want, "splits=%d" % splits)
    assert mha.device_status() == 0
