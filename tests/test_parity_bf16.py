"""bf16 tensor-core path (TMA + tcgen05 + TMEM) against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from masked_head_attention_gb300 import synthetic
from parity_util import as_np, check_bf16, dev, lens_tensor, randn, sample_rows

CASES = [
    (1, 1, 1, 1, 64, 0, None),
    (1, 1, 1, 1, 128, 1, None),
    (2, 3, 7, 7, 64, 1, None),
    (1, 2, 128, 128, 128, 1, None),
    (2, 2, 129, 129, 64, 1, None),
    (1, 2, 300, 300, 128, 1, None),
    (2, 2, 65, 300, 64, 0, None),
    (2, 2, 200, 77, 128, 1, None),
    (2, 1, 77, 200, 64, 1, None),
    (4, 2, 260, 260, 64, 2, [0, 1, 260, 130]),
    (3, 2, 257, 257, 128, 2, [400, -3, 128]),
    (4, 2, 390, 390, 128, 3, [1, 127, 128, 390]),
    (2, 4, 512, 512, 64, 3, [300, 512]),
]


def _run(B, H, Lq, Lk, D, mask, lens, std=1.0, seed=0):
    q = randn((B, H, Lq, D), seed, std, torch.bfloat16)
    k = randn((B, H, Lk, D), seed + 1, std, torch.bfloat16)
    v = randn((B, H, Lk, D), seed + 2, 1.0, torch.bfloat16)
    out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), mask, lens)
    return as_np(out), want


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%dm%d" % c[:6])
def test_bf16_small(case):
    got, want = _run(*case)
    check_bf16(got, want, str(case))
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_bf16_peaky_logits_stress_max_shift():
    # Logit std 2.5 (span about [-10, 10]) as in the long causal workload.
    got, want = _run(1, 4, 600, 600, 128, 1, None, std=2.5 ** 0.5, seed=3)
    check_bf16(got, want, "peaky")


@pytest.mark.gpu
def test_bf16_large_logits_finite():
    # Logits around +-100: exp would overflow fp32 without the max shift.
    got, want = _run(1, 2, 256, 256, 64, 1, None, std=4.0, seed=4)
    assert np.all(np.isfinite(got))
    check_bf16(got, want, "large logits")


@pytest.mark.gpu
def test_bf16_c3_full_workload():
    w = synthetic.WORKLOADS["c3_causal_bf16"]
    x = synthetic.make(w, seed=0)
    out = mha.mha_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, None, scale=w.scale)
    torch.cuda.synchronize()
    want = oracle.mha_fwd(x["q"].float().numpy(), x["k"].float().numpy(), x["v"].float().numpy(),
                          w.mask, None, w.scale)
    r = check_bf16(as_np(out), want, w.name)
    print(w.name, r)


@pytest.mark.gpu
def test_bf16_c5_sampled_rows():
    w = synthetic.WORKLOADS["c5_long_causal_bf16"]
    x = synthetic.make(w, seed=0)
    out = mha.mha_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, None, scale=w.scale)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.H, w.Lq, 160, seed=5)
    want = oracle.mha_rows(x["q"].float().numpy(), x["k"].float().numpy(),
                           x["v"].float().numpy(), rows, w.mask, None, w.scale)
    o = out.float().cpu()
    got = np.stack([o[b, h, i].numpy() for b, h, i in rows]).astype(np.float64)
    r = check_bf16(got, want, w.name)
    print(w.name, r)


@pytest.mark.gpu
def test_bf16_c5_full_workload():
    """Every element of the long causal workload (B2 H32 L8192 D128, 67 M
    outputs) against the fp64 oracle, run on all host cores."""
    w = synthetic.WORKLOADS["c5_long_causal_bf16"]
    x = synthetic.make(w, seed=0)
    out = mha.mha_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, None, scale=w.scale)
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    got = as_np(out)
    del out
    want = oracle.mha_fwd(x["q"].float().numpy(), x["k"].float().numpy(), x["v"].float().numpy(),
                          w.mask, None, w.scale)
    r = check_bf16(got, want, w.name)
    print(w.name, r)


@pytest.mark.gpu
def test_bf16_masked_keys_contribute_exactly_zero():
    B, H, L, D = 2, 2, 300, 128
    q = randn((B, H, L, D), 5, dtype=torch.bfloat16)
    k = randn((B, H, L, D), 6, dtype=torch.bfloat16)
    v = randn((B, H, L, D), 7, dtype=torch.bfloat16)
    lens = torch.tensor([140, 300], dtype=torch.int32)
    a = mha.mha_fwd(dev(q), dev(k), dev(v), 3, dev(lens)).cpu()
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 140:] = randn((H, L - 140, D), 8, 30.0, torch.bfloat16)
    v2[0, :, 140:] = randn((H, L - 140, D), 9, 30.0, torch.bfloat16)
    k2[1, :, 11] += 5.0
    b = mha.mha_fwd(dev(q), dev(k2), dev(v2), 3, dev(lens)).cpu()
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1, :, :11], b[1, :, :11])


@pytest.mark.gpu
def test_bf16_zero_keys_and_persistent_grid():
    q = randn((2, 2, 9, 64), 1, dtype=torch.bfloat16).cuda()
    kv = torch.empty((2, 2, 0, 64), device="cuda", dtype=torch.bfloat16)
    out = mha.mha_fwd(q, kv, kv, 0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.float()).item() == 0
    # The same problem on a capped (persistent) grid matches the default grid.
    x = [randn((2, 3, 700, 128), s, dtype=torch.bfloat16).cuda() for s in (11, 12, 13)]
    a = mha.mha_fwd(*x, 1)
    try:
        mha.set_bf16_grid(5)
        b = mha.mha_fwd(*x, 1)
    finally:
        mha.set_bf16_grid(0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_repeat_runs_bit_identical(D):
    # P shares TMEM columns with S when D = 128; any ordering hazard between
    # the P.V product and the next QK^T would show up as run-to-run noise.
    x = [randn((2, 16, 1536, D), s, 1.0, torch.bfloat16).cuda() for s in (31, 32, 33)]
    ref = mha.mha_fwd(*x, 1)
    for _ in range(25):
        out = mha.mha_fwd(*x, 1)
        assert torch.equal(out, ref)
    torch.cuda.synchronize()
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ctas", [1, 3])
def test_bf16_many_items_per_cta_mixed_work(D, ctas):
    # Few CTAs walk many items: runs of items with no key tile (length 0),
    # query tiles past Lq (no work for the second tile), and more key tiles
    # than ring stages.  Exercises every hand-off between the roles; repeated
    # because a hand-off race would show up only now and then.
    B, H, L = 5, 2, 300
    q = randn((B, H, L, D), 41, 1.0, torch.bfloat16)
    k = randn((B, H, L, D), 42, 1.0, torch.bfloat16)
    v = randn((B, H, L, D), 43, 1.0, torch.bfloat16)
    lens = [0, 0, 300, 1, 129]
    lt = dev(lens_tensor(lens))
    dq, dk, dv = dev(q), dev(k), dev(v)
    try:
        mha.set_bf16_grid(0)
        ref = mha.mha_fwd(dq, dk, dv, 3, lt)
        mha.set_bf16_grid(ctas)
        for _ in range(10):
            out = mha.mha_fwd(dq, dk, dv, 3, lt)
            torch.cuda.synchronize()
            assert mha.device_status() == 0
            assert torch.equal(out, ref)
    finally:
        mha.set_bf16_grid(0)
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 3, lens)
    check_bf16(as_np(out), want, "many items D=%d ctas=%d" % (D, ctas))


@pytest.mark.gpu
def test_single_visible_key_returns_its_v_row():
    """A row with exactly one visible key has softmax weight 1 on it, so its
    output is that key's V row, bit for bit in bf16 -- whatever the sign of
    the logit (the row maximum is that logit itself)."""
    B, H, Lq, Lk, D = 2, 3, 300, 129, 64
    q = randn((B, H, Lq, D), 131, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 132, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 133, 1.0, torch.bfloat16)
    lens = torch.tensor([1, 129], dtype=torch.int32)
    for mask in (2, 3):
        out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lens)).cpu()
        assert torch.equal(out[0], v[0, :, 0:1, :].expand(H, Lq, D)), "mask %d" % mask
        if mask & 1:   # causal: row 0 of every batch sees key 0 only
            assert torch.equal(out[1, :, 0], v[1, :, 0])
    assert mha.device_status() == 0
