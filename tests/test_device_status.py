"""Failure detection without a GPU fault: every bounded device-side wait of
the tensor-core kernels (bf16 forward and its Pre-LN variant, fp32 3xTF32
forward, bf16 backward)
reports its expiry through mha_device_status, the word is cleared on
request, and the next call with the normal limit is correct again.

A test hook shortens the wait limit to 1 ns, so the first wait that is not
satisfied at once expires: the kernel sets its status bit, lets the copies
and products already in flight finish (those drains keep the normal limit),
releases its tensor memory and returns.  Nothing traps, faults or hangs.
"""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, check_f32, dev, randn

UNITS = {0: "bf16 forward", 1: "fp32 tensor-core forward", 2: "bf16 tensor-core backward",
         3: "bf16 decode"}
FLAG_SUM, FLAG_NONFINITE = 1 << 16, 1 << 17


@pytest.mark.gpu
@pytest.mark.parametrize("unit", sorted(UNITS), ids=lambda u: UNITS[u])
def test_status_word_of_every_unit_is_reported_and_cleared(unit):
    assert mha.device_status(clear=True) == 0
    mha.test_set_device_status(unit, 1 << 6)
    try:
        assert mha.device_status() == 1 << 6
        assert mha.device_status(clear=True) == 1 << 6
        assert mha.device_status() == 0
    finally:
        mha.device_status(clear=True)


def _bf16_fwd():
    q, k, v = (randn((2, 2, 300, 128), s, 1.0, torch.bfloat16) for s in (61, 62, 63))

    def run():
        return mha.mha_fwd(dev(q), dev(k), dev(v), mha.MASK_CAUSAL)

    def check(out):
        want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), 1)
        check_bf16(as_np(out), want, "bf16 forward after expiry")
    return run, check


def _prenorm_fwd():
    """Pre-LN forward (row statistics formed inside the kernel first)."""
    B, H, Lq, Lk, D = 2, 4, 300, 200, 64
    x = randn((B, Lq, H * D), 71, 1.0, torch.bfloat16)
    k, v = (randn((B, H, Lk, D), s, 1.0, torch.bfloat16) for s in (72, 73))
    g = torch.linspace(0.5, 1.5, H * D, dtype=torch.float32)
    b = torch.linspace(-0.2, 0.2, H * D, dtype=torch.float32)
    lens = torch.tensor([200, 77], dtype=torch.int32)

    def run():
        return mha.prenorm_cross_attn_fwd(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v), dev(lens))

    def check(out):
        want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                         k.float().numpy(), v.float().numpy(), lens.numpy())
        check_bf16(as_np(out), want, "Pre-LN forward after expiry")
    return run, check


def _tf32_fwd():
    q, k, v = (randn((2, 2, 300, 64), s) for s in (64, 65, 66))
    lens = torch.tensor([300, 123], dtype=torch.int32)

    def run():
        return mha.mha_fwd(dev(q), dev(k), dev(v), 3, dev(lens))

    def check(out):
        want = oracle.mha_fwd(q.numpy(), k.numpy(), v.numpy(), 3, lens.numpy())
        check_f32(as_np(out), want, "3xTF32 forward after expiry")
    return run, check


def _bf16_bwd():
    q, k, v, g = (randn((1, 2, 200, 128), s, 1.0, torch.bfloat16) for s in (67, 68, 69, 70))
    o, lse = mha.mha_fwd_lse(dev(q), dev(k), dev(v), mha.MASK_CAUSAL)
    torch.cuda.synchronize()
    assert mha.device_status() == 0

    def run():
        return torch.cat([t.flatten() for t in mha.mha_bwd(dev(q), dev(k), dev(v), o, dev(g), lse,
                                                             mha.MASK_CAUSAL)])

    def check(out):
        want = oracle.mha_bwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                              g.float().numpy(), 1)
        w = np.concatenate([x.ravel() for x in want])
        s = max(1.0, np.abs(w).max())
        err = np.abs(as_np(out) - w)
        assert err.max() <= 2e-2 * s and err.mean() <= 1e-3 * s
    return run, check


CASES = {"bf16 forward": (_bf16_fwd, 0), "Pre-LN forward": (_prenorm_fwd, 0),
         "3xTF32 forward": (_tf32_fwd, 1), "bf16 backward": (_bf16_bwd, 2)}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_expired_wait_sets_status_and_the_next_call_recovers(name):
    make, unit = CASES[name]
    assert mha.device_status(clear=True) == 0
    run, check = make()
    ref = run()
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    mha.test_set_wait_limit_ns(1)
    try:
        run()                       # returns MHA_OK: the launch itself succeeds
        torch.cuda.synchronize()
    finally:
        mha.test_set_wait_limit_ns(0)
    bits = mha.device_status()
    assert bits != 0, "no wait expired under a 1 ns limit"
    # While the word is set, the unit's kernels return at once: the call still
    # succeeds on the host, and the status stays visible to the caller.
    run()
    torch.cuda.synchronize()
    assert mha.device_status(clear=True) == bits
    assert mha.device_status() == 0
    out = run()
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    assert torch.equal(out, ref)    # these kernels are deterministic
    check(out)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["bf16", "tf32x3", "decode"])
def test_non_finite_input_raises_numeric_flags_without_stopping_later_calls(kind):
    """The pages call a softmax sum other than one an error: a NaN in one query
    row makes that row's sum and output non-finite, which the kernels report
    as status bits 16 and 17; those bits do not stop later launches, and the
    other rows are unaffected."""
    dtype = torch.float32 if kind == "tf32x3" else torch.bfloat16
    Lq = 1 if kind == "decode" else 200
    D = 64 if kind == "tf32x3" else 128
    q = randn((2, 2, Lq, D), 91, 1.0, dtype)
    k = randn((2, 2, 300, D), 92, 1.0, dtype)
    v = randn((2, 2, 300, D), 93, 1.0, dtype)
    assert mha.device_status(clear=True) == 0
    clean = mha.mha_fwd(dev(q), dev(k), dev(v), 0)
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    bad = q.clone()
    bad[1, 0, Lq - 1, 3] = float("nan")
    out = mha.mha_fwd(dev(bad), dev(k), dev(v), 0)
    torch.cuda.synchronize()
    bits = mha.device_status(clear=True)
    assert bits & FLAG_NONFINITE, hex(bits)
    assert bits & FLAG_SUM, hex(bits)
    assert bits & 0xFFFF == 0, hex(bits)          # no wait expired
    o = out.cpu()
    assert not torch.isfinite(o[1, 0, Lq - 1]).any()
    keep = torch.ones(o.shape[:3], dtype=torch.bool)
    keep[1, 0, Lq - 1] = False
    assert torch.equal(o[keep], clean.cpu()[keep])   # every other row as before
    again = mha.mha_fwd(dev(q), dev(k), dev(v), 0)
    torch.cuda.synchronize()
    assert torch.equal(again, clean)
    assert mha.device_status() == 0
