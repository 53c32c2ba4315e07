"""Pre-LayerNorm cross-attention kernel against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from masked_head_attention_gb300 import synthetic
from parity_util import as_np, check_bf16, check_bf16_sum, dev, lens_tensor, randn, sample_rows

CASES = [
    (1, 1, 1, 1, 64, None),
    (2, 4, 70, 90, 64, [90, 45]),
    (2, 2, 130, 300, 128, [0, 257]),
    (1, 16, 256, 200, 64, None),
    (3, 2, 257, 129, 128, [1, 129, 500]),
]


def _inputs(B, H, Lq, Lk, D, seed):
    N = H * D
    x = (randn((B, Lq, N), seed, 1.5) + 0.3).to(torch.bfloat16)
    g = 1.0 + 0.1 * randn((N,), seed + 1)
    b = 0.1 * randn((N,), seed + 2)
    k = randn((B, H, Lk, D), seed + 3, dtype=torch.bfloat16)
    v = randn((B, H, Lk, D), seed + 4, dtype=torch.bfloat16)
    return x, g, b, k, v


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%d" % c[:5])
def test_prenorm_small(case):
    B, H, Lq, Lk, D, lens = case
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 21)
    out = mha.prenorm_cross_attn_fwd(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v),
                                     dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                     k.float().numpy(), v.float().numpy(), lens)
    check_bf16(as_np(out), want, str(case))
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_prenorm_c4_sampled_rows():
    w = synthetic.WORKLOADS["c4_prenorm_bf16"]
    xs = synthetic.make(w, seed=0)
    out = mha.prenorm_cross_attn_fwd(dev(xs["x"]), dev(xs["gamma"]), dev(xs["beta"]), w.eps,
                                     dev(xs["k"]), dev(xs["v"]), dev(xs["kv_lengths"]),
                                     scale=w.scale)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.H, w.Lq, 160, seed=6)
    want = oracle.prenorm_rows(xs["x"].float().numpy(), xs["gamma"].numpy(), xs["beta"].numpy(),
                               w.eps, xs["k"].float().numpy(), xs["v"].float().numpy(), rows,
                               xs["kv_lengths"].numpy(), w.scale)
    o = out.float().cpu()
    got = np.stack([o[b, i, h * w.D:(h + 1) * w.D].numpy() for b, h, i in rows]).astype(np.float64)
    r = check_bf16(got, want, w.name)
    print(w.name, r)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ctas", [1, 2])
def test_prenorm_chunks_of_heads_share_row_statistics(D, ctas):
    """A capped grid makes the kernel group several heads of the same 256 rows
    into one chunk (the default grid runs one head per chunk at this size),
    whose row statistics are formed once (D = 64: by the CTA's prologue, with
    two CTAs a cluster pair splitting them; D = 128: by the softmax warps at
    the chunk start), and walk many chunks per CTA, with empty and ragged
    batches.  The result must not depend on the grouping."""
    B, H, Lq, Lk = 3, 4, 300, 260
    lens = [260, 0, 131]
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 31)
    args = (dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v), dev(lens_tensor(lens)))
    ref = mha.prenorm_cross_attn_fwd(*args)
    ref_r = mha.prenorm_cross_attn_residual_fwd(*args)
    try:
        mha.set_bf16_grid(ctas)
        for _ in range(5):
            out = mha.prenorm_cross_attn_fwd(*args)
            out_r = mha.prenorm_cross_attn_residual_fwd(*args)
            torch.cuda.synchronize()
            assert mha.device_status() == 0
            assert torch.equal(out, ref)
            assert torch.equal(out_r, ref_r)
    finally:
        mha.set_bf16_grid(0)
    want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                     k.float().numpy(), v.float().numpy(), lens)
    check_bf16(as_np(out), want, "chunks D=%d ctas=%d" % (D, ctas))


@pytest.mark.gpu
def test_prenorm_more_chunks_than_the_prologue_holds():
    """One CTA walking 40 chunks: the prologue forms the statistics of the
    first 32 (its shared-memory table), the softmax warps those of the rest
    at their chunk starts.  Every row against the oracle."""
    B, H, Lq, Lk, D = 1, 1, 40 * 256 - 70, 100, 64
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 35)
    args = (dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v), None)
    ref = mha.prenorm_cross_attn_fwd(*args)
    try:
        mha.set_bf16_grid(1)
        out = mha.prenorm_cross_attn_fwd(*args)
        torch.cuda.synchronize()
    finally:
        mha.set_bf16_grid(0)
    assert mha.device_status() == 0
    assert torch.equal(out, ref)
    want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                     k.float().numpy(), v.float().numpy(), None)
    check_bf16(as_np(out), want, "40 chunks on one CTA")


@pytest.mark.gpu
def test_prenorm_many_batches_keep_index_order():
    """More batches than the kernel ranks by length (128): chunks then run in
    batch order; lengths include zero and values past Lk."""
    B, H, Lq, Lk, D = 130, 2, 20, 50, 64
    lens = [(7 * i) % 61 for i in range(B)]
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 37)
    out = mha.prenorm_cross_attn_fwd(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v),
                                     dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                     k.float().numpy(), v.float().numpy(), lens)
    check_bf16(as_np(out), want, "130 batches")
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_prenorm_wide_rows_take_several_segments():
    """Rows of 16 x 128 = 2048 features: the statistics routine runs two
    segments per row and re-reads x for the second pass."""
    B, H, Lq, Lk, D = 1, 16, 130, 70, 128
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 33)
    out = mha.prenorm_cross_attn_fwd(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v), None)
    torch.cuda.synchronize()
    want = oracle.prenorm_cross_attn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                     k.float().numpy(), v.float().numpy(), None)
    check_bf16(as_np(out), want, "wide rows")
    assert mha.device_status() == 0


def _c4():
    w = synthetic.WORKLOADS["c4_prenorm_bf16"]
    return w, synthetic.make(w, seed=0)


def _c4_oracle(fn, w, xs):
    return fn(xs["x"].float().numpy(), xs["gamma"].numpy(), xs["beta"].numpy(), w.eps,
              xs["k"].float().numpy(), xs["v"].float().numpy(), xs["kv_lengths"].numpy(), w.scale)


@pytest.mark.gpu
def test_prenorm_c4_full_workload():
    """Every element of the Pre-LN workload (B32 H16 Lq2048 d_model 1024,
    67 M outputs) against the fp64 oracle."""
    w, xs = _c4()
    out = mha.prenorm_cross_attn_fwd(dev(xs["x"]), dev(xs["gamma"]), dev(xs["beta"]), w.eps,
                                     dev(xs["k"]), dev(xs["v"]), dev(xs["kv_lengths"]),
                                     scale=w.scale)
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    got = as_np(out)
    del out
    r = check_bf16(got, _c4_oracle(oracle.prenorm_cross_attn, w, xs), w.name)
    print(w.name, r)


@pytest.mark.gpu
def test_prenorm_residual_c4_full_workload():
    w, xs = _c4()
    out = mha.prenorm_cross_attn_residual_fwd(dev(xs["x"]), dev(xs["gamma"]), dev(xs["beta"]),
                                              w.eps, dev(xs["k"]), dev(xs["v"]),
                                              dev(xs["kv_lengths"]), scale=w.scale)
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    got = as_np(out)
    del out
    r = check_bf16_sum(got, _c4_oracle(oracle.prenorm_cross_attn_residual, w, xs),
                       w.name + " residual")
    print(w.name, "residual", r)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%d" % c[:5])
def test_prenorm_residual_small(case):
    B, H, Lq, Lk, D, lens = case
    x, g, b, k, v = _inputs(B, H, Lq, Lk, D, 23)
    out = mha.prenorm_cross_attn_residual_fwd(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v),
                                              dev(lens_tensor(lens)))
    torch.cuda.synchronize()
    want = oracle.prenorm_cross_attn_residual(x.float().numpy(), g.numpy(), b.numpy(), 1e-5,
                                              k.float().numpy(), v.float().numpy(), lens)
    check_bf16_sum(as_np(out), want, str(case))
    assert mha.device_status() == 0
    if lens is not None and 0 in lens:
        # A batch with no visible key returns x unchanged, bit for bit.
        z = lens.index(0)
        assert torch.equal(out[z].cpu(), x[z])


@pytest.mark.gpu
def test_prenorm_residual_c4_sampled_rows():
    w = synthetic.WORKLOADS["c4_prenorm_bf16"]
    xs = synthetic.make(w, seed=0)
    out = mha.prenorm_cross_attn_residual_fwd(dev(xs["x"]), dev(xs["gamma"]), dev(xs["beta"]),
                                              w.eps, dev(xs["k"]), dev(xs["v"]),
                                              dev(xs["kv_lengths"]), scale=w.scale)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.H, w.Lq, 160, seed=7)
    want = oracle.prenorm_residual_rows(xs["x"].float().numpy(), xs["gamma"].numpy(),
                                        xs["beta"].numpy(), w.eps, xs["k"].float().numpy(),
                                        xs["v"].float().numpy(), rows, xs["kv_lengths"].numpy(),
                                        w.scale)
    o = out.float().cpu()
    got = np.stack([o[b, i, h * w.D:(h + 1) * w.D].numpy() for b, h, i in rows]).astype(np.float64)
    r = check_bf16_sum(got, want, w.name + " residual")
    print(w.name, "residual", r)
    assert mha.device_status() == 0
