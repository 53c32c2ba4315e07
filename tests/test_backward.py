"""Backward pass (fp32 on CUDA cores) and the forward's row log-sum-exp
against the fp64 oracle (GPU).

Tolerance: the forward's fp32 bound (1e-4 max abs) scaled by the size of the
gradient, max |gpu - oracle| <= 1e-4 * max(1, max |oracle|) per tensor.  Each
gradient element is an fp32 sum over up to Lq (dk, dv) or Lk (dq) products
whose terms are of the order of the largest gradient, so its rounding error
grows with that scale, not with the fixed 1e-4 of an output bounded by |v|.
"""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from masked_head_attention_gb300 import synthetic
from parity_util import as_np, check_f32, dev, lens_tensor, randn

BWD_REL = 1e-4

# (B, H, Lq, Lk, D, mask, lengths): tiles of 64 with ragged tails; Lq < Lk and
# Lq > Lk under the causal rule; a batch with no visible key; a single key.
CASES = [
    (1, 1, 1, 1, 64, 0, None),
    (2, 2, 70, 90, 64, 2, [90, 45]),
    (1, 2, 130, 200, 128, 1, None),
    (2, 3, 257, 129, 64, 3, [1, 129]),
    (2, 1, 100, 300, 128, 1, None),
    (1, 2, 300, 60, 64, 1, None),
    (2, 2, 64, 64, 128, 2, [0, 64]),
    (1, 1, 200, 1, 128, 0, None),
    (2, 2, 192, 256, 64, 3, [256, 100]),
]


def check_grad(got, want, what):
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), "%s: non-finite gradient" % what
    err = np.abs(got - want).max() if got.size else 0.0
    tol = BWD_REL * max(1.0, float(np.abs(want).max()) if want.size else 1.0)
    assert err <= tol, "%s: max abs %.3g > %.3g" % (what, err, tol)
    return err


def run_case(B, H, Lq, Lk, D, mask, lens, seed, scale=None):
    q = randn((B, H, Lq, D), seed, 1.0)
    k = randn((B, H, Lk, D), seed + 1, 1.0)
    v = randn((B, H, Lk, D), seed + 2, 1.0)
    g = randn((B, H, Lq, D), seed + 3, 1.0)
    lt = lens_tensor(lens)
    out, lse = mha.mha_fwd_lse(dev(q), dev(k), dev(v), mask, dev(lt), scale=scale)
    dq, dk, dv = mha.mha_bwd(dev(q), dev(k), dev(v), out, dev(g), lse, mask, dev(lt),
                             scale=scale)
    torch.cuda.synchronize()
    return (q, k, v, g), (out, lse, dq, dk, dv)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%dm%d" % c[:6])
def test_backward_parity(case):
    B, H, Lq, Lk, D, mask, lens = case
    (q, k, v, g), (out, lse, dq, dk, dv) = run_case(*case, seed=81)
    qn, kn, vn, gn = (t.numpy() for t in (q, k, v, g))
    check_f32(as_np(out), oracle.mha_fwd(qn, kn, vn, mask, lens), "out %s" % (case,))
    want_lse = oracle.mha_lse(qn, kn, mask, lens)
    got_lse = as_np(lse)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(got_lse), fin), "lse: -inf rows differ"
    if fin.any():
        assert np.abs(got_lse[fin] - want_lse[fin]).max() <= 1e-5, "lse"
    wq, wk, wv = oracle.mha_bwd(qn, kn, vn, gn, mask, lens)
    errs = [check_grad(as_np(t), w, "%s %s" % (n, case))
            for n, t, w in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv))]
    print(case, "dq %.2e dk %.2e dv %.2e" % tuple(errs))
    assert mha.device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [1, 2], ids=["tiled", "short"])
def test_lse_both_forward_kernels(kernel):
    """Both fp32 forward kernels write the same statistic."""
    mha.set_f32_kernel(kernel)
    try:
        (q, k, _, _), (out, lse, _, _, _) = run_case(2, 2, 100, 128, 64, 3, [128, 70], seed=91)
    finally:
        mha.set_f32_kernel(0)
    want = oracle.mha_lse(q.numpy(), k.numpy(), 3, [128, 70])
    assert np.abs(as_np(lse) - want).max() <= 1e-5


@pytest.mark.gpu
def test_backward_hidden_keys_exact():
    """Keys past a batch's length get exactly zero dk and dv; changing their
    values leaves dk and dv of the visible keys bit-identical (dq is summed
    with atomics, so only its values are compared)."""
    B, H, Lq, Lk, D = 2, 2, 150, 200, 64
    lens = [120, 200]
    (q, k, v, g), (_, _, dq, dk, dv) = run_case(B, H, Lq, Lk, D, 3, lens, seed=101)
    assert torch.count_nonzero(dk[0, :, 120:]) == 0 and torch.count_nonzero(dv[0, :, 120:]) == 0
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 120:] = randn((H, Lk - 120, D), 102, 20.0)
    v2[0, :, 120:] = randn((H, Lk - 120, D), 103, 20.0)
    lt = dev(lens_tensor(lens))
    out2, lse2 = mha.mha_fwd_lse(dev(q), dev(k2), dev(v2), 3, lt)
    dq2, dk2, dv2 = mha.mha_bwd(dev(q), dev(k2), dev(v2), out2, dev(g), lse2, 3, lt)
    torch.cuda.synchronize()
    assert torch.equal(dk2[:, :, :120], dk[:, :, :120]) and torch.equal(dv2, dv)
    assert torch.count_nonzero(dk2[0, :, 120:]) == 0
    assert (dq2 - dq).abs().max().item() <= 1e-5


@pytest.mark.gpu
def test_backward_no_query_rows():
    """Lq == 0: no row sees a key, so dk and dv are written as zeros."""
    k = randn((1, 2, 70, 64), 111, 1.0).cuda()
    v = randn((1, 2, 70, 64), 112, 1.0).cuda()
    q = torch.empty((1, 2, 0, 64), device="cuda")
    lse = torch.empty((1, 2, 0), device="cuda")
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    mha.mha_bwd(q, k, v, q, q, lse, 0, None, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


@pytest.mark.gpu
def test_backward_workload_full():
    """The backward workload of the benchmark, every gradient element
    against the oracle."""
    w = synthetic.WORKLOADS["b2_padding_f32_bwd"]
    x = synthetic.make(w, seed=0)
    lt = dev(x["kv_lengths"])
    out, lse = mha.mha_fwd_lse(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, lt, scale=w.scale)
    dq, dk, dv = mha.mha_bwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), out, dev(x["dout"]), lse,
                             w.mask, lt, scale=w.scale)
    torch.cuda.synchronize()
    lens = x["kv_lengths"].numpy()
    wq, wk, wv = oracle.mha_bwd(x["q"].numpy(), x["k"].numpy(), x["v"].numpy(),
                                x["dout"].numpy(), w.mask, lens, w.scale)
    errs = [check_grad(as_np(t), ww, n) for n, t, ww in (("dq", dq, wq), ("dk", dk, wk),
                                                        ("dv", dv, wv))]
    print(w.name, "dq %.2e dk %.2e dv %.2e" % tuple(errs))
    assert mha.device_status() == 0


# bf16: the same computation in fp32 from bf16 inputs, gradients rounded to
# bf16 once.  Error sources beyond fp32 rounding: the bf16 output rounding of
# each gradient (half an ulp, 2^-9 relative) and Delta = dout . o formed from
# the forward's bf16-rounded o (each o element within 2^-9 relative), which
# moves dS = P (dP - Delta) by P * |dout| * |o| * 2^-9 per row.  Bound:
#   per element |gpu - oracle| <= ulp_bf16(oracle) / 2 + BF16_GRAD_ABS * s
#   mean |gpu - oracle| <= BF16_GRAD_MEAN * s,  s = max(1, max |oracle|)
BF16_GRAD_ABS = 1e-2
BF16_GRAD_MEAN = 1e-3

BF16_CASES = [
    (1, 1, 1, 1, 64, 0, None),
    (2, 2, 70, 90, 64, 2, [90, 45]),
    (1, 2, 130, 200, 128, 1, None),
    (2, 3, 257, 129, 64, 3, [1, 129]),
    (2, 2, 64, 64, 128, 2, [0, 64]),
    (2, 2, 4, 700, 128, 2, [700, 300]),   # few query rows: the decode kernel's log-sum-exp
]


def check_grad_bf16(got, want, what):
    from parity_util import ulp_bf16
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), "%s: non-finite gradient" % what
    if got.size == 0:
        return 0.0, 0.0
    s = max(1.0, float(np.abs(want).max()))
    err = np.abs(got - want)
    tol = ulp_bf16(want) / 2 + BF16_GRAD_ABS * s
    bad = err > tol
    assert not bad.any(), "%s: %d elements over tolerance, worst %.3g (scale %.3g)" % (
        what, bad.sum(), err.max(), s)
    assert err.mean() <= BF16_GRAD_MEAN * s, "%s: mean abs %.3g > %.3g" % (
        what, err.mean(), BF16_GRAD_MEAN * s)
    return float(err.max() / s), float(err.mean() / s)


@pytest.fixture
def bwd_kernel(request):
    mha.set_bwd_kernel(request.param)
    yield request.param
    mha.set_bwd_kernel(0)


@pytest.mark.gpu
@pytest.mark.parametrize("bwd_kernel", [0, 1], indirect=True, ids=["tensor", "cudacore"])
@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "B%dH%dLq%dLk%dD%dm%d" % c[:6])
def test_backward_parity_bf16(case, bwd_kernel):
    B, H, Lq, Lk, D, mask, lens = case
    q = randn((B, H, Lq, D), 121, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 122, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 123, 1.0, torch.bfloat16)
    g = randn((B, H, Lq, D), 124, 1.0, torch.bfloat16)
    lt = dev(lens_tensor(lens))
    out, lse = mha.mha_fwd_lse(dev(q), dev(k), dev(v), mask, lt)
    dq, dk, dv = mha.mha_bwd(dev(q), dev(k), dev(v), out, dev(g), lse, mask, lt)
    torch.cuda.synchronize()
    assert dq.dtype == torch.bfloat16 and dk.dtype == torch.bfloat16
    qn, kn, vn, gn = (t.float().numpy() for t in (q, k, v, g))
    want_lse = oracle.mha_lse(qn, kn, mask, lens)
    got_lse = as_np(lse)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(got_lse), fin), "lse: -inf rows differ"
    if fin.any():
        assert np.abs(got_lse[fin] - want_lse[fin]).max() <= 1e-4, "lse"
    wq, wk, wv = oracle.mha_bwd(qn, kn, vn, gn, mask, lens)
    r = [check_grad_bf16(as_np(t), w, "%s %s" % (n, case))
         for n, t, w in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv))]
    print(case, bwd_kernel, "relative max/mean: dq %.1e/%.1e dk %.1e/%.1e dv %.1e/%.1e" % (
        r[0] + r[1] + r[2]))
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_backward_bf16_tensor_deterministic_and_hidden_keys():
    """The tensor-core bf16 backward writes every element once: two runs are
    bit-identical, keys past the length get exactly zero dk and dv, and
    changing their values changes no gradient bit of the visible keys."""
    B, H, Lq, Lk, D = 2, 2, 200, 300, 128
    lens = [130, 300]
    q = randn((B, H, Lq, D), 141, 1.0, torch.bfloat16)
    k = randn((B, H, Lk, D), 142, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 143, 1.0, torch.bfloat16)
    g = randn((B, H, Lq, D), 144, 1.0, torch.bfloat16)
    lt = dev(lens_tensor(lens))

    def run(kk, vv):
        out, lse = mha.mha_fwd_lse(dev(q), dev(kk), dev(vv), 3, lt)
        return mha.mha_bwd(dev(q), dev(kk), dev(vv), out, dev(g), lse, 3, lt)

    a = run(k, v)
    b = run(k, v)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert torch.count_nonzero(a[1][0, :, 130:]) == 0 and torch.count_nonzero(a[2][0, :, 130:]) == 0
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 130:] = randn((H, Lk - 130, D), 145, 20.0, torch.bfloat16)
    v2[0, :, 130:] = randn((H, Lk - 130, D), 146, 20.0, torch.bfloat16)
    c = run(k2, v2)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, c))
    assert mha.device_status() == 0


@pytest.mark.gpu
def test_backward_bf16_workload_sampled_heads():
    """The bf16 backward workload of the benchmark (B1 H32 L2048 D128 causal):
    every gradient element of three heads (first, middle, last) against the
    oracle run on those heads alone (heads are independent problems)."""
    w = synthetic.WORKLOADS["b5_causal_bf16_bwd"]
    x = synthetic.make(w, seed=0)
    out, lse = mha.mha_fwd_lse(dev(x["q"]), dev(x["k"]), dev(x["v"]), w.mask, None, scale=w.scale)
    dq, dk, dv = mha.mha_bwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), out, dev(x["dout"]), lse,
                             w.mask, None, scale=w.scale)
    torch.cuda.synchronize()
    for h in (0, w.H // 2, w.H - 1):
        sl = lambda t: t[:, h:h + 1].float().numpy()
        wq, wk, wv = oracle.mha_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["dout"]), w.mask,
                                    None, w.scale)
        r = [check_grad_bf16(as_np(t[:, h:h + 1]), ww, "%s head %d" % (n, h))
             for n, t, ww in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv))]
        print(w.name, "head", h, "relative max/mean: dq %.1e/%.1e dk %.1e/%.1e dv %.1e/%.1e" % (
            r[0] + r[1] + r[2]))
    assert mha.device_status() == 0
