"""Seeded random sweep: shapes, masks, lengths, scales and dtypes drawn at
random (small enough for the oracle), every output element of mha_fwd,
mha_fwd_lse and mha_fwd_host against the fp64 oracle (GPU).  The fixed cases
elsewhere cover tile boundaries deliberately; this sweep covers the
combinations nobody thought of."""
import numpy as np
import pytest
import torch

import masked_head_attention_gb300 as mha
import oracle
from parity_util import as_np, check_bf16, check_bf16_sum, check_f32, dev, lens_tensor, randn

N_CASES = 40


def _case(i):
    r = np.random.default_rng(1000 + i)
    B = int(r.integers(1, 4))
    H = int(r.integers(1, 5))
    D = int(r.choice([64, 128]))
    Lq = int(r.choice([1, 2, 5, 8, int(r.integers(1, 700))]))
    Lk = int(r.choice([0, 1, 31, 129, int(r.integers(1, 900))]))
    mask = int(r.integers(0, 4))
    lens = None
    if mask & 2:
        lens = [int(x) for x in r.integers(0, Lk + 40, size=B)]
    dtype = torch.float32 if r.random() < 0.4 else torch.bfloat16
    scale = float(r.choice([1.0 / np.sqrt(D), 0.05, 0.3]))
    std = float(r.choice([0.5, 1.0, 3.0]))
    if dtype == torch.float32:
        # The fp32 bound (1e-4 absolute) holds for logits of unit scale, the
        # pages' workloads; the 3xTF32 split's relative error (about 2^-20 per
        # product) grows with |s|.
        scale, std = 1.0 / np.sqrt(D), float(r.choice([0.5, 1.0]))
    return B, H, Lq, Lk, D, mask, lens, dtype, scale, std


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    B, H, Lq, Lk, D, mask, lens, dtype, scale, std = _case(i)
    what = "case %d: B%d H%d Lq%d Lk%d D%d mask%d %s scale %.3g std %.2g lens %s" % (
        i, B, H, Lq, Lk, D, mask, dtype, scale, std, lens)
    q = randn((B, H, Lq, D), 5000 + i, std, dtype)
    k = randn((B, H, Lk, D), 6000 + i, std, dtype)
    v = randn((B, H, Lk, D), 7000 + i, 1.0, dtype)
    lt = lens_tensor(lens)
    want = oracle.mha_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), mask, lens, scale)
    check = check_f32 if dtype == torch.float32 else check_bf16
    out = mha.mha_fwd(dev(q), dev(k), dev(v), mask, dev(lt), scale=scale)
    o2, lse = mha.mha_fwd_lse(dev(q), dev(k), dev(v), mask, dev(lt), scale=scale)
    oh = mha.mha_fwd_host(q.contiguous(), k.contiguous(), v.contiguous(), mask, lt, scale=scale)
    torch.cuda.synchronize()
    check(as_np(out), want, what)
    check(as_np(o2), want, what + " (lse call)")
    check(as_np(oh), want, what + " (host call)")
    # The row log-sum-exp against the oracle's, where a key is visible.
    want_lse = oracle.mha_lse(q.float().numpy(), k.float().numpy(), mask, lens, scale)
    got_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(got_lse), fin), what + ": rows with no visible key"
    if fin.any():
        assert np.max(np.abs(got_lse[fin] - want_lse[fin])) <= 1e-3, what + ": lse"
    assert mha.device_status() == 0


N_PRENORM_CASES = 24


def _prenorm_case(i):
    r = np.random.default_rng(3000 + i)
    B = int(r.integers(1, 4))
    H = int(r.choice([1, 2, 3, 4, 6, 8]))
    D = int(r.choice([64, 128]))
    Lq = int(r.choice([1, 7, 130, 256, 257, int(r.integers(1, 800))]))
    Lk = int(r.choice([1, 64, 129, int(r.integers(1, 700))]))
    lens = None
    if r.random() < 0.6:
        lens = [int(x) for x in r.integers(0, Lk + 30, size=B)]
    shift = float(r.choice([0.0, 0.5, 4.0]))   # row means away from zero
    std = float(r.choice([0.5, 1.0, 2.0]))
    residual = bool(r.random() < 0.4)
    return B, H, Lq, Lk, D, lens, shift, std, residual


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_PRENORM_CASES))
def test_random_prenorm_shape(i):
    """Pre-LN cross-attention (with and without the residual add) on seeded
    random shapes: head counts that do and do not pair into clusters, both
    head sizes, ragged and empty batches, rows with non-zero means."""
    B, H, Lq, Lk, D, lens, shift, std, residual = _prenorm_case(i)
    what = "prenorm case %d: B%d H%d Lq%d Lk%d D%d lens %s shift %g std %g residual %s" % (
        i, B, H, Lq, Lk, D, lens, shift, std, residual)
    N = H * D
    x = (randn((B, Lq, N), 8000 + i, std) + shift).to(torch.bfloat16)
    g = 1.0 + 0.1 * randn((N,), 8100 + i)
    b = 0.1 * randn((N,), 8200 + i)
    k = randn((B, H, Lk, D), 8300 + i, 1.0, torch.bfloat16)
    v = randn((B, H, Lk, D), 8400 + i, 1.0, torch.bfloat16)
    lt = lens_tensor(lens)
    fn = mha.prenorm_cross_attn_residual_fwd if residual else mha.prenorm_cross_attn_fwd
    out = fn(dev(x), dev(g), dev(b), 1e-5, dev(k), dev(v), dev(lt))
    torch.cuda.synchronize()
    ofn = oracle.prenorm_cross_attn_residual if residual else oracle.prenorm_cross_attn
    want = ofn(x.float().numpy(), g.numpy(), b.numpy(), 1e-5, k.float().numpy(), v.float().numpy(),
               lens)
    (check_bf16_sum if residual else check_bf16)(as_np(out), want, what)
    assert mha.device_status() == 0
