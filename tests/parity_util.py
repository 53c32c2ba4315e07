"""Shared helpers for the GPU parity tests: seeded inputs, oracle calls and the
tolerances written into the tests.

Tolerances (fixed targets of the method):
  fp32 inputs: max abs error <= 1e-4 against the fp64 oracle.
  bf16 inputs: mean abs error <= 1e-3, and per element
      |gpu - oracle| <= ulp_bf16(oracle) / 2 + 1e-2.
  The 1e-2 is the method's budget for the arithmetic (fp32 accumulation, P
  rounded to bf16 before the P.V product).  The half ulp is the one rounding
  of the result to bf16 that the output format itself imposes: it alone
  costs up to 2^-7 = 0.0078 for |O| in [2, 4) and 2^-6 = 0.0156 for |O| in
  [4, 8), so a literal 1e-2 bound can fail for a perfect kernel; below
  |O| = 0.5 the half ulp is at most 2^-10 and the bound is 1e-2 plus that.
  Tests also report how many elements exceed 1e-2.
"""
import math

import numpy as np
import torch

import oracle

F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 1e-2
BF16_MEAN_ABS = 1e-3


def dev(t):
    return None if t is None else t.contiguous().cuda()


def ulp_bf16(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_f32(got, want, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    assert err.max() <= F32_MAX_ABS, "%s: max abs %.3g > %.0e" % (what, err.max(), F32_MAX_ABS)
    return float(err.max())


def check_bf16(got, want, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    tol = 0.5 * ulp_bf16(want) + BF16_MAX_ABS
    bad = err > tol
    assert not bad.any(), "%s: %d elements over tolerance, worst %.3g at oracle %.3g" % (
        what, bad.sum(), err.max(), want.ravel()[err.argmax()])
    assert err.mean() <= BF16_MEAN_ABS, "%s: mean abs %.3g > %.0e" % (what, err.mean(), BF16_MEAN_ABS)
    return dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                over_1e2=int((err > BF16_MAX_ABS).sum()))


def check_bf16_sum(got, want, what=""):
    """For outputs that add a bf16 input to an attention result and round the
    sum once (the residual variant): the rounding alone costs up to half an
    ulp of the result, on top of the attention's own error bounds (1e-2 per
    element, 1e-3 on average).  So per element |gpu - oracle| <=
    ulp_bf16(oracle) / 2 + 1e-2, and on average <= mean(ulp / 2) + 1e-3."""
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    half = 0.5 * ulp_bf16(want)
    bad = err > half + BF16_MAX_ABS
    assert not bad.any(), "%s: %d elements over tolerance, worst %.3g at oracle %.3g" % (
        what, bad.sum(), err.max(), want.ravel()[err.argmax()])
    assert err.mean() <= half.mean() + BF16_MEAN_ABS, "%s: mean abs %.3g > %.3g" % (
        what, err.mean(), half.mean() + BF16_MEAN_ABS)
    return dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                mean_half_ulp=float(half.mean()))


def as_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_rows(B, H, Lq, n, seed, extra=()):
    """(b, h, i) triples: first/last rows, tile boundaries and random rows."""
    r = np.random.default_rng(seed)
    rows = set(extra)
    for i in (0, 1, 63, 64, 127, 128, 129, Lq // 2, Lq - 129, Lq - 128, Lq - 2, Lq - 1):
        if 0 <= i < Lq:
            rows.add((int(r.integers(B)), int(r.integers(H)), i))
    while len(rows) < n:
        rows.add((int(r.integers(B)), int(r.integers(H)), int(r.integers(Lq))))
    return np.array(sorted(rows), np.int64)


def randn(shape, seed, std=1.0, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def lens_tensor(vals):
    return None if vals is None else torch.tensor(vals, dtype=torch.int32)
