"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each check takes an optional `path` to a liboracle build so the same suite can
be run against deliberately broken copies of the oracle (tests/test_oracle_mutants.py).
A check returns None on success or a short failure string.

Sources: "masked multi head attention" CUDA article (2kiu.com), sections 3.1
and 3.2; "why attention computes the max first" essay (gsyq.cn), sections
2.1, 3.1, 4.1 and 5.2; "fuse cross-attention and layer-norm" answer
(cms365.cn), knowledge points and steps two and three.
"""
import glob
import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _brute(q, k, v, mask_kind, lens, scale):
    """Independent restatement in pure Python: exp(s)/sum exp(s) with no shift
    (values are small, so nothing overflows), visible keys only."""
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    out = np.zeros((B, H, Lq, D))
    for b in range(B):
        n = Lk if lens is None else max(0, min(Lk, int(lens[b])))
        for h in range(H):
            for i in range(Lq):
                ws = []
                for j in range(Lk):
                    if j >= n or ((mask_kind & 1) and j > i):
                        continue
                    s = scale * sum(float(q[b, h, i, d]) * float(k[b, h, j, d]) for d in range(D))
                    ws.append((j, math.exp(s)))
                z = sum(w for _, w in ws)
                for j, w in ws:
                    for d in range(D):
                        out[b, h, i, d] += (w / z) * float(v[b, h, j, d])
    return out


def _visible(mask_kind, lens, B, Lq, Lk):
    vis = np.ones((B, Lq, Lk), bool)
    if mask_kind & 1:
        vis &= np.tril(np.ones((Lq, Lk), bool))[None]
    if mask_kind & 2:
        for b in range(B):
            vis[b, :, int(lens[b]):] = False
    return vis


def _sdpa(q, k, v, mask_kind, lens, scale):
    """torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU,
    with a boolean mask built from the same rule (library routine)."""
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    vis = torch.from_numpy(_visible(mask_kind, lens, B, Lq, Lk))[:, None]
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    return torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), attn_mask=vis, scale=scale).numpy()


def check_brute_force(path=None):
    r = _rng(1)
    for (B, H, Lq, Lk, D) in [(1, 1, 1, 1, 1), (2, 2, 5, 7, 3), (1, 3, 8, 8, 4), (2, 1, 6, 4, 2)]:
        for mk in (0, 1, 2, 3):
            q, k, v = (r.standard_normal((B, H, L, D)) for L in (Lq, Lk, Lk))
            lens = r.integers(1, Lk + 1, size=B).astype(np.int32) if mk & 2 else None
            sc = 1.0 / math.sqrt(D)
            got = oracle.mha_fwd(q, k, v, mk, lens, sc, path=path)
            want = _brute(q, k, v, mk, lens, sc)
            if not np.allclose(got, want, rtol=0, atol=1e-12):
                return "brute force mismatch %s mask %d: %g" % (
                    (B, H, Lq, Lk, D), mk, np.abs(got - want).max())
    return None


def check_sdpa(path=None):
    r = _rng(2)
    for (B, H, Lq, Lk, D) in [(2, 3, 33, 33, 16), (1, 2, 17, 40, 8), (3, 1, 64, 64, 32)]:
        for mk in (0, 1, 2, 3):
            q, k, v = (r.standard_normal((B, H, L, D)) for L in (Lq, Lk, Lk))
            lens = r.integers(1, Lk + 1, size=B).astype(np.int32) if mk & 2 else None
            sc = 0.37
            got = oracle.mha_fwd(q, k, v, mk, lens, sc, path=path)
            want = _sdpa(q, k, v, mk, lens, sc)
            if not np.allclose(got, want, rtol=0, atol=1e-12):
                return "sdpa mismatch %s mask %d: %g" % ((B, H, Lq, Lk, D), mk,
                                                         np.abs(got - want).max())
    return None


def check_golden(path=None):
    files = sorted(glob.glob(os.path.join(GOLDEN, "closed_form_*.json")))
    if not files:
        return "no golden fixtures"
    for f in files:
        g = json.load(open(f))
        tol = g["tol"]
        if g["op"] == "mha":
            s = g["shape"]
            B, H, Lq, Lk, D = s["B"], s["H"], s["Lq"], s["Lk"], s["D"]
            q = np.array(g["q"], float).reshape(B, H, Lq, D)
            k = np.array(g["k"], float).reshape(B, H, Lk, D)
            v = np.array(g["v"], float).reshape(B, H, Lk, D)
            lens = g.get("kv_lengths")
            out = oracle.mha_fwd(q, k, v, g["mask_kind"], lens, g["scale"], path=path)
            if np.abs(out.ravel() - np.array(g["expected_out"])).max() > tol:
                return "golden %s: out %s" % (os.path.basename(f), out.ravel())
            if "expected_p" in g:
                p = oracle.softmax_probs(q, k, g["mask_kind"], lens, g["scale"], path=path)
                if np.abs(p.ravel() - np.array(g["expected_p"])).max() > tol:
                    return "golden %s: p %s" % (os.path.basename(f), p.ravel())
        elif g["op"] == "layer_norm":
            for sfx in ("", "2"):
                y = oracle.layer_norm(np.array(g["rows" + sfx]), g["gamma" + sfx],
                                      g["beta" + sfx], g["eps" + sfx], path=path)
                if np.abs(y - np.array(g["expected" + sfx])).max() > tol:
                    return "golden %s%s: %s" % (os.path.basename(f), sfx, y)
    return None


def check_shift_invariance(path=None):
    """Adding one vector w to every key adds scale*q_i.w to every logit of row i,
    a per-row constant, so the output must not move (max-shift, essay 3.1)."""
    r = _rng(3)
    B, H, L, D = 2, 2, 24, 8
    q, k, v = (r.standard_normal((B, H, L, D)) for _ in range(3))
    w = 3.0 * r.standard_normal(D)
    for mk in (0, 1):
        a = oracle.mha_fwd(q, k, v, mk, None, 0.5, path=path)
        b = oracle.mha_fwd(q, k + w, v, mk, None, 0.5, path=path)
        if np.abs(a - b).max() > 1e-12:
            return "shift invariance broken: %g" % np.abs(a - b).max()
    return None


def check_rows_sum_to_one(path=None):
    r = _rng(4)
    B, H, Lq, Lk, D = 2, 2, 9, 13, 4
    q, k = r.standard_normal((B, H, Lq, D)), r.standard_normal((B, H, Lk, D))
    lens = np.array([5, 13], np.int32)
    for mk in (0, 1, 2, 3):
        p = oracle.softmax_probs(q, k, mk, lens if mk & 2 else None, 0.5, path=path)
        if np.abs(p.sum(-1) - 1).max() > 1e-13:
            return "rows do not sum to 1 (mask %d)" % mk
        vis = _visible(mk, lens, B, Lq, Lk)[:, None]
        if np.any(p[~np.broadcast_to(vis, p.shape)] != 0.0):
            return "hidden key has nonzero weight (mask %d)" % mk
        if np.any(p[np.broadcast_to(vis, p.shape)] <= 0.0):
            return "visible key has zero weight (mask %d)" % mk
    return None


def check_zero_query_is_mean(path=None):
    r = _rng(5)
    B, H, L, D = 2, 3, 11, 5
    k, v = r.standard_normal((B, H, L, D)), r.standard_normal((B, H, L, D))
    q = np.zeros((B, H, L, D))
    lens = np.array([4, 11], np.int32)
    o = oracle.mha_fwd(q, k, v, 3, lens, 0.9, path=path)
    for b in range(B):
        for i in range(L):
            n = min(i + 1, int(lens[b]))
            want = v[b, :, :n].mean(axis=1)
            if np.abs(o[b, :, i] - want).max() > 1e-13:
                return "Q=0 row %d of batch %d is not the mean of its visible keys" % (i, b)
    return None


def check_causal_rules(path=None):
    r = _rng(6)
    B, H, L, D = 1, 2, 16, 4
    q, k, v = (r.standard_normal((B, H, L, D)) for _ in range(3))
    o = oracle.mha_fwd(q, k, v, 1, None, 0.5, path=path)
    if not np.array_equal(o[:, :, 0], v[:, :, 0]):
        return "causal row 0 is not V[0]"
    for i in (0, 5, 14):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = r.standard_normal(k2[:, :, i + 1:].shape) * 50
        v2[:, :, i + 1:] = r.standard_normal(v2[:, :, i + 1:].shape) * 50
        o2 = oracle.mha_fwd(q, k2, v2, 1, None, 0.5, path=path)
        if not np.array_equal(o[:, :, i], o2[:, :, i]):
            return "causal row %d depends on later keys" % i
    return None


def check_padding_rules(path=None):
    r = _rng(7)
    B, H, L, D = 3, 2, 12, 4
    q, k, v = (r.standard_normal((B, H, L, D)) for _ in range(3))
    lens = np.array([1, 7, 12], np.int32)
    o = oracle.mha_fwd(q, k, v, 2, lens, 0.5, path=path)
    if not np.array_equal(o[0], np.broadcast_to(v[0, :, :1], o[0].shape)):
        return "len 1 rows are not V[0]"
    k2, v2 = k.copy(), v.copy()
    k2[1, :, 7:] = 1e6
    v2[1, :, 7:] = -1e6
    o2 = oracle.mha_fwd(q, k2, v2, 2, lens, 0.5, path=path)
    if not np.array_equal(o, o2):
        return "keys beyond the length changed the output"
    perm = np.concatenate([r.permutation(7), np.arange(7, L)])
    o3 = oracle.mha_fwd(q, k[:, :, perm], v[:, :, perm], 2, lens, 0.5, path=path)
    if np.abs(o3[1] - o[1]).max() > 1e-13:
        return "permuting visible keys changed the output"
    oz = oracle.mha_fwd(q, k, v, 2, np.array([0, 7, 12], np.int32), 0.5, path=path)
    if np.any(oz[0] != 0) or np.any(np.isnan(oz)):
        return "a row with no visible key is not zero"
    return None


def check_hard_max_and_overflow(path=None):
    r = _rng(8)
    D = 4
    k = r.standard_normal((1, 1, 6, D)) * 0.1
    v = r.standard_normal((1, 1, 6, D))
    q = np.zeros((1, 1, 1, D))
    q[..., 0] = 1.0
    k[0, 0, 3, 0] = 50.0                  # logit gap of about 50
    o = oracle.mha_fwd(q, k, v, 0, None, 1.0, path=path)
    if np.abs(o[0, 0, 0] - v[0, 0, 3]).max() > 1e-12:
        return "hard-max limit not reached"
    big = oracle.mha_fwd(q * 1000.0, k, v, 0, None, 1.0, path=path)   # logits ~5e4
    if not np.all(np.isfinite(big)) or np.abs(big[0, 0, 0] - v[0, 0, 3]).max() > 1e-12:
        return "large logits overflow"
    return None


def check_rows_api(path=None):
    r = _rng(9)
    B, H, Lq, Lk, D = 2, 2, 10, 13, 8
    q, k, v = r.standard_normal((B, H, Lq, D)), r.standard_normal((B, H, Lk, D)), \
        r.standard_normal((B, H, Lk, D))
    lens = np.array([3, 13], np.int32)
    full = oracle.mha_fwd(q, k, v, 3, lens, 0.3, path=path)
    rows = [(0, 1, 9), (1, 0, 0), (1, 1, 5)]
    got = oracle.mha_rows(q, k, v, rows, 3, lens, 0.3, path=path)
    want = np.stack([full[b, h, i] for b, h, i in rows])
    if not np.array_equal(got, want):
        return "row API differs from the full forward"
    return None


def check_layer_norm(path=None):
    r = _rng(10)
    x = r.standard_normal((7, 96)) * 3 + 1.5
    g, b = r.standard_normal(96), r.standard_normal(96)
    y = oracle.layer_norm(x, g, b, 1e-5, path=path)
    t = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g),
                                       torch.from_numpy(b), 1e-5).numpy()
    if np.abs(y - t).max() > 1e-12:
        return "layer_norm differs from torch: %g" % np.abs(y - t).max()
    y1 = oracle.layer_norm(x, np.ones(96), np.zeros(96), 0.0, path=path)
    if np.abs(y1.mean(-1)).max() > 1e-13 or np.abs(y1.var(-1) - 1).max() > 1e-12:
        return "unit layer_norm rows are not zero-mean unit-variance"
    return None


def check_prenorm(path=None):
    """Pre-LN cross-attention against an independent torch composition:
    layer_norm -> head split -> SDPA with the length mask -> head merge."""
    r = _rng(11)
    B, H, Lq, Lk, D = 2, 3, 9, 14, 8
    x = r.standard_normal((B, Lq, H * D)) * 2 + 0.5
    g = 1 + 0.1 * r.standard_normal(H * D)
    be = 0.1 * r.standard_normal(H * D)
    k, v = r.standard_normal((B, H, Lk, D)), r.standard_normal((B, H, Lk, D))
    lens = np.array([5, 14], np.int32)
    got = oracle.prenorm_cross_attn(x, g, be, 1e-5, k, v, lens, 0.35, path=path)
    xn = torch.nn.functional.layer_norm(torch.from_numpy(x), (H * D,), torch.from_numpy(g),
                                        torch.from_numpy(be), 1e-5)
    q = xn.reshape(B, Lq, H, D).permute(0, 2, 1, 3).numpy()
    o = _sdpa(q, k, v, 2, lens, 0.35)
    want = o.transpose(0, 2, 1, 3).reshape(B, Lq, H * D)
    if np.abs(got - want).max() > 1e-12:
        return "prenorm differs from LN+SDPA: %g" % np.abs(got - want).max()
    rows = [(0, 2, 8), (1, 0, 0), (1, 1, 4)]
    pr = oracle.prenorm_rows(x, g, be, 1e-5, k, v, rows, lens, 0.35, path=path)
    for n, (b, h, i) in enumerate(rows):
        if np.abs(pr[n] - got[b, i, h * D:(h + 1) * D]).max() > 1e-13:
            return "prenorm row API differs from the full op"
    cst = np.full((1, 2, H * D), 4.25)
    kk, vv = r.standard_normal((1, H, 3, D)), r.standard_normal((1, H, 3, D))
    oc = oracle.prenorm_cross_attn(cst, g, be, 1e-5, kk, vv, None, 0.35, path=path)
    qc = np.broadcast_to(be.reshape(H, D)[None, :, None, :], (1, H, 2, D))
    wc = oracle.mha_fwd(qc, kk, vv, 0, None, 0.35, path=path).transpose(0, 2, 1, 3).reshape(1, 2, -1)
    if np.abs(oc - wc).max() > 1e-12:
        return "constant rows do not normalise to beta"
    return None


def check_prenorm_residual(path=None):
    """Residual variant ("How to fuse cross-attention and layer-norm into a
    single CUDA kernel?", answer step four: output + src).  gamma = beta = 0
    makes every LN row zero, so Q = 0 and each head's attention is the mean of
    its visible V rows: out = x + that mean (a closed form).  V = 0 leaves
    exactly x.  The row API must agree with the full op."""
    r = _rng(12)
    B, H, Lq, Lk, D = 2, 3, 5, 7, 4
    x = r.standard_normal((B, Lq, H * D)) * 1.5 - 0.25
    k, v = r.standard_normal((B, H, Lk, D)), r.standard_normal((B, H, Lk, D))
    lens = np.array([3, 7], np.int32)
    z = np.zeros(H * D)
    got = oracle.prenorm_cross_attn_residual(x, z, z, 1e-5, k, v, lens, 0.5, path=path)
    want = x.copy()
    for b in range(B):
        for h in range(H):
            want[b, :, h * D:(h + 1) * D] += v[b, h, :lens[b]].mean(axis=0)
    if np.abs(got - want).max() > 1e-12:
        return "gamma = beta = 0 is not x + mean of visible V: %g" % np.abs(got - want).max()
    g = 1 + 0.1 * r.standard_normal(H * D)
    be = 0.1 * r.standard_normal(H * D)
    got0 = oracle.prenorm_cross_attn_residual(x, g, be, 1e-5, k, np.zeros_like(v), lens, 0.5,
                                              path=path)
    if np.abs(got0 - x).max() > 1e-15:
        return "V = 0 does not return x"
    full = oracle.prenorm_cross_attn_residual(x, g, be, 1e-5, k, v, lens, 0.5, path=path)
    rows = [(0, 2, 4), (1, 0, 0), (1, 1, 3)]
    pr = oracle.prenorm_residual_rows(x, g, be, 1e-5, k, v, rows, lens, 0.5, path=path)
    for n, (b, h, i) in enumerate(rows):
        if np.abs(pr[n] - full[b, i, h * D:(h + 1) * D]).max() > 1e-13:
            return "residual row API differs from the full op"
    return None


def _loss(q, k, v, g, mk, lens, sc, path):
    return float((oracle.mha_fwd(q, k, v, mk, lens, sc, path=path) * g).sum())


def check_bwd_finite_difference(path=None):
    """Every gradient element against a central difference of the (pinned)
    forward oracle's loss sum(dout * O): error O(eps^2), far below 1e-8.
    Covers all masks, Lq != Lk both ways and a batch with no visible key."""
    r = _rng(21)
    eps = 1e-5
    cases = [(1, 1, 1, 1, 1, 0, None), (2, 2, 5, 6, 3, 0, None), (2, 2, 5, 6, 3, 1, None),
             (2, 2, 5, 6, 3, 2, [4, 0]), (2, 1, 5, 6, 3, 3, [2, 6]), (1, 2, 4, 7, 2, 1, None),
             (1, 2, 6, 3, 2, 3, [3])]
    for (B, H, Lq, Lk, D, mk, lens) in cases:
        q, k, v = (r.standard_normal((B, H, L, D)) for L in (Lq, Lk, Lk))
        g = r.standard_normal((B, H, Lq, D))
        lens = None if lens is None else np.array(lens, np.int32)
        sc = 0.8
        grads = oracle.mha_bwd(q, k, v, g, mk, lens, sc, path=path)
        for name, x, gx in zip("qkv", (q, k, v), grads):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p["qkv".index(name)] = xp
                args_m["qkv".index(name)] = xm
                fd = (_loss(*args_p, g, mk, lens, sc, path) -
                      _loss(*args_m, g, mk, lens, sc, path)) / (2 * eps)
                if abs(fd - gx[idx]) > 1e-8:
                    return "d%s%s: oracle %.12g, finite difference %.12g (case %s)" % (
                        name, idx, gx[idx], fd, (B, H, Lq, Lk, D, mk))
    return None


def check_bwd_autograd(path=None):
    """Against torch autograd through fp64 SDPA with the same boolean mask
    (library routine); every row keeps at least one visible key."""
    r = _rng(22)
    for (B, H, Lq, Lk, D) in [(2, 3, 17, 23, 8), (1, 2, 40, 40, 16)]:
        for mk in (0, 1, 2, 3):
            q, k, v = (r.standard_normal((B, H, L, D)) for L in (Lq, Lk, Lk))
            g = r.standard_normal((B, H, Lq, D))
            lens = r.integers(1, Lk + 1, size=B).astype(np.int32) if mk & 2 else None
            sc = 0.3
            got = oracle.mha_bwd(q, k, v, g, mk, lens, sc, path=path)
            t = [torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, k, v)]
            vis = torch.from_numpy(_visible(mk, lens, B, Lq, Lk))[:, None]
            o = torch.nn.functional.scaled_dot_product_attention(*t, attn_mask=vis, scale=sc)
            o.backward(torch.from_numpy(g))
            for name, a, tt in zip("qkv", got, t):
                err = np.abs(a - tt.grad.numpy()).max()
                if err > 1e-12:
                    return "d%s differs from autograd by %g (shape %s mask %d)" % (
                        name, err, (B, H, Lq, Lk, D), mk)
    return None


def check_bwd_invariants(path=None):
    """Closed forms: softmax rows sum to one, so sum_j dv_j = sum of dout over
    rows with a visible key, and shifting every key by one vector leaves O
    unchanged, so sum_j dk_j = 0; hidden keys get exactly zero gradient; with
    a single key O = v_0 for every row, so dq = dk = 0 and dv_0 = sum_i dout_i;
    with q = 0 the weights are uniform over the n_i visible keys, so
    dv_j = sum_{i sees j} dout_i / n_i."""
    r = _rng(23)
    B, H, Lq, Lk, D = 3, 2, 19, 26, 5
    q, k, v = (r.standard_normal((B, H, L, D)) for L in (Lq, Lk, Lk))
    g = r.standard_normal((B, H, Lq, D))
    lens = np.array([9, 0, 26], np.int32)
    for mk in (2, 3):
        dq, dk, dv = oracle.mha_bwd(q, k, v, g, mk, lens, 0.5, path=path)
        vis = _visible(mk, lens, B, Lq, Lk)
        rows = vis.any(axis=2)
        for b in range(B):
            want = (g[b] * rows[b][None, :, None]).sum(axis=1)
            if np.abs(dv[b].sum(axis=1) - want).max() > 1e-12:
                return "sum of dv is not the sum of dout (mask %d, batch %d)" % (mk, b)
            if np.abs(dk[b].sum(axis=1)).max() > 1e-12:
                return "sum of dk is not zero (mask %d, batch %d)" % (mk, b)
            hidden = ~vis[b].any(axis=0)
            if np.any(dk[b][:, hidden] != 0) or np.any(dv[b][:, hidden] != 0):
                return "a hidden key received gradient (mask %d, batch %d)" % (mk, b)
            if not rows[b].all() and np.any(dq[b][:, ~rows[b]] != 0):
                return "a row with no visible key passed gradient to q"
    k1, v1 = r.standard_normal((1, 2, 1, D)), r.standard_normal((1, 2, 1, D))
    q1, g1 = r.standard_normal((1, 2, 7, D)), r.standard_normal((1, 2, 7, D))
    dq, dk, dv = oracle.mha_bwd(q1, k1, v1, g1, 0, None, 0.5, path=path)
    if np.abs(dq).max() > 1e-13 or np.abs(dk).max() > 1e-13:
        return "single key: dq/dk not zero"
    if np.abs(dv[0, :, 0] - g1[0].sum(axis=1)).max() > 1e-12:
        return "single key: dv is not the sum of dout"
    z = np.zeros((B, H, Lq, D))
    for mk in (0, 1, 3):
        _, _, dv = oracle.mha_bwd(z, k, v, g, mk, lens, 0.5, path=path)
        vis = _visible(mk, lens, B, Lq, Lk).astype(float)
        n = vis.sum(axis=2, keepdims=True)
        w = np.divide(vis, n, out=np.zeros_like(vis), where=n > 0)
        want = np.einsum("bij,bhid->bhjd", w, g)
        if np.abs(dv - want).max() > 1e-12:
            return "q = 0: dv is not the uniform-weight sum (mask %d)" % mk
    return None


def check_lse(path=None):
    """Row log-sum-exp: brute force with plain exp/log on small logits; q = 0
    gives log(number of visible keys); no visible key gives -inf; huge logits
    (exp would overflow) give max + log(1 + sum exp(s - max)) exactly."""
    r = _rng(24)
    B, H, Lq, Lk, D = 2, 2, 6, 5, 3
    q, k = r.standard_normal((B, H, Lq, D)), r.standard_normal((B, H, Lk, D))
    lens = np.array([3, 0], np.int32)
    for mk in (0, 1, 2, 3):
        got = oracle.mha_lse(q, k, mk, lens, 0.7, path=path)
        vis = _visible(mk, lens, B, Lq, Lk)
        for b, h, i in np.ndindex(B, H, Lq):
            js = [j for j in range(Lk) if vis[b, i, j]]
            if not js:
                if got[b, h, i] != -np.inf:
                    return "empty row lse %r" % got[b, h, i]
                continue
            want = math.log(sum(math.exp(0.7 * float(q[b, h, i] @ k[b, h, j])) for j in js))
            if abs(got[b, h, i] - want) > 1e-13:
                return "lse brute force (%d,%d,%d) mask %d: %r vs %r" % (b, h, i, mk, got[b, h, i], want)
    z = oracle.mha_lse(np.zeros((B, H, Lq, D)), k, 3, np.array([4, 2], np.int32), 0.7, path=path)
    n = _visible(3, np.array([4, 2]), B, Lq, Lk).sum(axis=2)
    if np.abs(z - np.log(n)[:, None, :]).max() > 1e-14:
        return "q = 0: lse is not log(n)"
    qh = np.array([[[[1.0]]]])
    kh = np.array([[[[1000.0], [999.0], [-5.0]]]])
    got = oracle.mha_lse(qh, kh, 0, None, 1.0, path=path)[0, 0, 0]
    want = 1000.0 + math.log1p(math.exp(-1.0) + math.exp(-1005.0))
    if not np.isfinite(got) or abs(got - want) > 1e-12:
        return "large logits: lse %r want %r" % (got, want)
    return None


ALL = [check_brute_force, check_sdpa, check_golden, check_shift_invariance,
       check_rows_sum_to_one, check_zero_query_is_mean, check_causal_rules,
       check_padding_rules, check_hard_max_and_overflow, check_rows_api,
       check_layer_norm, check_prenorm, check_prenorm_residual, check_bwd_finite_difference,
       check_bwd_autograd, check_bwd_invariants, check_lse]


def run_all(path=None):
    fails = []
    for c in ALL:
        try:
            msg = c(path)
        except Exception as e:  # a crash of a broken build counts as caught
            msg = "%s raised %r" % (c.__name__, e)
        if msg:
            fails.append("%s: %s" % (c.__name__, msg))
    return fails
