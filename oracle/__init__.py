"""fp64 CPU oracle for masked multi-head attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It is the plain definition the CUDA
kernels are checked against and shares no code with them; see oracle.c for
the page sections each function follows.

All functions take numpy arrays of any float dtype, upcast them to fp64 and
return fp64 arrays.  Mask kinds are bit flags: 1 = causal, 2 = kv-length.
"""
import ctypes
import os

import numpy as np

from . import build as _build

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KV_LEN = 2

_lib = None


def lib(path: str = None):
    """Load (building if needed) liboracle.so; a path loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(L):
    P = ctypes.c_void_p
    i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
    L.oracle_num_threads.restype = i
    L.oracle_mha_fwd.argtypes = [P, P, P, i, P, P, i, i, i, i, i, d]
    L.oracle_mha_rows.argtypes = [P, P, P, i, P, P, i64, P, i, i, i, i, i, d]
    L.oracle_softmax_probs.argtypes = [P, P, i, P, P, i, i, i, i, i, d]
    L.oracle_layer_norm.argtypes = [P, P, P, d, P, i64, i]
    L.oracle_prenorm_cross_attn.argtypes = [P, P, P, d, P, P, P, P, i, i, i, i, i, d]
    L.oracle_prenorm_cross_attn_residual.argtypes = [P, P, P, d, P, P, P, P, i, i, i, i, i, d]
    L.oracle_prenorm_rows.argtypes = [P, P, P, d, P, P, P, P, i64, P, i, i, i, i, i, d]
    L.oracle_prenorm_residual_rows.argtypes = [P, P, P, d, P, P, P, P, i64, P, i, i, i, i, i, d]
    L.oracle_mha_lse.argtypes = [P, P, i, P, P, i, i, i, i, i, d]
    L.oracle_mha_bwd.argtypes = [P, P, P, P, i, P, P, P, P, i, i, i, i, i, d]
    for f in ("oracle_mha_fwd", "oracle_mha_rows", "oracle_softmax_probs",
              "oracle_mha_lse", "oracle_mha_bwd",
              "oracle_layer_norm", "oracle_prenorm_cross_attn", "oracle_prenorm_rows",
              "oracle_prenorm_cross_attn_residual", "oracle_prenorm_residual_rows"):
        getattr(L, f).restype = i
    return L


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _lens(kv_lengths):
    if kv_lengths is None:
        return None
    return np.ascontiguousarray(np.asarray(kv_lengths, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError("%s failed with code %d" % (what, rc))


def num_threads(path=None) -> int:
    return lib(path).oracle_num_threads()


def mha_fwd(q, k, v, mask_kind=MASK_NONE, kv_lengths=None, scale=None, path=None):
    """O [B,H,Lq,D] from q [B,H,Lq,D], k/v [B,H,Lk,D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    lens = _lens(kv_lengths)
    out = np.zeros((B, H, Lq, D), np.float64)
    _check(lib(path).oracle_mha_fwd(_p(q), _p(k), _p(v), mask_kind, _p(lens), _p(out),
                                    B, H, Lq, Lk, D, scale), "oracle_mha_fwd")
    return out


def mha_rows(q, k, v, rows, mask_kind=MASK_NONE, kv_lengths=None, scale=None, path=None):
    """Output rows for (b, h, i) triples in `rows` -> [n, D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((rows.shape[0], D), np.float64)
    _check(lib(path).oracle_mha_rows(_p(q), _p(k), _p(v), mask_kind, _p(_lens(kv_lengths)),
                                     _p(rows), rows.shape[0], _p(out), B, H, Lq, Lk, D, scale),
           "oracle_mha_rows")
    return out


def softmax_probs(q, k, mask_kind=MASK_NONE, kv_lengths=None, scale=None, path=None):
    """The softmax matrix P [B,H,Lq,Lk] (small cases)."""
    q, k = _f64(q), _f64(k)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    p = np.zeros((B, H, Lq, Lk), np.float64)
    _check(lib(path).oracle_softmax_probs(_p(q), _p(k), mask_kind, _p(_lens(kv_lengths)), _p(p),
                                          B, H, Lq, Lk, D, scale), "oracle_softmax_probs")
    return p


def mha_lse(q, k, mask_kind=MASK_NONE, kv_lengths=None, scale=None, path=None):
    """Row log-sum-exp of the scaled, masked logits -> [B,H,Lq] (-inf: no visible key)."""
    q, k = _f64(q), _f64(k)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    lse = np.zeros((B, H, Lq), np.float64)
    _check(lib(path).oracle_mha_lse(_p(q), _p(k), mask_kind, _p(_lens(kv_lengths)), _p(lse),
                                    B, H, Lq, Lk, D, scale), "oracle_mha_lse")
    return lse


def mha_bwd(q, k, v, dout, mask_kind=MASK_NONE, kv_lengths=None, scale=None, path=None):
    """Gradients (dq, dk, dv) of sum(dout * mha_fwd(q, k, v)) -> shapes of q, k, v."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    _check(lib(path).oracle_mha_bwd(_p(q), _p(k), _p(v), _p(g), mask_kind,
                                    _p(_lens(kv_lengths)), _p(dq), _p(dk), _p(dv),
                                    B, H, Lq, Lk, D, scale), "oracle_mha_bwd")
    return dq, dk, dv


def layer_norm(x, gamma, beta, eps, path=None):
    x, g, b = _f64(x), _f64(gamma), _f64(beta)
    N = x.shape[-1]
    y = np.zeros_like(x)
    _check(lib(path).oracle_layer_norm(_p(x), _p(g), _p(b), float(eps), _p(y),
                                       x.size // N, N), "oracle_layer_norm")
    return y


def prenorm_cross_attn(x, gamma, beta, eps, k, v, kv_lengths=None, scale=None, path=None):
    """out [B,Lq,H*D] = heads(LN(x)) attended over k/v [B,H,Lk,D]."""
    x, g, b, k, v = _f64(x), _f64(gamma), _f64(beta), _f64(k), _f64(v)
    B, Lq, N = x.shape
    _, H, Lk, D = k.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((B, Lq, N), np.float64)
    _check(lib(path).oracle_prenorm_cross_attn(_p(x), _p(g), _p(b), float(eps), _p(k), _p(v),
                                               _p(_lens(kv_lengths)), _p(out),
                                               B, H, Lq, Lk, D, scale),
           "oracle_prenorm_cross_attn")
    return out


def prenorm_rows(x, gamma, beta, eps, k, v, rows, kv_lengths=None, scale=None, path=None):
    """Rows (b, h, i) of the Pre-LN output, each the head-h slice -> [n, D]."""
    x, g, b, k, v = _f64(x), _f64(gamma), _f64(beta), _f64(k), _f64(v)
    B, Lq, N = x.shape
    _, H, Lk, D = k.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((rows.shape[0], D), np.float64)
    _check(lib(path).oracle_prenorm_rows(_p(x), _p(g), _p(b), float(eps), _p(k), _p(v),
                                         _p(_lens(kv_lengths)), _p(rows), rows.shape[0],
                                         _p(out), B, H, Lq, Lk, D, scale),
           "oracle_prenorm_rows")
    return out


def prenorm_cross_attn_residual(x, gamma, beta, eps, k, v, kv_lengths=None, scale=None,
                                path=None):
    """out [B,Lq,H*D] = x + heads(LN(x)) attended over k/v [B,H,Lk,D]."""
    x, g, b, k, v = _f64(x), _f64(gamma), _f64(beta), _f64(k), _f64(v)
    B, Lq, N = x.shape
    _, H, Lk, D = k.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((B, Lq, N), np.float64)
    _check(lib(path).oracle_prenorm_cross_attn_residual(
        _p(x), _p(g), _p(b), float(eps), _p(k), _p(v), _p(_lens(kv_lengths)), _p(out),
        B, H, Lq, Lk, D, scale), "oracle_prenorm_cross_attn_residual")
    return out


def prenorm_residual_rows(x, gamma, beta, eps, k, v, rows, kv_lengths=None, scale=None,
                          path=None):
    """Rows (b, h, i) of the residual variant, each the head-h slice -> [n, D]."""
    x, g, b, k, v = _f64(x), _f64(gamma), _f64(beta), _f64(k), _f64(v)
    B, Lq, N = x.shape
    _, H, Lk, D = k.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((rows.shape[0], D), np.float64)
    _check(lib(path).oracle_prenorm_residual_rows(_p(x), _p(g), _p(b), float(eps), _p(k), _p(v),
                                                  _p(_lens(kv_lengths)), _p(rows), rows.shape[0],
                                                  _p(out), B, H, Lq, Lk, D, scale),
           "oracle_prenorm_residual_rows")
    return out

