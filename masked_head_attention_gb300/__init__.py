"""GB300 (sm_103a) fused masked multi-head attention: forward, decode and backward.

Thin ctypes binding over the C ABI of libmha.so (include/mha.h).  Every step
of the computation runs in the library's CUDA kernels; this module only
checks tensor metadata and passes device pointers, sizes and the current
CUDA stream.  PyTorch provides device memory and streams, nothing else.

There is no fallback: if libmha.so has not been built (see build.py, or
``__graft_entry__.build()``), every call raises ``MhaError``.
"""
import ctypes
import math
import os

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KV_LEN = 2
F32 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmha.so")
_lib = None


class MhaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, _strerror_safe(status), status))


def _strerror_safe(code):
    try:
        return lib().mha_strerror(code).decode()
    except Exception:  # library itself unavailable
        return "status %d" % code


def lib():
    """The loaded libmha.so (raises MhaError when it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MhaError(-4, "loading %s (not built)" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.mha_fwd.argtypes = [P, P, P, i, P, P, i, i, i, i, i, f, i, P]
        L.mha_fwd.restype = i
        L.prenorm_cross_attn_fwd.argtypes = [P, P, P, f, P, P, P, P, i, i, i, i, i, f, i, P]
        L.prenorm_cross_attn_fwd.restype = i
        L.prenorm_cross_attn_residual_fwd.argtypes = [P, P, P, f, P, P, P, P, i, i, i, i, i, f, i, P]
        L.prenorm_cross_attn_residual_fwd.restype = i
        L.mha_fwd_lse.argtypes = [P, P, P, i, P, P, P, i, i, i, i, i, f, i, P]
        L.mha_fwd_lse.restype = i
        L.mha_bwd.argtypes = [P, P, P, P, P, P, i, P, P, P, P, i, i, i, i, i, f, i, P,
                              ctypes.c_size_t, P]
        L.mha_bwd.restype = i
        L.mha_bwd_workspace_size.argtypes = [i, i, i, i, i]
        L.mha_bwd_workspace_size.restype = ctypes.c_size_t
        L.mha_fwd_host.argtypes = [P, P, P, i, P, P, i, i, i, i, i, f, i, P, ctypes.c_size_t, P]
        L.mha_fwd_host.restype = i
        L.mha_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
        L.mha_fwd_host_workspace_size.restype = ctypes.c_size_t
        L.mha_test_set_device_status.argtypes = [i, ctypes.c_uint32]
        L.mha_test_set_device_status.restype = i
        L.mha_test_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.mha_test_set_wait_limit_ns.restype = i
        L.mha_strerror.argtypes = [i]
        L.mha_strerror.restype = ctypes.c_char_p
        L.mha_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i]
        L.mha_device_status.restype = i
        L.mha_selftest_umma.argtypes = [i, i, P, P, P, P]
        L.mha_selftest_umma.restype = i
        L.mha_set_bf16_grid.argtypes = [i]
        L.mha_set_bf16_grid.restype = None
        L.mha_plan_prenorm.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int64)]
        L.mha_plan_prenorm.restype = i
        L.mha_set_f32_kernel.argtypes = [i]
        L.mha_set_f32_kernel.restype = None
        L.mha_set_bf16_decode.argtypes = [i]
        L.mha_set_bf16_decode.restype = None
        L.mha_set_bf16_decode_splits.argtypes = [i]
        L.mha_set_bf16_decode_splits.restype = None
        L.mha_set_bwd_kernel.argtypes = [i]
        L.mha_set_bwd_kernel.restype = None
        L.mha_set_pdl.argtypes = [i]
        L.mha_set_pdl.restype = None
        _lib = L
    return _lib


_torch_mod = None
_raw_stream = None


def _torch():
    global _torch_mod, _raw_stream
    if _torch_mod is None:
        import torch
        _torch_mod = torch
        # The raw handle of the current stream without building a Stream object
        # (a few microseconds per call otherwise).
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    return _torch_mod


def _stream(stream, device_index=None):
    torch = _torch()
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device() if device_index is None else device_index)
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dev(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _check(status, what):
    if status != 0:
        raise MhaError(status, what)


def mha_fwd(q, k, v, mask_kind=MASK_NONE, kv_lengths=None, out=None, scale=None, stream=None):
    """Fused masked MHA forward; q [B,H,Lq,D], k/v [B,H,Lk,D] (fp32 or bf16).

    mask_kind: MASK_CAUSAL and/or MASK_KV_LEN bits; kv_lengths int32 [B] on
    the device when MASK_KV_LEN is set.  Returns `out` [B,H,Lq,D]."""
    torch = _torch()
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B,H,Lk,D] matching q")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    else:
        _dev(out, "out", q.dtype)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().mha_fwd(_ptr(q), _ptr(k), _ptr(v), int(mask_kind), _ptr(kv_lengths), _ptr(out),
                         B, H, Lq, Lk, D, scale, _dtype_code(q), _stream(stream, q.get_device())),
           "mha_fwd")
    return out


def mha_fwd_lse(q, k, v, mask_kind=MASK_NONE, kv_lengths=None, out=None, lse=None, scale=None,
                stream=None):
    """mha_fwd that also returns each row's log-sum-exp (fp32 or bf16 inputs).

    Returns (out [B,H,Lq,D] of q's dtype, lse [B,H,Lq] fp32, natural log,
    -inf for a row with no visible key)."""
    torch = _torch()
    _dev(q, "q")
    _dev(k, "k", q.dtype)
    _dev(v, "v", q.dtype)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B,H,Lk,D] matching q")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    out = torch.empty_like(q) if out is None else _dev(out, "out", q.dtype)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    else:
        _dev(lse, "lse", torch.float32)
        if tuple(lse.shape) != (B, H, Lq):
            raise ValueError("lse must be [B,H,Lq]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().mha_fwd_lse(_ptr(q), _ptr(k), _ptr(v), int(mask_kind), _ptr(kv_lengths),
                             _ptr(out), _ptr(lse), B, H, Lq, Lk, D, scale, _dtype_code(q),
                             _stream(stream, q.get_device())), "mha_fwd_lse")
    return out, lse


def _host(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def mha_fwd_host_workspace_size(B, H, Lq, Lk, D, dtype):
    """Bytes of device workspace mha_fwd_host needs (dtype: F32 or BF16 code)."""
    return int(lib().mha_fwd_host_workspace_size(int(B), int(H), int(Lq), int(Lk), int(D),
                                                 int(dtype)))


def mha_fwd_host(q, k, v, mask_kind=MASK_NONE, kv_lengths=None, out=None, scale=None,
                 workspace=None, device=None, stream=None):
    """mha_fwd on HOST tensors (pinned memory for overlapped copies): copies in,
    computes and copies out in pieces, the copies overlapping the kernels.

    q [B,H,Lq,D], k/v [B,H,Lk,D] (fp32 or bf16), kv_lengths host int32 [B].
    `out` (host, pinned when omitted) receives the result once the stream
    reaches the end of the call (synchronise before reading it).
    `workspace` is a device uint8 tensor of at least
    mha_fwd_host_workspace_size(...) bytes; when omitted, one is taken from
    torch's allocator for this call (the library itself never allocates)."""
    torch = _torch()
    _host(q, "q")
    _host(k, "k", q.dtype)
    _host(v, "v", q.dtype)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B,H,Lk,D] matching q")
    if kv_lengths is not None:
        _host(kv_lengths, "kv_lengths", torch.int32)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    else:
        _host(out, "out", q.dtype)
    dt = _dtype_code(q)
    dev_index = torch.cuda.current_device() if device is None else int(device)
    need = mha_fwd_host_workspace_size(B, H, Lq, Lk, D, dt)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8,
                                device=torch.device("cuda", dev_index))
    else:
        _dev(workspace, "workspace")
        dev_index = workspace.get_device()
    wbytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().mha_fwd_host(_ptr(q), _ptr(k), _ptr(v), int(mask_kind), _ptr(kv_lengths),
                              _ptr(out), B, H, Lq, Lk, D, scale, dt, _ptr(workspace), wbytes,
                              _stream(stream, dev_index)), "mha_fwd_host")
    return out


def mha_bwd_workspace_size(B, H, Lq, D, dtype):
    """Bytes of device workspace mha_bwd needs (dtype: F32 or BF16 code)."""
    return int(lib().mha_bwd_workspace_size(int(B), int(H), int(Lq), int(D), int(dtype)))


def mha_bwd(q, k, v, out, dout, lse, mask_kind=MASK_NONE, kv_lengths=None, dq=None, dk=None,
            dv=None, scale=None, stream=None, workspace=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for out, lse = mha_fwd_lse(q, k, v, ...).

    fp32 or bf16 (q, k, v, out, dout and the gradients of one dtype; lse fp32);
    every tensor contiguous on the same device.  q, k, v, mask_kind,
    kv_lengths and scale must be those of the forward call.  `workspace` is
    a device uint8 tensor of at least mha_bwd_workspace_size(...) bytes; when
    omitted, one is taken from torch's allocator for this call (the library
    itself never allocates)."""
    torch = _torch()
    _dev(q, "q")
    for t, n in ((k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _dev(t, n, q.dtype)
    _dev(lse, "lse", torch.float32)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B,H,Lk,D] matching q")
    if tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("out and dout must have the shape of q")
    if tuple(lse.shape) != (B, H, Lq):
        raise ValueError("lse must be [B,H,Lq]")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    dq = torch.empty_like(q) if dq is None else _dev(dq, "dq", q.dtype)
    dk = torch.empty_like(k) if dk is None else _dev(dk, "dk", q.dtype)
    dv = torch.empty_like(v) if dv is None else _dev(dv, "dv", q.dtype)
    dt = _dtype_code(q)
    need = mha_bwd_workspace_size(B, H, Lq, D, dt)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    else:
        _dev(workspace, "workspace")
    wbytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().mha_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                         int(mask_kind), _ptr(kv_lengths), _ptr(dq), _ptr(dk), _ptr(dv),
                         B, H, Lq, Lk, D, scale, dt, _ptr(workspace), wbytes,
                         _stream(stream, q.get_device())), "mha_bwd")
    return dq, dk, dv


def prenorm_cross_attn_fwd(x_q, gamma, beta, eps, k, v, kv_lengths=None, out=None, scale=None,
                           stream=None):
    """Pre-LayerNorm cross-attention; x_q [B,Lq,H*D] bf16, gamma/beta fp32
    [H*D], k/v [B,H,Lk,D] bf16.  Returns `out` [B,Lq,H*D] bf16."""
    torch = _torch()
    _dev(x_q, "x_q", torch.bfloat16)
    _dev(gamma, "gamma", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(k, "k", torch.bfloat16)
    _dev(v, "v", torch.bfloat16)
    B, H, Lk, D = k.shape
    Lq = x_q.shape[1]
    if tuple(x_q.shape) != (B, Lq, H * D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("x_q must be [B,Lq,H*D] and v [B,H,Lk,D]")
    if gamma.numel() != H * D or beta.numel() != H * D:
        raise ValueError("gamma and beta must have H*D elements")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    if out is None:
        out = torch.empty_like(x_q)
    else:
        _dev(out, "out", torch.bfloat16)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().prenorm_cross_attn_fwd(_ptr(x_q), _ptr(gamma), _ptr(beta), float(eps), _ptr(k),
                                        _ptr(v), _ptr(kv_lengths), _ptr(out), B, H, Lq, Lk, D,
                                        scale, BF16, _stream(stream, x_q.get_device())),
           "prenorm_cross_attn_fwd")
    return out


def prenorm_cross_attn_residual_fwd(x_q, gamma, beta, eps, k, v, kv_lengths=None, out=None,
                                    scale=None, stream=None):
    """x_q + prenorm_cross_attn_fwd(x_q, ...), summed in fp32 and rounded once.
    Same arguments and layouts as prenorm_cross_attn_fwd; `out` must not
    overlap x_q."""
    torch = _torch()
    _dev(x_q, "x_q", torch.bfloat16)
    _dev(gamma, "gamma", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(k, "k", torch.bfloat16)
    _dev(v, "v", torch.bfloat16)
    B, H, Lk, D = k.shape
    Lq = x_q.shape[1]
    if tuple(x_q.shape) != (B, Lq, H * D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("x_q must be [B,Lq,H*D] and v [B,H,Lk,D]")
    if gamma.numel() != H * D or beta.numel() != H * D:
        raise ValueError("gamma and beta must have H*D elements")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    if out is None:
        out = torch.empty_like(x_q)
    else:
        _dev(out, "out", torch.bfloat16)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(lib().prenorm_cross_attn_residual_fwd(_ptr(x_q), _ptr(gamma), _ptr(beta), float(eps),
                                                 _ptr(k), _ptr(v), _ptr(kv_lengths), _ptr(out),
                                                 B, H, Lq, Lk, D, scale, BF16,
                                                 _stream(stream, x_q.get_device())),
           "prenorm_cross_attn_residual_fwd")
    return out


def mha_strerror(status):
    return lib().mha_strerror(int(status)).decode()


def device_status(clear=False):
    """Union of the kernels' device status words: bits 0-15 name bounded
    waits that expired, bit 16 a softmax row sum that was not positive and
    finite, bit 17 a non-finite output.  `clear` resets the words after
    reading them."""
    bits = ctypes.c_uint32(0)
    _check(lib().mha_device_status(ctypes.byref(bits), 1 if clear else 0), "mha_device_status")
    return bits.value


def test_set_device_status(unit, bits):
    """Test hook: OR `bits` into kernel unit `unit`'s device status word
    (0 bf16 forward, 1 fp32 tensor-core forward, 2 bf16 backward, 3 bf16
    decode)."""
    _check(lib().mha_test_set_device_status(int(unit), int(bits)), "mha_test_set_device_status")


def test_set_wait_limit_ns(ns):
    """Test hook: limit of every bounded device wait (0 restores 2 s)."""
    _check(lib().mha_test_set_wait_limit_ns(int(ns)), "mha_test_set_wait_limit_ns")


def selftest_umma(variant, kn, a, b, c, stream=None):
    """Diagnostic tcgen05 GEMM tile (see mha_selftest_umma in include/mha.h)."""
    _check(lib().mha_selftest_umma(int(variant), int(kn), _ptr(a), _ptr(b), _ptr(c),
                                   _stream(stream)), "mha_selftest_umma")
    return c


def set_bf16_grid(ctas):
    lib().mha_set_bf16_grid(int(ctas))


def plan_prenorm(B, H, Lq, Lk, D, grid, stats_given=False):
    """Test hook: the Pre-LN forward's launch plan for these sizes on `grid`
    CTAs (host logic; no device needed): dict with G (heads per chunk), n_hg,
    cs (CTAs per cluster), pre_chunks, grid, n_chunks."""
    out = (ctypes.c_int64 * 6)()
    _check(lib().mha_plan_prenorm(int(B), int(H), int(Lq), int(Lk), int(D), int(grid),
                                  1 if stats_given else 0, out), "mha_plan_prenorm")
    return dict(zip(("G", "n_hg", "cs", "pre_chunks", "grid", "n_chunks"), (int(v) for v in out)))


def set_bf16_decode(mode):
    """0 automatic (decode kernel for bf16 calls with Lq <= 8), 1 never."""
    lib().mha_set_bf16_decode(int(mode))


def set_bf16_decode_splits(splits):
    """Force the decode kernel's CTAs per (b, h) (1..8); 0 = automatic."""
    lib().mha_set_bf16_decode_splits(int(splits))


def set_bwd_kernel(which):
    """Backward kernels: 0 automatic (bf16 on the tensor cores), 1 CUDA cores."""
    lib().mha_set_bwd_kernel(int(which))


def set_pdl(on):
    """Test hook: programmatic dependent launch on (1, default) or off (0) for
    calls made from this thread."""
    lib().mha_set_pdl(1 if on else 0)


def set_f32_kernel(which):
    """0 automatic (tensor cores, 3xTF32, for D = 64), 1 tiled CUDA-core kernel
    only, 2 short-key-range CUDA-core kernel where it applies, 3 as 0."""
    lib().mha_set_f32_kernel(int(which))


def prenorm_cross_attn_fwd_noalloc(x_q, gamma, beta, eps, k, v, kv_lengths=None, out=None,
                                   scale=None, stream=None):
    """prenorm_cross_attn_fwd without any allocation by the library: for
    callers whose device memory is planned and owned elsewhere (e.g. a
    serving runtime that reserves all GPU memory for its own pools).  The
    row statistics use a fixed 2 MiB device array (B*Lq <= 262144); calls
    that overlap on the GPU share that array and race.  `out` should be
    passed in by such callers (it is created here only when omitted)."""
    torch = _torch()
    L = lib()
    if not getattr(L, "_noalloc_bound", False):
        P, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.prenorm_cross_attn_fwd_noalloc.argtypes = [P, P, P, f, P, P, P, P, i, i, i, i, i, f, i, P]
        L.prenorm_cross_attn_fwd_noalloc.restype = i
        L._noalloc_bound = True
    _dev(x_q, "x_q", torch.bfloat16)
    _dev(gamma, "gamma", torch.float32)
    _dev(beta, "beta", torch.float32)
    _dev(k, "k", torch.bfloat16)
    _dev(v, "v", torch.bfloat16)
    B, H, Lk, D = k.shape
    Lq = x_q.shape[1]
    if tuple(x_q.shape) != (B, Lq, H * D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("x_q must be [B,Lq,H*D] and v [B,H,Lk,D]")
    if kv_lengths is not None:
        _dev(kv_lengths, "kv_lengths", torch.int32)
    if out is None:
        out = torch.empty_like(x_q)
    else:
        _dev(out, "out", torch.bfloat16)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(L.prenorm_cross_attn_fwd_noalloc(_ptr(x_q), _ptr(gamma), _ptr(beta), float(eps),
                                            _ptr(k), _ptr(v), _ptr(kv_lengths), _ptr(out), B, H,
                                            Lq, Lk, D, scale, BF16, _stream(stream, x_q.get_device())),
           "prenorm_cross_attn_fwd_noalloc")
    return out
