"""ctypes binding of the C ABI in include/fa.h (libfa_sm103.so).

Argument marshalling only: every step of attention runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); the library is loaded from this package directory and is never
replaced by another implementation -- if it is missing or cannot load, calls
raise.
"""
import ctypes
import math
import os

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_sm103.so")
_lib = None


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s returned %s" % (where, status_string(status)))


def load_library():
    """Load libfa_sm103.so (built by build.py); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("%s is not built; run exact_io_aware_40_gb300/build.py "
                           "(or __graft_entry__.build())" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_kvlen.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp]
    lib.fa_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, vp]
    u64 = ctypes.c_uint64
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, f, u64, vp]
    lib.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i,
                                   vp, f, u64, vp, sz, vp]
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_bytes.restype = sz
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, f, f, i, vp, vp, sz, vp]
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.fa_bwd_masked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp,
                                  vp, sz, vp]
    lib.fa_bwd_prepare.argtypes = [vp, vp, i, i, i, i, vp, sz, vp]
    lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp]
    lib.fa_bwd_noalloc.restype = ctypes.c_int
    lib.fa_selftest_stalled_wait.argtypes = [ctypes.c_uint64, vp]
    lib.fa_check_error.argtypes = [vp]
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    for fn in ("fa_fwd", "fa_fwd_kvlen", "fa_fwd_masked", "fa_bwd", "fa_bwd_masked",
               "fa_fwd_dropout", "fa_bwd_dropout", "fa_fwd_fp8",
               "fa_bwd_prepare", "fa_bwd_dkdv",
               "fa_bwd_dq", "fa_check_error", "fa_selftest_stalled_wait"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status):
    return load_library().fa_status_string(int(status)).decode()


fa_status_string = status_string


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, ref):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(ref.device).cuda_stream)


def _check(status, where):
    if status != FA_OK:
        raise FAError(status, where)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    return tuple(int(x) for x in q.shape)


def _expect(t, name, dtype, shape):
    if t is None:
        raise ValueError("%s is required" % name)
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != shape:
        raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s" % (name, dtype, shape))


# ------------------------------------------------------------------ raw ABI

def fa_fwd(q, k, v, o, L, scale, causal, stream=None):
    """fa_fwd on torch tensors (bf16 [B,H,N,d] q/k/v/o, fp32 [B,H,N] L)."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d,
                                 float(scale), int(bool(causal)), _stream(stream, q)), "fa_fwd")


def fa_fwd_kvlen(q, k, v, o, L, scale, causal, kv_len, stream=None):
    """fa_fwd_kvlen on torch tensors; kv_len is a CUDA int32 [B] tensor or None."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_fwd_kvlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d,
                                       float(scale), int(bool(causal)), _ptr(kv_len),
                                       _stream(stream, q)), "fa_fwd_kvlen")


def fa_fwd_masked(q, k, v, o, L, scale, causal, kv_len, window, block_mask, stream=None):
    """fa_fwd_masked; window is an int (-1: none), block_mask a CUDA uint8
    [ceil(N/128), ceil(N/128)] tensor or None."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d,
                                        float(scale), int(bool(causal)), _ptr(kv_len), int(window),
                                        _ptr(block_mask), _stream(stream, q)), "fa_fwd_masked")


def fa_fwd_dropout(q, k, v, o, L, scale, causal, kv_len, window, block_mask, dropout_p, seed,
                   stream=None):
    """fa_fwd_dropout: the masked forward with dropout (p in [0, 1), 64-bit seed)."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d,
                                         float(scale), int(bool(causal)), _ptr(kv_len),
                                         int(window), _ptr(block_mask), float(dropout_p),
                                         int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream, q)),
           "fa_fwd_dropout")


def fa_bwd_dropout(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, window, block_mask,
                   dropout_p, seed, workspace, stream=None):
    """fa_bwd_dropout on torch tensors (same masks, p and seed as the forward)."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                         _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                         int(bool(causal)), _ptr(kv_len), int(window),
                                         _ptr(block_mask), float(dropout_p),
                                         int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(workspace),
                                         workspace.numel(), _stream(stream, q)), "fa_bwd_dropout")


def fa_fwd_fp8_workspace_bytes(B, H, N, d):
    return int(load_library().fa_fwd_fp8_workspace_bytes(B, H, N, d))


def fa_fwd_fp8(q8, k8, v8, o, L, scale, descale_q, descale_k, descale_v, causal, kv_len,
               workspace, stream=None):
    """fa_fwd_fp8: q8/k8/v8 are CUDA uint8 tensors of e4m3 codes [B,H,N,d]; O bf16."""
    B, H, N, d = _shape(q8)
    _check(load_library().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(o), _ptr(L), B, H, N, d,
                                     float(scale), float(descale_q), float(descale_k),
                                     float(descale_v), int(bool(causal)), _ptr(kv_len),
                                     _ptr(workspace), workspace.numel(), _stream(stream, q8)),
           "fa_fwd_fp8")


def fa_bwd_workspace_bytes(B, H, N, d):
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, workspace, stream=None):
    """fa_bwd on torch tensors; workspace is a CUDA byte tensor."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L), _ptr(dq),
                                 _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                 _ptr(kv_len), _ptr(workspace), workspace.numel(),
                                 _stream(stream, q)), "fa_bwd")


def fa_bwd_masked(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, window, block_mask,
                  workspace, stream=None):
    """fa_bwd_masked on torch tensors (masks as in fa_fwd_masked)."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                        _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                        int(bool(causal)), _ptr(kv_len), int(window),
                                        _ptr(block_mask), _ptr(workspace), workspace.numel(),
                                        _stream(stream, q)), "fa_bwd_masked")


def fa_bwd_prepare(o, do, workspace, stream=None):
    """fa_bwd_prepare: D = rowsum(dO * O) into the workspace."""
    B, H, N, d = _shape(o)
    _check(load_library().fa_bwd_prepare(_ptr(o), _ptr(do), B, H, N, d, _ptr(workspace),
                                         workspace.numel(), _stream(stream, o)), "fa_bwd_prepare")


def fa_bwd_dkdv(q, k, v, do, L, dk, dv, scale, causal, kv_len, workspace, stream=None):
    """fa_bwd_dkdv: dK and dV from a prepared workspace."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(L), _ptr(dk),
                                      _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                      _ptr(kv_len), _ptr(workspace), workspace.numel(),
                                      _stream(stream, q)), "fa_bwd_dkdv")


def fa_bwd_dq(q, k, v, do, L, dq, scale, causal, kv_len, workspace, stream=None):
    """fa_bwd_dq: dQ from a prepared workspace."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(L), _ptr(dq),
                                    B, H, N, d, float(scale), int(bool(causal)), _ptr(kv_len),
                                    _ptr(workspace), workspace.numel(), _stream(stream, q)),
           "fa_bwd_dq")


def fa_bwd_noalloc(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, stream=None):
    """fa_bwd_noalloc: the backward pass with the library's fixed scratch as the
    workspace, for callers that cannot allocate device memory (see fa.h)."""
    B, H, N, d = _shape(q)
    _check(load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(L),
                                         _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                         int(bool(causal)), _ptr(kv_len), _stream(stream, q)),
           "fa_bwd_noalloc")


def fa_selftest_stalled_wait(limit_ns, stream=None):
    """Enqueue the stalled-wait self test; fa_check_error then reports FA_ERR_TIMEOUT."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(load_library().fa_selftest_stalled_wait(int(limit_ns), ctypes.c_void_p(int(stream))),
           "fa_selftest_stalled_wait")


def fa_check_error(stream=None, device=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device).cuda_stream
    _check(load_library().fa_check_error(ctypes.c_void_p(int(stream))), "fa_check_error")


# ------------------------------------------------------------------ convenience

MASK_BLOCK = 128  # block size of block_mask (FA_MASK_BLOCK)


def _same_device(*ts):
    devs = {t.device for t in ts if t is not None}
    if len(devs) > 1:
        raise ValueError("all tensors must be on one CUDA device, got %s" % sorted(map(str, devs)))


def _expect_mask(block_mask, N):
    import torch
    if block_mask is not None:
        nb = (N + MASK_BLOCK - 1) // MASK_BLOCK
        _expect(block_mask, "block_mask", torch.uint8, (nb, nb))


def attention_fwd(q, k, v, causal=False, scale=None, kv_len=None, out=None, lse=None, stream=None,
                  window=-1, block_mask=None, dropout_p=0.0, seed=0):
    """Exact attention forward.  Returns (O bf16 [B,H,N,d], L fp32 [B,H,N]).

    window (int, -1 = none) and block_mask (CUDA uint8 [ceil(N/128)]^2 or None)
    select the sliding-window and block-sparse mask terms of fa_fwd_masked."""
    import torch
    B, H, N, d = _shape(q)
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _expect(t, nm, torch.bfloat16, (B, H, N, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _expect(out, "out", torch.bfloat16, (B, H, N, d))
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _expect(lse, "lse", torch.float32, (B, H, N))
    if kv_len is not None:
        _expect(kv_len, "kv_len", torch.int32, (B,))
    _same_device(q, k, v, out, lse, kv_len, block_mask)
    with torch.cuda.device(q.device):
        if dropout_p > 0.0:
            _expect_mask(block_mask, N)
            fa_fwd_dropout(q, k, v, out, lse, scale, causal, kv_len, window, block_mask,
                           dropout_p, seed, stream)
        elif window >= 0 or block_mask is not None:
            _expect_mask(block_mask, N)
            fa_fwd_masked(q, k, v, out, lse, scale, causal, kv_len, window, block_mask, stream)
        else:
            fa_fwd_kvlen(q, k, v, out, lse, scale, causal, kv_len, stream)
    return out, lse


def attention_bwd(q, k, v, o, do, L, causal=False, scale=None, kv_len=None, workspace=None,
                  stream=None, window=-1, block_mask=None, dropout_p=0.0, seed=0):
    """Exact attention backward.  Returns (dQ, dK, dV), bf16 [B,H,N,d]."""
    import torch
    B, H, N, d = _shape(q)
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _expect(t, nm, torch.bfloat16, (B, H, N, d))
    _expect(L, "L", torch.float32, (B, H, N))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if kv_len is not None:
        _expect(kv_len, "kv_len", torch.int32, (B,))
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _expect(workspace, "workspace", torch.uint8, (workspace.numel(),))
    _same_device(q, k, v, o, do, L, kv_len, block_mask, workspace)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with torch.cuda.device(q.device):
        if dropout_p > 0.0:
            _expect_mask(block_mask, N)
            fa_bwd_dropout(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, window,
                           block_mask, dropout_p, seed, workspace, stream)
        elif window >= 0 or block_mask is not None:
            _expect_mask(block_mask, N)
            fa_bwd_masked(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, window,
                          block_mask, workspace, stream)
        else:
            fa_bwd(q, k, v, o, do, L, dq, dk, dv, scale, causal, kv_len, workspace, stream)
    return dq, dk, dv


# ------------------------------------------------------------------ autograd

_FLASH_FN = None


def _flash_function():
    """The torch.autograd.Function over attention_fwd / attention_bwd (built on
    first use so that importing this module does not import torch)."""
    global _FLASH_FN
    if _FLASH_FN is None:
        import torch

        class FlashAttnFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale, kv_len, window, block_mask, dropout_p, seed):
                o, L = attention_fwd(q, k, v, causal=causal, scale=scale, kv_len=kv_len,
                                     window=window, block_mask=block_mask,
                                     dropout_p=dropout_p, seed=seed)
                ctx.save_for_backward(q, k, v, o, L)
                ctx.rest = (causal, scale, kv_len, window, block_mask, dropout_p, seed)
                ctx.mark_non_differentiable(L)
                return o, L

            @staticmethod
            def backward(ctx, do, _dL):
                q, k, v, o, L = ctx.saved_tensors
                causal, scale, kv_len, window, block_mask, dropout_p, seed = ctx.rest
                dq, dk, dv = attention_bwd(q, k, v, o, do.contiguous(), L, causal=causal,
                                           scale=scale, kv_len=kv_len, window=window,
                                           block_mask=block_mask, dropout_p=dropout_p, seed=seed)
                return dq, dk, dv, None, None, None, None, None, None, None

        _FLASH_FN = FlashAttnFunction
    return _FLASH_FN


def flash_attn_func(q, k, v, causal=False, softmax_scale=None, kv_len=None, window=-1,
                    block_mask=None, dropout_p=0.0, seed=0, return_lse=False):
    """Exact attention as a differentiable op: O = softmax(scale * Q K^T + mask) V.

    The drop-in form of the method's interface (bxzpzcl.cn article, section
    "5分钟快速部署指南", basic usage example: Q, K, V and a causal flag in, the
    attention output out) with torch autograd: the backward runs
    attention_bwd, recomputing P from the saved logsumexp L.  Tensors are
    contiguous bf16 CUDA [B, H, N, d] (heads before tokens); softmax_scale
    defaults to 1/sqrt(d); the mask and dropout arguments are those of
    attention_fwd.  Returns O, or (O, L) with return_lse (L is not
    differentiable)."""
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    o, L = _flash_function().apply(q, k, v, bool(causal), scale, kv_len, int(window), block_mask,
                                   float(dropout_p), int(seed))
    return (o, L) if return_lse else o
