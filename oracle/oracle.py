"""ctypes access to the fp64 CPU oracle (``attn_oracle.c``) -- TEST INFRASTRUCTURE.

The oracle is the plain definition of attention with S and P materialised,
computed in fp64 on the host (see the header of ``attn_oracle.c`` for the
formulas and the page sections they follow).  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may use it.

Inputs are numpy float64 arrays, contiguous ``[B, H, N, d]``; bf16 inputs are
widened exactly by the caller before they reach this module.

Mask arguments shared by every function: ``causal``; ``kv_len`` (or the
per-head ``length``); ``window`` (``w >= 0`` keeps only keys ``i - w <= j <=
i``; ``-1`` for none); ``block_mask`` (uint8 ``[ceil(N/block), ceil(N/block)]``
over (query block, key block) pairs, 0 = left out; ``None`` for none).
Dropout: ``dropout_p`` in [0, 1) and a 64-bit ``seed`` (Philox4x32-10 keyed
decisions, see attn_oracle.c); the per-head entry points also take the head's
batch and head index ``b``, ``h`` (they are part of the generator's counter).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile attn_oracle.c into liboracle.so (plain gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i, d = ctypes.c_int, ctypes.c_double
        bp = ctypes.POINTER(ctypes.c_ubyte)
        up = ctypes.POINTER(ctypes.c_uint)
        u64 = ctypes.c_ulonglong
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, i, i, i, i, d, i, ip, i, bp, i, d, u64,
                                        dp, dp, i]
        lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, i, i, i, i, d, i, ip, i, bp, i, d, u64,
                                        dp, dp, dp, i]
        lib.oracle_fwd_rows.argtypes = [dp, dp, dp, i, i, d, i, i, i, bp, i, d, u64, i, i, i, ip,
                                        dp, dp]
        lib.oracle_bwd_dq_rows.argtypes = [dp, dp, dp, dp, i, i, d, i, i, i, bp, i, d, u64, i, i,
                                           i, ip, dp]
        lib.oracle_bwd_dkdv_cols.argtypes = [dp, dp, dp, dp, i, i, d, i, i, i, bp, i, d, u64, i,
                                             i, i, ip, dp, dp, i]
        lib.oracle_philox4x32_10.argtypes = [up, up, up]
        lib.oracle_dropout_mult.argtypes = [i, i, i, d, u64, dp]
        for f in ("oracle_attn_fwd", "oracle_attn_bwd", "oracle_fwd_rows",
                  "oracle_bwd_dq_rows", "oracle_bwd_dkdv_cols", "oracle_philox4x32_10",
                  "oracle_dropout_mult"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _mask(block_mask, N, block):
    """(keep-alive array, pointer) of a block mask, checked against N."""
    if block_mask is None:
        return None, None
    nb = (N + block - 1) // block
    m = np.ascontiguousarray(block_mask, dtype=np.uint8)
    if m.shape != (nb, nb):
        raise ValueError("block_mask must be [%d, %d] for N=%d, block=%d" % (nb, nb, N, block))
    return m, m.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def _check(rc, name):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (name, rc))


def philox4x32_10(ctr, key):
    """One Philox4x32-10 call: four 32-bit counter words, two key words."""
    lib = _load()
    c = (ctypes.c_uint * 4)(*[int(x) & 0xffffffff for x in ctr])
    k = (ctypes.c_uint * 2)(*[int(x) & 0xffffffff for x in key])
    o = (ctypes.c_uint * 4)()
    _check(lib.oracle_philox4x32_10(c, k, o), "philox4x32_10")
    return [int(x) for x in o]


def dropout_mult(b, h, N, dropout_p, seed):
    """[N, N] dropout multipliers Z_ij / q of head (b, h): 0 or 1/q."""
    lib = _load()
    out = np.empty((N, N), np.float64)
    _check(lib.oracle_dropout_mult(int(b), int(h), int(N), float(dropout_p), int(seed),
                                   _f64(out)[1]), "dropout_mult")
    return out


def attn_fwd(q, k, v, scale, causal=False, kv_len=None, nthreads=None, window=-1,
             block_mask=None, block=128, dropout_p=0.0, seed=0):
    """Standard attention forward.  Returns (O [B,H,N,d], L [B,H,N]) in fp64."""
    lib = _load()
    B, H, N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    o = np.empty((B, H, N, d), np.float64)
    L = np.empty((B, H, N), np.float64)
    if kv_len is not None:
        kv, kvp = _i32(kv_len)
    else:
        kv, kvp = None, None
    bm, bmp = _mask(block_mask, N, block)
    rc = lib.oracle_attn_fwd(qp, kp, vp, B, H, N, d, float(scale), int(bool(causal)), kvp,
                             int(window), bmp, int(block), float(dropout_p), int(seed),
                             _f64(o)[1], _f64(L)[1], int(nthreads or default_threads()))
    _check(rc, "attn_fwd")
    return o, L


def attn_bwd(q, k, v, dout, scale, causal=False, kv_len=None, nthreads=None, window=-1,
             block_mask=None, block=128, dropout_p=0.0, seed=0):
    """Gradients of standard attention.  Returns (dQ, dK, dV), fp64 [B,H,N,d]."""
    lib = _load()
    B, H, N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    dout, dop = _f64(dout)
    dq = np.empty((B, H, N, d), np.float64)
    dk = np.empty((B, H, N, d), np.float64)
    dv = np.empty((B, H, N, d), np.float64)
    if kv_len is not None:
        kv, kvp = _i32(kv_len)
    else:
        kv, kvp = None, None
    bm, bmp = _mask(block_mask, N, block)
    rc = lib.oracle_attn_bwd(qp, kp, vp, dop, B, H, N, d, float(scale), int(bool(causal)), kvp,
                             int(window), bmp, int(block), float(dropout_p), int(seed),
                             _f64(dq)[1], _f64(dk)[1], _f64(dv)[1],
                             int(nthreads or default_threads()))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def fwd_rows(q, k, v, scale, causal, length, rows, window=-1, block_mask=None, block=128,
             dropout_p=0.0, seed=0, b=0, h=0):
    """O and L rows of ONE head (q, k, v are [N, d]) at the listed query rows."""
    lib = _load()
    N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    rows, rp = _i32(rows)
    o = np.empty((len(rows), d), np.float64)
    L = np.empty((len(rows),), np.float64)
    bm, bmp = _mask(block_mask, N, block)
    rc = lib.oracle_fwd_rows(qp, kp, vp, N, d, float(scale), int(bool(causal)), int(length),
                             int(window), bmp, int(block), float(dropout_p), int(seed), int(b),
                             int(h), len(rows), rp, _f64(o)[1], _f64(L)[1])
    _check(rc, "fwd_rows")
    return o, L


def bwd_dq_rows(q, k, v, dout, scale, causal, length, rows, window=-1, block_mask=None,
                block=128, dropout_p=0.0, seed=0, b=0, h=0):
    """dQ rows of ONE head at the listed query rows."""
    lib = _load()
    N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    dout, dop = _f64(dout)
    rows, rp = _i32(rows)
    dq = np.empty((len(rows), d), np.float64)
    bm, bmp = _mask(block_mask, N, block)
    rc = lib.oracle_bwd_dq_rows(qp, kp, vp, dop, N, d, float(scale), int(bool(causal)),
                                int(length), int(window), bmp, int(block), float(dropout_p),
                                int(seed), int(b), int(h), len(rows), rp, _f64(dq)[1])
    _check(rc, "bwd_dq_rows")
    return dq


def bwd_dkdv_cols(q, k, v, dout, scale, causal, length, cols, nthreads=None, window=-1,
                  block_mask=None, block=128, dropout_p=0.0, seed=0, b=0, h=0):
    """dK and dV rows of ONE head at the listed key indices."""
    lib = _load()
    N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    dout, dop = _f64(dout)
    cols, cp = _i32(cols)
    dk = np.empty((len(cols), d), np.float64)
    dv = np.empty((len(cols), d), np.float64)
    bm, bmp = _mask(block_mask, N, block)
    rc = lib.oracle_bwd_dkdv_cols(qp, kp, vp, dop, N, d, float(scale), int(bool(causal)),
                                  int(length), int(window), bmp, int(block), float(dropout_p),
                                  int(seed), int(b), int(h), len(cols), cp,
                                  _f64(dk)[1], _f64(dv)[1],
                                  int(nthreads or default_threads()))
    _check(rc, "bwd_dkdv_cols")
    return dk, dv
