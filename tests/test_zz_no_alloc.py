"""fa_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (code whose device memory belongs to a host framework's pool,
or latency-critical paths where cudaMalloc/cudaFree may synchronise the
device).  It must give what fa_bwd gives with a caller-allocated workspace,
call after call, since every call reuses the same fixed scratch array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import helpers as H
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from exact_io_aware_40_gb300 import build as fab, fa
    fab.build()
    return fa.load_library()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def noalloc_bwd(lib, case, o, L, causal):
    """Calls fa_bwd_noalloc directly through the C ABI."""
    import torch
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(L), _p(dq), _p(dk), _p(dv),
                            case.B, case.H, case.N, case.d, ctypes.c_float(case.scale),
                            int(causal), _p(case.kv_len_dev),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return dq, dk, dv


def test_noalloc_matches_fa_bwd_on_calls_in_a_row(lib):
    from exact_io_aware_40_gb300 import fa
    cases = [
        (H.Case(7001, 2, 4, 1000, 128), False),
        (H.Case(7002, 4, 8, 777, 64, kv_range=(300, 777)), True),
        (H.Case(7003, 1, 4, 600, 256), True),
    ]
    # the first shape again after the second: stale scratch must not leak in
    for case, causal in cases + cases[:1]:
        q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
        o, L = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale, kv_len=case.kv_len_dev)
        ref = fa.attention_bwd(q, k, v, o, do, L, causal=causal, scale=case.scale,
                               kv_len=case.kv_len_dev)
        got = noalloc_bwd(lib, case, o, L, causal)
        fa.fa_check_error()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            e = H.err_rel(H.to_f64(g), H.to_f64(r))
            assert e <= H.TOL_GRAD_REL, (name, case.N, causal, e)
        # the backward pass is deterministic: the gradients match bit for bit
        for g, r in zip(got, ref):
            np.testing.assert_array_equal(H.to_f64(g), H.to_f64(r))


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    import torch
    from exact_io_aware_40_gb300 import fa
    # 8 * 64 * 8200 = 4,198,400 rows of fp32 row terms: just over 16 MiB
    B, Hh, N, d = 8, 64, 8200, 64
    assert fa.fa_bwd_workspace_bytes(B, Hh, N, d) > 16 * 1024 * 1024
    x = torch.zeros(B, Hh, N, d, dtype=torch.bfloat16, device="cuda")
    L = torch.zeros(B, Hh, N, dtype=torch.float32, device="cuda")
    st = lib.fa_bwd_noalloc(_p(x), _p(x), _p(x), _p(x), _p(x), _p(L), _p(x), _p(x), _p(x),
                            B, Hh, N, d, ctypes.c_float(0.125), 0, _p(None),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fa.FA_ERR_UNSUPPORTED
    fa.fa_check_error()


def test_noalloc_matches_the_oracle(lib):
    # d = 256 with key padding, compared with the fp64 oracle directly
    from exact_io_aware_40_gb300 import fa
    case = H.Case(7004, 2, 2, 333, 256)
    case.set_kv_len([333, 150])
    q, k, v = (case.dev[n] for n in ("Q", "K", "V"))
    o, L = fa.attention_fwd(q, k, v, causal=True, scale=case.scale, kv_len=case.kv_len_dev)
    got = noalloc_bwd(lib, case, o, L, True)
    fa.fa_check_error()
    ref = oracle.attn_bwd(case.f64["Q"], case.f64["K"], case.f64["V"], case.f64["dO"],
                          case.scale, True, kv_len=case.kv_len)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        e = H.err_rel(H.to_f64(g), r)
        assert e <= H.TOL_GRAD_REL, (name, e)


def test_noalloc_refuses_an_unsupported_head_dim(lib):
    import torch
    from exact_io_aware_40_gb300 import fa
    x = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device="cuda")
    L = torch.zeros(1, 1, 64, dtype=torch.float32, device="cuda")
    st = lib.fa_bwd_noalloc(_p(x), _p(x), _p(x), _p(x), _p(x), _p(L), _p(x), _p(x), _p(x),
                            1, 1, 64, 96, ctypes.c_float(0.1), 0, _p(None),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fa.FA_ERR_UNSUPPORTED
    fa.fa_check_error()
