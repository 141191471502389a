"""GPU parity of the sliding-window and block-sparse mask terms (forward and
backward, through fa_fwd_masked / fa_bwd_masked) against the fp64 oracle.

Whole-tensor comparisons at sizes the oracle finishes in seconds, spanning
several 128-wide tiles and ragged tails; sampled rows and columns at 16K
tokens; the degenerate cases (window 0, a window wider than the sequence,
query blocks that keep no key block, an all-ones block mask) and bitwise
agreement with the unmasked entry points where the masks change nothing.
"""
import numpy as np
import pytest

import helpers as H
from exact_io_aware_40_gb300 import inputs
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from exact_io_aware_40_gb300 import build as fab, fa
    fab.build()
    return fa.load_library()


def dev_mask(bm):
    import torch
    return None if bm is None else torch.from_numpy(np.ascontiguousarray(bm)).to("cuda:0")


def run(case, causal, window, bm):
    from exact_io_aware_40_gb300 import fa
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    m = dev_mask(bm)
    o, L = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale, kv_len=case.kv_len_dev,
                            window=window, block_mask=m)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, L, causal=causal, scale=case.scale,
                                  kv_len=case.kv_len_dev, window=window, block_mask=m)
    fa.fa_check_error()
    return [H.to_f64(t) for t in (o, L, dq, dk, dv)]


def check_full(case, causal, window, bm):
    o, L, dq, dk, dv = run(case, causal, window, bm)
    args = (case.f64["Q"], case.f64["K"], case.f64["V"])
    kw = dict(kv_len=case.kv_len, window=window, block_mask=bm, block=128)
    o_ref, L_ref = oracle.attn_fwd(*args, case.scale, causal, **kw)
    g_ref = oracle.attn_bwd(*args, case.f64["dO"], case.scale, causal, **kw)
    assert H.err_o(o, o_ref) <= H.TOL_O_ABS, ("O", H.err_o(o, o_ref))
    assert H.err_l(L, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L, L_ref))
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        e = H.err_rel(g, r)
        assert e <= H.TOL_GRAD_REL, (name, e)
    # rows that keep no key: O = 0, L = -inf, dQ = 0
    empty = np.isneginf(L_ref)
    assert np.all(o[empty] == 0.0) and np.all(dq[empty] == 0.0)
    return o, L


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,window", [(200, 0), (200, 1), (383, 127), (383, 128), (700, 300),
                                      (700, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_sliding_window(d, N, window, causal):
    check_full(H.Case(1100 + N, 1, 2, N, d), causal, window, None)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_sliding_window_with_key_padding(d):
    case = H.Case(1201, 3, 2, 640, d)
    case.set_kv_len([640, 300, 37])
    check_full(case, True, 200, None)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,density,diagonal", [(300, 0.5, True), (1000, 0.3, True),
                                                (1000, 0.4, False), (1153, 0.6, False)])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse(d, N, density, diagonal, causal):
    nb = (N + 127) // 128
    bm = inputs.block_mask(1300 + N, nb, density, diagonal)
    check_full(H.Case(1300 + N, 2, 2, N, d), causal, -1, bm)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_block_sparse_empty_rows_window_and_padding(d):
    N = 900
    nb = (N + 127) // 128
    bm = inputs.block_mask(1401, nb, 0.5, True)
    bm[2, :] = 0          # query block 2 keeps nothing: empty rows
    bm[:, 5] = 0          # key block 5 is never reached: dK = dV = 0 there
    case = H.Case(1401, 2, 2, N, d)
    case.set_kv_len([900, 500])
    check_full(case, True, 400, bm)
    check_full(case, False, -1, bm)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_masks_that_change_nothing_change_nothing(d, causal):
    # An all-ones block mask, and a window wider than the sequence (with the
    # causal term it implies), keep every pair.  The forward then runs the
    # kernel instantiation with the window and block-mask terms (same tiles,
    # same order; held to a few bf16 ulps, not bitwise, since the two are
    # compiled separately); the backward kernels visit the same tiles with
    # the same element masks: given the same O and L they agree bit for bit.
    from exact_io_aware_40_gb300 import fa
    N = 777
    case = H.Case(1501, 1, 3, N, d)
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    o0, L0 = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale)
    g0 = fa.attention_bwd(q, k, v, o0, do, L0, causal=causal, scale=case.scale)
    ones = dev_mask(np.ones(((N + 127) // 128,) * 2, np.uint8))
    variants = [dict(block_mask=ones, causal=causal)]
    if causal:
        variants.append(dict(window=N, causal=False))
    for kw in variants:
        o1, L1 = fa.attention_fwd(q, k, v, scale=case.scale, **kw)
        g1 = fa.attention_bwd(q, k, v, o0, do, L0, scale=case.scale, **kw)
        fa.fa_check_error()
        a0, a1 = H.to_f64(o0), H.to_f64(o1)
        assert float(np.abs(a0 - a1).max()) <= 2.0 ** -6 * max(1.0, float(np.abs(a0).max()))
        assert float(np.abs(H.to_f64(L0) - H.to_f64(L1)).max()) <= 1e-5
        assert all(bool((x == y).all()) for x, y in zip(g0, g1))


@pytest.mark.parametrize("kind", ["window", "block_sparse"])
def test_long_sequence_sampled(kind):
    # B=1, H=4, N=16384, d=128: sampled rows (O, L, dQ) and key columns (dK, dV)
    N, d = 16384, 128
    case = H.Case(1003, 1, 4, N, d)
    nb = N // 128
    if kind == "window":
        window, bm, causal = 1024, None, True
    else:
        # local band of 3 blocks plus 4 global key blocks, a common sparse layout
        i = np.arange(nb)[:, None]
        j = np.arange(nb)[None, :]
        bm = ((np.abs(i - j) <= 1) | (j < 4)).astype(np.uint8)
        window, causal = -1, False
    o, L, dq, dk, dv = run(case, causal, window, bm)
    rows = np.array([0, 1, 127, 128, 1000, 5000, 9999, 16383])
    cols = np.array([0, 3, 511, 512, 4097, 12000, 16383])
    kw = dict(window=window, block_mask=bm, block=128)
    for h in (0, 3):
        qh, kh, vh, doh = (case.f64[n][0, h] for n in ("Q", "K", "V", "dO"))
        o_ref, L_ref = oracle.fwd_rows(qh, kh, vh, case.scale, causal, N, rows, **kw)
        assert H.err_o(o[0, h, rows], o_ref) <= H.TOL_O_ABS
        assert H.err_l(L[0, h, rows], L_ref) <= H.TOL_L_ABS
        dq_ref = oracle.bwd_dq_rows(qh, kh, vh, doh, case.scale, causal, N, rows, **kw)
        dk_ref, dv_ref = oracle.bwd_dkdv_cols(qh, kh, vh, doh, case.scale, causal, N, cols, **kw)
        for name, g, r in (("dQ", dq[0, h, rows], dq_ref), ("dK", dk[0, h, cols], dk_ref),
                           ("dV", dv[0, h, cols], dv_ref)):
            assert H.err_rel(g, r) <= H.TOL_GRAD_REL, (name, h, H.err_rel(g, r))
