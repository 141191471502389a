"""GPU parity of dropout on the attention weights (fa_fwd_dropout /
fa_bwd_dropout) against the fp64 oracle, which draws the same decisions from
its own Philox4x32-10: the keep decisions themselves are compared exactly, L
and the gradients within the usual tolerances, O within the bound the bf16
arithmetic allows.

O with dropout is not a convex combination of V: the kept weights are scaled
by 1/q, so rows with few keys reach |O| >= 4, where the bf16 spacing is
2^-5 and even the correctly rounded exact value can miss a flat 1e-2.  The O
bound therefore adds the two bf16 roundings (the dropped weights fed to the
product, and O itself), each at most 2^-9 relative, with a factor two of
margin: |dO_ic| <= max(1e-2, 2^-8 (|O_ic| + sum_j Pd_ij |v_jc|)), the sum taken
by the oracle on |V|."""
import numpy as np
import pytest

import helpers as H
from exact_io_aware_40_gb300 import inputs
from oracle import oracle

pytestmark = pytest.mark.gpu

SEED = 0x5EED0123456789AB


@pytest.fixture(scope="module", autouse=True)
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from exact_io_aware_40_gb300 import build as fab, fa
    fab.build()
    return fa.load_library()


def p32(p):
    # the library takes p as a C float: give the oracle the same value
    return float(np.float32(p))


def run(case, causal, p, seed, window=-1, bm=None):
    import torch
    from exact_io_aware_40_gb300 import fa
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    m = None if bm is None else torch.from_numpy(np.ascontiguousarray(bm)).to("cuda:0")
    o, L = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale, kv_len=case.kv_len_dev,
                            window=window, block_mask=m, dropout_p=p, seed=seed)
    g = fa.attention_bwd(q, k, v, o, do, L, causal=causal, scale=case.scale,
                         kv_len=case.kv_len_dev, window=window, block_mask=m, dropout_p=p,
                         seed=seed)
    fa.fa_check_error()
    return [H.to_f64(t) for t in (o, L) + tuple(g)]


def o_bound(o_ref, a_ref):
    """Per-element O tolerance under dropout (module docstring)."""
    return np.maximum(H.TOL_O_ABS, 2.0 ** -8 * (np.abs(o_ref) + a_ref))


def check_o(o, o_ref, a_ref):
    excess = np.abs(o - o_ref) - o_bound(o_ref, a_ref)
    assert excess.max() <= 0.0, ("O", float(np.abs(o - o_ref).max()), float(excess.max()))


def check_full(case, causal, p, seed, window=-1, bm=None):
    o, L, dq, dk, dv = run(case, causal, p, seed, window, bm)
    args = (case.f64["Q"], case.f64["K"], case.f64["V"])
    kw = dict(kv_len=case.kv_len, window=window, block_mask=bm, dropout_p=p32(p), seed=seed)
    o_ref, L_ref = oracle.attn_fwd(*args, case.scale, causal, **kw)
    a_ref, _ = oracle.attn_fwd(args[0], args[1], np.abs(args[2]), case.scale, causal, **kw)
    g_ref = oracle.attn_bwd(*args, case.f64["dO"], case.scale, causal, **kw)
    check_o(o, o_ref, a_ref)
    assert H.err_l(L, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L, L_ref))
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        e = H.err_rel(g, r)
        assert e <= H.TOL_GRAD_REL, (name, e)


def test_keep_decisions_are_the_oracles():
    # Q = 0 gives uniform weights 1/64 over the 64 keys; V = identity makes
    # O_ij = P_ij Z_ij / q, so the nonzero pattern of O is the keep pattern.
    import torch
    from exact_io_aware_40_gb300 import fa
    B, Hh, N, d, p = 2, 3, 64, 64, 0.3
    q = torch.zeros(B, Hh, N, d, dtype=torch.bfloat16, device="cuda:0")
    k = torch.randn(B, Hh, N, d, device="cuda:0").to(torch.bfloat16)
    v = torch.eye(N, dtype=torch.bfloat16, device="cuda:0").expand(B, Hh, N, d).contiguous()
    for seed in (0, 1, SEED):
        o, _ = fa.attention_fwd(q, k, v, dropout_p=p, seed=seed)
        fa.fa_check_error()
        got = (o.float() != 0).cpu().numpy()
        for b in range(B):
            for h in range(Hh):
                ref = oracle.dropout_mult(b, h, N, p32(p), seed) > 0
                assert np.array_equal(got[b, h], ref), (seed, b, h)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,p", [(200, 0.1), (383, 0.5), (700, 0.25)])
@pytest.mark.parametrize("causal", [False, True])
def test_dropout_parity(d, N, p, causal):
    check_full(H.Case(1600 + N, 2, 2, N, d), causal, p, SEED + N)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_dropout_with_key_padding_window_and_block_mask(d):
    N = 900
    case = H.Case(1701, 2, 2, N, d)
    case.set_kv_len([900, 611])
    bm = inputs.block_mask(1701, (N + 127) // 128, 0.6, True)
    check_full(case, True, 0.2, 99, window=500)
    check_full(case, False, 0.2, 99, bm=bm)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_zero_probability_is_the_plain_kernel_bitwise(d):
    import torch
    from exact_io_aware_40_gb300 import fa
    case = H.Case(1801, 1, 2, 500, d)
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    o0, L0 = fa.attention_fwd(q, k, v, causal=True, scale=case.scale)
    g0 = fa.attention_bwd(q, k, v, o0, do, L0, causal=True, scale=case.scale)
    o1, L1 = torch.empty_like(o0), torch.empty_like(L0)
    fa.fa_fwd_dropout(q, k, v, o1, L1, case.scale, True, None, -1, None, 0.0, 123)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 2, 500, d), dtype=torch.uint8, device="cuda:0")
    g1 = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd_dropout(q, k, v, o1, do, L1, *g1, case.scale, True, None, -1, None, 0.0, 123, ws)
    fa.fa_check_error()
    assert bool((o0 == o1).all()) and bool((L0 == L1).all())
    assert all(bool((a == b).all()) for a, b in zip(g0, g1))


def test_long_sequence_sampled_with_dropout():
    N, d, p, seed = 16384, 128, 0.1, 42
    case = H.Case(1003, 1, 2, N, d)
    o, L, dq, dk, dv = run(case, True, p, seed)
    rows = np.array([0, 1, 127, 128, 5000, 16383])
    cols = np.array([0, 3, 512, 9000, 16383])
    kw = dict(dropout_p=p32(p), seed=seed)
    for h in (0, 1):
        qh, kh, vh, doh = (case.f64[n][0, h] for n in ("Q", "K", "V", "dO"))
        o_ref, L_ref = oracle.fwd_rows(qh, kh, vh, case.scale, True, N, rows, b=0, h=h, **kw)
        a_ref, _ = oracle.fwd_rows(qh, kh, np.abs(vh), case.scale, True, N, rows, b=0, h=h, **kw)
        check_o(o[0, h, rows], o_ref, a_ref)
        assert H.err_l(L[0, h, rows], L_ref) <= H.TOL_L_ABS
        dq_ref = oracle.bwd_dq_rows(qh, kh, vh, doh, case.scale, True, N, rows, b=0, h=h, **kw)
        dk_ref, dv_ref = oracle.bwd_dkdv_cols(qh, kh, vh, doh, case.scale, True, N, cols, b=0,
                                              h=h, **kw)
        for name, g, r in (("dQ", dq[0, h, rows], dq_ref), ("dK", dk[0, h, cols], dk_ref),
                           ("dV", dv[0, h, cols], dv_ref)):
            assert H.err_rel(g, r) <= H.TOL_GRAD_REL, (name, h, H.err_rel(g, r))
