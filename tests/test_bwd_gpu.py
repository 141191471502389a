"""GPU parity of the backward pass (pre, main and post kernels) against the
fp64 oracle, through the C ABI.  The GPU's own O and L feed its backward (as in
training); the oracle recomputes everything from Q, K, V, dO alone."""
import numpy as np
import pytest

import helpers as H
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


def run_bwd(case, causal):
    from exact_io_aware_40_gb300 import fa
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    o, L = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale, kv_len=case.kv_len_dev)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, L, causal=causal, scale=case.scale,
                                  kv_len=case.kv_len_dev)
    fa.fa_check_error()
    return H.to_f64(dq), H.to_f64(dk), H.to_f64(dv)


def check_full(case, causal):
    got = run_bwd(case, causal)
    ref = oracle.attn_bwd(case.f64["Q"], case.f64["K"], case.f64["V"], case.f64["dO"],
                          case.scale, causal, kv_len=case.kv_len)
    errs = [H.err_rel(g, r) for g, r in zip(got, ref)]
    H.report("bwd", case, causal, err_dQ=errs[0], err_dK=errs[1], err_dV=errs[2])
    for name, e in zip(("dQ", "dK", "dV"), errs):
        assert e <= H.TOL_GRAD_REL, (name, e)
    return errs


def check_sampled(case, causal, heads, rows, cols):
    dq, dk, dv = run_bwd(case, causal)
    worst = {"dQ": 0.0, "dK": 0.0, "dV": 0.0}
    for (b, h) in heads:
        qh, kh, vh, doh = (case.f64[n][b, h] for n in ("Q", "K", "V", "dO"))
        ln = case.length(b)
        dq_ref = oracle.bwd_dq_rows(qh, kh, vh, doh, case.scale, causal, ln, rows)
        dk_ref, dv_ref = oracle.bwd_dkdv_cols(qh, kh, vh, doh, case.scale, causal, ln, cols)
        # relative-to-max-norm, the max taken over the sampled reference values
        for name, g, r in (("dQ", dq[b, h, rows], dq_ref), ("dK", dk[b, h, cols], dk_ref),
                           ("dV", dv[b, h, cols], dv_ref)):
            e = H.err_rel(g, r)
            worst[name] = max(worst[name], e)
            assert e <= H.TOL_GRAD_REL, (name, b, h, e)
    H.report("bwd_sampled", case, causal, err_dQ=worst["dQ"], err_dK=worst["dK"],
             err_dV=worst["dV"])


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    check_full(H.Case(1000, 1, 2, 128, 64), causal)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 2, 63, 127, 129, 200, 383])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(d, N, causal):
    check_full(H.Case(4000 + N, 2, 2, N, d), causal)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_edges(d, causal):
    case = H.Case(5000, 4, 2, 300, d)
    case.set_kv_len([0, 1, 129, 300])
    dq, dk, dv = run_bwd(case, causal)
    ref = oracle.attn_bwd(case.f64["Q"], case.f64["K"], case.f64["V"], case.f64["dO"],
                          case.scale, causal, kv_len=case.kv_len)
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)
    # padded keys get exactly zero gradient
    assert np.all(dk[1, :, 1:] == 0) and np.all(dv[1, :, 1:] == 0)
    assert np.all(dk[2, :, 129:] == 0) and np.all(dv[2, :, 129:] == 0)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert H.err_rel(g, r) <= H.TOL_GRAD_REL, name


def test_bert_large_shaped():
    check_full(H.Case(1001, 16, 16, 512, 64, kv_range=(256, 512)), False)


def test_gpt2_shaped():
    check_full(H.Case(1002, 8, 12, 1024, 64), True)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(causal):
    case = H.Case(1003, 1, 16, 16384, 128)
    rows = np.array([0, 1, 127, 128, 5000, 8191, 8192, 16255, 16256, 16383])
    check_sampled(case, causal, [(0, 3)], rows, rows)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_sampled(d, N, causal):
    B, Hh = 16384 // N, 2048 // d
    case = H.Case(1004, B, Hh, N, d)
    # The tolerance is relative to the tensor's max norm; the sampled rows
    # include the early ones, where causal rows (few keys) have the largest
    # gradients, so the max over the sample stands for the tensor's.
    rows = np.unique(np.array([0, 1, 2, 3, 64, 127, 128, 129, N // 2, N - 129, N - 128, N - 1]))
    check_sampled(case, causal, [(0, 0), (B // 2, Hh // 2), (B - 1, Hh - 1)], rows, rows)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_whole_head(causal):
    """Every element of O, L, dQ, dK and dV of one head of the benchmark
    workload (B=1, H=16, N=16384, d=128, all 16 heads launched together, as
    the benchmark times them) against the oracle run on that head's slice.
    The oracle deals the head's row panels out to the host threads: about
    0.5 TFLOP of fp64 work non-causal, some 15-40 s on 16 host cores."""
    from exact_io_aware_40_gb300 import fa
    case = H.Case(1003, 1, 16, 16384, 128)
    q, k, v, do = (case.dev[n] for n in ("Q", "K", "V", "dO"))
    o, L = fa.attention_fwd(q, k, v, causal=causal, scale=case.scale)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, L, causal=causal, scale=case.scale)
    fa.fa_check_error()
    h = 5
    sl = {n: case.f64[n][:, h:h + 1] for n in ("Q", "K", "V", "dO")}
    o_ref, L_ref = oracle.attn_fwd(sl["Q"], sl["K"], sl["V"], case.scale, causal)
    g_ref = oracle.attn_bwd(sl["Q"], sl["K"], sl["V"], sl["dO"], case.scale, causal)
    o_h, L_h = H.to_f64(o[:, h:h + 1]), H.to_f64(L[:, h:h + 1])
    assert H.err_o(o_h, o_ref) <= H.TOL_O_ABS, ("O", H.err_o(o_h, o_ref))
    assert H.err_l(L_h, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L_h, L_ref))
    errs = [H.err_rel(H.to_f64(g[:, h:h + 1]), r) for g, r in zip((dq, dk, dv), g_ref)]
    H.report("whole_head", case, causal, err_O=H.err_o(o_h, o_ref), err_L=H.err_l(L_h, L_ref),
             err_dQ=errs[0], err_dK=errs[1], err_dV=errs[2])
    for name, e in zip(("dQ", "dK", "dV"), errs):
        assert e <= H.TOL_GRAD_REL, (name, e)


@pytest.mark.parametrize("factor", [0.5, 2.0])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_other_scales(factor, d, causal):
    # scales other than 1/sqrt(d) on the usual iid inputs
    check_full(H.Case(4100 + d, 2, 2, 700, d, scale=factor / np.sqrt(d)), causal)


def test_deterministic():
    # no atomics anywhere in the backward pass: identical inputs give identical bits
    case = H.Case(1006, 2, 4, 700, 128)
    a = run_bwd(case, True)
    b = run_bwd(case, True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
