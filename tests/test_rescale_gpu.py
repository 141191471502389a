"""GPU parity of the online-softmax rescale of the output accumulator.

The forward keeps, per query row, a running maximum m and row sum l, and
rescales the partial output by e^(m - m') when a later key block raises the
maximum to m' (apxml.com chapter "高效注意力算法实现 (FlashAttention)",
section "在线Softmax"; fmread.com summary, section 三.2 "增量Softmax计算").
The kernels hold that accumulator in tensor memory and rescale it only when
the maximum grows by more than 8 log2 units, which iid N(0,1) inputs at
scale 1/sqrt(d) never reach.  These tests feed inputs whose scores rise
along the key axis (helpers.scenario_bits: a rising gain, a spike of keys in
a middle block, a spike in the last block), count the rows whose maximum
grows past the threshold after their first key block -- each such row
rescales a nonzero accumulator -- and compare O, L and the gradients with
the fp64 oracle element by element.  tests/test_rescale_inputs.py shows on
the CPU that a rescale done wrongly on these inputs misses the O tolerance
tenfold.

Every plain forward instantiation (d = 64, 128, 256; causal or not), the
window / block-mask and dropout instantiations, the e4m3 forward, scales
other than 1/sqrt(d), and sampled rows at 16K tokens are covered.

O tolerance.  On these inputs a row's weights can concentrate on one key,
so |O| reaches 4 and more, where the spacing of bf16 is 2^-5 and even the
correctly rounded exact value can miss a flat 1e-2.  O is therefore checked
against the bound the bf16 arithmetic allows (the same as under dropout):
two bf16 roundings, of the weights fed to the product and of O, each at
most 2^-9 relative, with a factor two of margin --
|dO_ic| <= max(1e-2, 2^-8 (|O_ic| + sum_j p_ij |v_jc|)), the sum taken by the
oracle on |V|.  L and the gradients keep their tolerances."""
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


def scenario_case(kind, seed, B, Hh, N, d, scale=None):
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    return H.Case(seed, B, Hh, N, d, bits=H.scenario_bits(kind, seed, B, Hh, N, d, scale),
                  scale=scale)


def count_rescaled(case, causal, rows=None, window=-1, bm=None):
    rows = np.arange(case.N) if rows is None else np.asarray(rows)
    n = 0
    for b in range(case.B):
        vis = H.visible(case.N, rows, causal, case.length(b), window, bm)
        for h in range(case.H):
            n += H.rescaled_rows(case.f64["Q"][b, h], case.f64["K"][b, h], case.scale, vis,
                                 rows)
    return n


def run(case, causal, window=-1, bm=None, p=0.0, seed=0):
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


def check_full(case, causal, window=-1, bm=None, p=0.0, seed=0):
    n = count_rescaled(case, causal, window=window, bm=bm)
    assert n > 0, "no row rescales: the inputs miss the branch under test"
    o, L, dq, dk, dv = run(case, causal, window, bm, p, seed)
    args = (case.f64["Q"], case.f64["K"], case.f64["V"])
    pp = float(np.float32(p))
    kw = dict(kv_len=case.kv_len, window=window, block_mask=bm, block=128, dropout_p=pp,
              seed=seed)
    o_ref, L_ref = oracle.attn_fwd(*args, case.scale, causal, **kw)
    a_ref, _ = oracle.attn_fwd(args[0], args[1], np.abs(args[2]), case.scale, causal, **kw)
    excess = np.abs(o - o_ref) - H.o_bound_bf16(o_ref, a_ref)
    assert excess.max() <= 0.0, ("O", float(np.abs(o - o_ref).max()), float(excess.max()))
    assert H.err_l(L, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L, L_ref))
    g_ref = oracle.attn_bwd(*args, case.f64["dO"], case.scale, causal, **kw)
    errs = [H.err_rel(g, r) for g, r in zip((dq, dk, dv), g_ref)]
    H.report("rescale", case, causal, rows_rescaled=n, err_O=H.err_o(o, o_ref),
             err_L=H.err_l(L, L_ref), err_dQ=errs[0], err_dK=errs[1], err_dV=errs[2])
    for name, e in zip(("dQ", "dK", "dV"), errs):
        assert e <= H.TOL_GRAD_REL, (name, e)


@pytest.mark.parametrize("kind", H.RESCALE_SCENARIOS)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_plain(kind, d, causal):
    # N = 1000: 16 blocks of 64 keys, 8 query blocks, a ragged tail
    check_full(scenario_case(kind, 6000 + d, 1, 2, 1000, d), causal)


@pytest.mark.parametrize("kind", ["ramp", "mid"])
@pytest.mark.parametrize("factor", [0.5, 2.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_other_scales(kind, factor, d, causal):
    # The levels are set in log2 units of the scaled score, so the scenario
    # keeps its jumps at any scale; the kernels take the scale as given.
    check_full(scenario_case(kind, 6100 + d, 1, 2, 777, d, scale=factor / np.sqrt(d)), causal)


@pytest.mark.parametrize("kind", ["ramp", "mid"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_window_and_block_mask(kind, d, causal):
    N = 1000
    case = scenario_case(kind, 6200 + d, 1, 2, N, d)
    check_full(case, causal, window=300)
    bm = inputs.block_mask(6200 + d, (N + 127) // 128, 0.6, True)
    check_full(case, causal, bm=bm)


@pytest.mark.parametrize("kind", ["ramp", "mid"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_dropout(kind, d, causal):
    case = scenario_case(kind, 6300 + d, 1, 2, 1000, d)
    check_full(case, causal, p=0.1, seed=0x1234 + d)


@pytest.mark.parametrize("kind", H.RESCALE_SCENARIOS)
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_fp8(kind, causal):
    # e4m3 codes of the same scenario (dequantisation factors 1); tolerance of
    # the e4m3 forward: |dO| <= max(1e-2, 2^-4 (sum_j p |v_j| + |O|) + 2^-8 |O|)
    import torch
    from exact_io_aware_40_gb300 import fa
    B, Hh, N, d = 1, 2, 1000, 128
    scale = 1.0 / np.sqrt(d)
    codes = H.scenario_bits(kind, 6400, B, Hh, N, d, scale, fmt="e4m3")
    f = {n: inputs.e4m3_bits_to_f64(c) for n, c in codes.items()}
    rows = np.arange(N)
    vis = H.visible(N, rows, causal)
    n = sum(H.rescaled_rows(f["Q"][0, h], f["K"][0, h], scale, vis, rows) for h in range(Hh))
    assert n > 0
    dev = {nm: torch.from_numpy(c).to("cuda:0") for nm, c in codes.items()}
    o = torch.empty((B, Hh, N, d), dtype=torch.bfloat16, device="cuda:0")
    L = torch.empty((B, Hh, N), dtype=torch.float32, device="cuda:0")
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, Hh, N, d), dtype=torch.uint8,
                     device="cuda:0")
    fa.fa_fwd_fp8(dev["Q"], dev["K"], dev["V"], o, L, scale, 1.0, 1.0, 1.0, causal, None, ws)
    fa.fa_check_error()
    o, L = H.to_f64(o), H.to_f64(L)
    o_ref, L_ref = oracle.attn_fwd(f["Q"], f["K"], f["V"], scale, causal)
    a_ref, _ = oracle.attn_fwd(f["Q"], f["K"], np.abs(f["V"]), scale, causal)
    bound = np.maximum(H.TOL_O_ABS, 2.0 ** -4 * (a_ref + np.abs(o_ref)) + 2.0 ** -8 * np.abs(o_ref))
    assert (np.abs(o - o_ref) - bound).max() <= 0.0, ("O", float(np.abs(o - o_ref).max()))
    assert H.err_l(L, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L, L_ref))


@pytest.mark.parametrize("kind", ["ramp", "mid"])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_long_sequence_sampled(kind, causal):
    # B=1, H=2, N=16384, d=128: the benchmark's launch shape, sampled rows
    # and key columns of both heads
    N = 16384
    case = scenario_case(kind, 6500, 1, 2, N, 128)
    rows = np.array([0, 1, 127, 128, 4095, 8191, 8192, 8193, 8200, 12000, 16255, 16256, 16383])
    assert count_rescaled(case, causal, rows) > 0
    o, L, dq, dk, dv = run(case, causal)
    for h in range(2):
        qh, kh, vh, doh = (case.f64[n][0, h] for n in ("Q", "K", "V", "dO"))
        o_ref, L_ref = oracle.fwd_rows(qh, kh, vh, case.scale, causal, N, rows)
        a_ref, _ = oracle.fwd_rows(qh, kh, np.abs(vh), case.scale, causal, N, rows)
        assert (np.abs(o[0, h, rows] - o_ref) - H.o_bound_bf16(o_ref, a_ref)).max() <= 0.0
        assert H.err_l(L[0, h, rows], L_ref) <= H.TOL_L_ABS
        dq_ref = oracle.bwd_dq_rows(qh, kh, vh, doh, case.scale, causal, N, rows)
        dk_ref, dv_ref = oracle.bwd_dkdv_cols(qh, kh, vh, doh, case.scale, causal, N, rows)
        for name, g, r in (("dQ", dq[0, h, rows], dq_ref), ("dK", dk[0, h, rows], dk_ref),
                           ("dV", dv[0, h, rows], dv_ref)):
            assert H.err_rel(g, r) <= H.TOL_GRAD_REL, (name, h, H.err_rel(g, r))
