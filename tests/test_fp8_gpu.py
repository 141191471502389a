"""GPU parity of the e4m3 forward (fa_fwd_fp8) against the fp64 oracle run on
the dequantised inputs (factor x code, exact in fp64).

The products are exact up to fp32 accumulation, so L keeps its 1e-3
tolerance.  P enters the PV product rounded to e4m3 (3 mantissa bits: each
weight w_j within 2^-4 of p_j relative), and O is divided by the sum of the
unrounded weights, so O - O_ref = sum_j (w_j - p_j) v_jc / sum_j p_j and
|dO_ic| <= 2^-4 A_ic, A = sum_j p_ij |v_jc| (the oracle on |V|), plus the bf16
rounding of O (2^-8 |O| with margin).  The check allows 2^-4 (A_ic + |O_ic|) +
2^-8 |O_ic|, or 1e-2 where larger: the bound of dividing by the sum of the
rounded weights instead, which contains this one."""
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


def make(seed, B, Hh, N, d=128):
    codes = {n: inputs.normal_e4m3_bits(seed, inputs.STREAM[n], (B, Hh, N, d))
             for n in ("Q", "K", "V")}
    return codes


def run_fp8(codes, scale, dq, dk, dv, causal, kv_len=None):
    import torch
    from exact_io_aware_40_gb300 import fa
    dev = {n: torch.from_numpy(c).to("cuda:0") for n, c in codes.items()}
    B, Hh, N, d = codes["Q"].shape
    o = torch.empty((B, Hh, N, d), dtype=torch.bfloat16, device="cuda:0")
    L = torch.empty((B, Hh, N), dtype=torch.float32, device="cuda:0")
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, Hh, N, d), dtype=torch.uint8,
                     device="cuda:0")
    kv = None if kv_len is None else torch.from_numpy(np.asarray(kv_len, np.int32)).to("cuda:0")
    fa.fa_fwd_fp8(dev["Q"], dev["K"], dev["V"], o, L, scale, dq, dk, dv, causal, kv, ws)
    fa.fa_check_error()
    return H.to_f64(o), H.to_f64(L)


def check(codes, causal, dq=1.0, dk=1.0, dv=1.0, kv_len=None, rows=None):
    B, Hh, N, d = codes["Q"].shape
    scale = 1.0 / np.sqrt(d)
    f = {n: inputs.e4m3_bits_to_f64(c) * s for (n, c), s in zip(codes.items(), (dq, dk, dv))}
    o, L = run_fp8(codes, scale, dq, dk, dv, causal, kv_len)
    if rows is None:
        o_ref, L_ref = oracle.attn_fwd(f["Q"], f["K"], f["V"], scale, causal, kv_len=kv_len)
        a_ref, _ = oracle.attn_fwd(f["Q"], f["K"], np.abs(f["V"]), scale, causal, kv_len=kv_len)
    else:
        o_ref = np.zeros((B, Hh, len(rows), d)); L_ref = np.zeros((B, Hh, len(rows)))
        a_ref = np.zeros_like(o_ref)
        for b in range(B):
            for h in range(Hh):
                o_ref[b, h], L_ref[b, h] = oracle.fwd_rows(f["Q"][b, h], f["K"][b, h], f["V"][b, h],
                                                           scale, causal, N, rows)
                a_ref[b, h], _ = oracle.fwd_rows(f["Q"][b, h], f["K"][b, h],
                                                 np.abs(f["V"][b, h]), scale, causal, N, rows)
        o, L = o[:, :, rows], L[:, :, rows]
    bound = np.maximum(H.TOL_O_ABS, 2.0 ** -4 * (a_ref + np.abs(o_ref)) + 2.0 ** -8 * np.abs(o_ref))
    excess = np.abs(o - o_ref) - bound
    assert excess.max() <= 0.0, ("O", float(np.abs(o - o_ref).max()), float(excess.max()))
    assert H.err_l(L, L_ref) <= H.TOL_L_ABS, ("L", H.err_l(L, L_ref))
    return float(np.abs(o - o_ref).max())


@pytest.mark.parametrize("N", [1, 100, 128, 129, 383, 700])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_parity(N, causal):
    check(make(2500 + N, 2, 2, N), causal)


def test_fp8_forward_dequantisation_factors_and_key_padding():
    codes = make(2601, 3, 2, 520)
    check(codes, False, dq=0.5, dk=2.0, dv=0.25, kv_len=[520, 300, 0])
    check(codes, True, dq=1.5, dk=0.75, dv=3.0)


def test_fp8_forward_long_sequence_sampled():
    codes = make(2701, 1, 2, 16384)
    rows = np.array([0, 1, 127, 128, 5000, 16383])
    for causal in (False, True):
        check(codes, causal, rows=rows)


def test_fp8_forward_is_close_to_the_bf16_forward_on_the_same_values():
    # The same e4m3 values through the bf16 kernel (bf16 holds every e4m3
    # value exactly): the two differ only by the rounding of P.
    import torch
    from exact_io_aware_40_gb300 import fa
    codes = make(2801, 1, 4, 2048)
    o8, L8 = run_fp8(codes, 1 / np.sqrt(128), 1.0, 1.0, 1.0, True)
    t = {n: torch.from_numpy(inputs.e4m3_bits_to_f64(c)).to("cuda:0").to(torch.bfloat16)
         for n, c in codes.items()}
    o16, L16 = fa.attention_fwd(t["Q"], t["K"], t["V"], causal=True)
    fa.fa_check_error()
    assert float(np.abs(H.to_f64(L16) - L8).max()) <= 1e-3
    assert float(np.abs(H.to_f64(o16) - o8).max()) <= 0.1
