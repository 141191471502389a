"""Failure detection on the GPU without faulting it: a pipeline wait that can
never complete must end in FA_ERR_TIMEOUT after its time limit, and the
context must stay usable (the next attention call still matches the oracle)."""
import time

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


def test_stalled_wait_times_out_and_context_survives():
    from exact_io_aware_40_gb300 import fa
    fa.fa_check_error()  # start from a clean error word
    t0 = time.monotonic()
    fa.fa_selftest_stalled_wait(50_000_000)  # 50 ms limit
    with pytest.raises(fa.FAError) as exc:
        fa.fa_check_error()
    elapsed = time.monotonic() - t0
    assert exc.value.status == fa.FA_ERR_TIMEOUT
    assert elapsed < 5.0
    fa.fa_check_error()  # the error word was cleared by the previous read
    case = H.Case(1000, 1, 2, 200, 64)
    o, L = fa.attention_fwd(case.dev["Q"], case.dev["K"], case.dev["V"], causal=True,
                            scale=case.scale)
    fa.fa_check_error()
    o_ref, L_ref = oracle.attn_fwd(case.f64["Q"], case.f64["K"], case.f64["V"], case.scale, True)
    assert H.err_o(H.to_f64(o), o_ref) <= H.TOL_O_ABS
    assert H.err_l(H.to_f64(L), L_ref) <= H.TOL_L_ABS
