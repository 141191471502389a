"""CPU checks of the rising-score inputs that the GPU rescale tests use.

They show, without a GPU, that those inputs reach what the GPU tests claim
to reach: (1) many rows have a maximum that grows by more than 8 log2 units
after their first key block, so the kernels' conditional rescale of a
nonzero output accumulator runs; (2) the conditional rescale itself (keys
in blocks of 64, rescale only when the row maximum grows by more than 8 log2
units, the final division using the same reference maximum for numerator
and denominator) is exact -- it reaches the oracle's result to 1e-12; and
(3) the inputs are sharp: a rescale done wrongly (skipped, applied twice,
applied to half of the columns, or to the output but not to the row sum)
moves O from the oracle's result by ten times the 1e-2 tolerance or more, so
a GPU kernel with such a mistake fails the parity tests.

Online softmax with running maximum and sum: apxml.com chapter
"高效注意力算法实现 (FlashAttention)", section "在线Softmax"; fmread.com
summary, section 三.2 "增量Softmax计算"."""
import numpy as np
import pytest

import helpers as H
from exact_io_aware_40_gb300 import inputs
from oracle import oracle


def head(kind, N, d, scale, seed=77):
    bits = H.scenario_bits(kind, seed, 1, 1, N, d, scale, with_dout=False)
    return [inputs.bf16_bits_to_f64(bits[n])[0, 0] for n in ("Q", "K", "V")]


def conditional_rescale(q, k, v, scale, causal, Bc=64, thresh=8.0, mistake=None):
    """Test-only fp64 statement of the forward's recurrence in log2 units,
    with an optional planted mistake in the rescale step."""
    N, d = q.shape
    t_all = scale * H.LOG2E * (q @ k.T)
    if causal:
        t_all = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None], t_all, -np.inf)
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    acc = np.zeros((N, d))
    for j0 in range(0, N, Bc):
        t = t_all[:, j0:j0 + Bc]
        cand = np.maximum(m, t.max(axis=1))
        grow = cand > m + thresh
        m_new = np.where(grow, cand, m)
        with np.errstate(invalid="ignore"):
            alpha = np.where(grow, np.exp2(m - m_new), 1.0)
        alpha = np.where(np.isnan(alpha), 0.0, alpha)
        m_use = np.where(np.isneginf(m_new), 0.0, m_new)
        p = np.exp2(t - m_use[:, None])
        a_o = alpha
        if mistake == "skip":
            a_o = np.where(np.isneginf(m), 0.0, 1.0)
        elif mistake == "twice":
            a_o = alpha * alpha
        if mistake == "not_l":
            l = l + p.sum(axis=1)
        else:
            l = alpha * l + p.sum(axis=1)
        if mistake == "half":
            acc[:, :d // 2] *= alpha[:, None]
        else:
            acc *= a_o[:, None]
        acc += p @ v[j0:j0 + Bc]
        m = m_new
    return acc / l[:, None], (m + np.log2(l)) / H.LOG2E


@pytest.mark.parametrize("kind", H.RESCALE_SCENARIOS)
@pytest.mark.parametrize("causal", [False, True])
def test_rows_grow_past_the_threshold(kind, causal):
    N, d = 1000, 64
    scale = 1 / np.sqrt(d)
    q, k, _ = head(kind, N, d, scale)
    rows = np.arange(N)
    n = H.rescaled_rows(q, k, scale, H.visible(N, rows, causal), rows)
    # every scenario reaches some rows; the non-causal ramp and middle spike
    # reach nearly all of them
    assert n >= 1
    if not causal:
        assert n >= 0.95 * N, n
    if causal and kind == "mid":
        assert n >= 0.45 * N, n


@pytest.mark.parametrize("kind", H.RESCALE_SCENARIOS)
@pytest.mark.parametrize("causal", [False, True])
def test_conditional_rescale_is_exact(kind, causal):
    N, d = 700, 64
    scale = 1 / np.sqrt(d)
    q, k, v = head(kind, N, d, scale)
    o, L = conditional_rescale(q, k, v, scale, causal)
    o_ref, L_ref = oracle.attn_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_ref[0, 0], rtol=0, atol=1e-11)


@pytest.mark.parametrize("mistake", ["skip", "twice", "half", "not_l"])
@pytest.mark.parametrize("kind", ["mid", "last"])
def test_a_wrong_rescale_misses_the_tolerance(mistake, kind):
    N, d = 1000, 64
    scale = 1 / np.sqrt(d)
    q, k, v = head(kind, N, d, scale)
    o, _ = conditional_rescale(q, k, v, scale, False, mistake=mistake)
    o_ref, _ = oracle.attn_fwd(q[None, None], k[None, None], v[None, None], scale, False)
    assert np.abs(o - o_ref[0, 0]).max() > 10 * H.TOL_O_ABS
