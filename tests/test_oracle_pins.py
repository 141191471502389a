"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these checks compares the oracle with itself: each one is a closed
form, an invariant of softmax attention, a hand-derived worked example, a
finite-difference gradient, a restatement of the tiled online-softmax method
(which must give the same result, the pages' "exact attention" claim), or a
special case handled by an independent library routine.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(12345)


def rand(*shape):
    return rng.standard_normal(shape)


def visible_mask(N, causal, length):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    m = np.broadcast_to(j < length, (N, N))
    if causal:
        m = m & (j <= i)
    return m


# --- hand-derived worked example ------------------------------------------

def test_worked_example_golden():
    with open(os.path.join(HERE, "golden", "worked_example_n2_d1.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        sh = (1, 1, 2, 1)
        q, k, v, do = (np.array(case[n], np.float64).reshape(sh) for n in ("q", "k", "v", "dO"))
        o, L = oracle.attn_fwd(q, k, v, case["scale"], case["causal"])
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, case["scale"], case["causal"])
        np.testing.assert_allclose(o.ravel(), case["O"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(L.ravel(), case["L"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(dq.ravel(), case["dQ"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(dk.ravel(), case["dK"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(dv.ravel(), case["dV"], rtol=0, atol=1e-14, err_msg=case["name"])


# --- softmax structure: V = identity exposes P through O --------------------

@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("length", [8, 5])
def test_rows_of_P_sum_to_one_and_mask_is_zero(causal, length):
    N = d = 8
    q, k = rand(1, 1, N, d), rand(1, 1, N, d)
    v = np.eye(N).reshape(1, 1, N, d)           # O = P V = P
    o, _ = oracle.attn_fwd(q, k, v, 0.7, causal, kv_len=np.array([length]))
    P = o[0, 0]
    m = visible_mask(N, causal, length)
    assert np.all(P >= 0)
    assert np.all(P[~m] == 0.0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # P is the softmax of the visible scores: ratios follow exp(score difference)
    S = 0.7 * q[0, 0] @ k[0, 0].T
    for i in range(N):
        js = np.nonzero(m[i])[0]
        np.testing.assert_allclose(P[i, js] / P[i, js[0]], np.exp(S[i, js] - S[i, js[0]]),
                                   rtol=1e-13)


# --- closed forms ------------------------------------------------------------

@pytest.mark.parametrize("causal", [0, 1])
def test_identical_keys_give_mean_of_visible_values(causal):
    B, H, N, d = 2, 2, 9, 4
    q, v = rand(B, H, N, d), rand(B, H, N, d)
    k = np.broadcast_to(rand(1, 1, 1, d), (B, H, N, d)).copy()
    lens = np.array([9, 6])
    scale = 0.5
    o, L = oracle.attn_fwd(q, k, v, scale, causal, kv_len=lens)
    for b in range(B):
        m = visible_mask(N, causal, lens[b])
        for h in range(H):
            for i in range(N):
                cnt = m[i].sum()
                np.testing.assert_allclose(o[b, h, i], v[b, h, m[i]].mean(axis=0), atol=1e-14)
                np.testing.assert_allclose(L[b, h, i], scale * q[b, h, i] @ k[b, h, 0] + math.log(cnt),
                                           atol=1e-13)


def test_single_key_returns_v_and_scaled_score():
    q, k, v = rand(2, 3, 1, 16), rand(2, 3, 1, 16), rand(2, 3, 1, 16)
    for causal in (0, 1):
        o, L = oracle.attn_fwd(q, k, v, 0.25, causal)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(L, 0.25 * np.einsum("bhnc,bhnc->bhn", q, k), atol=1e-14)


@pytest.mark.parametrize("causal", [0, 1])
def test_zero_queries_give_uniform_weights(causal):
    B, H, N, d = 1, 2, 7, 3
    q = np.zeros((B, H, N, d))
    k, v = rand(B, H, N, d), rand(B, H, N, d)
    o, L = oracle.attn_fwd(q, k, v, 1.3, causal, kv_len=np.array([5]))
    m = visible_mask(N, causal, 5)
    for h in range(H):
        for i in range(N):
            np.testing.assert_allclose(o[0, h, i], v[0, h, m[i]].mean(axis=0), atol=1e-14)
            np.testing.assert_allclose(L[0, h, i], math.log(m[i].sum()), atol=1e-14)


# --- invariants --------------------------------------------------------------

@pytest.mark.parametrize("causal", [0, 1])
def test_key_shift_invariance(causal):
    B, H, N, d = 1, 1, 10, 5
    q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    c = rand(d)
    o1, L1 = oracle.attn_fwd(q, k, v, 0.6, causal)
    o2, L2 = oracle.attn_fwd(q, k + c, v, 0.6, causal)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(L2, L1 + 0.6 * q @ c, atol=1e-13)


def test_key_value_permutation_invariance():
    B, H, N, d = 1, 2, 11, 6
    q, k, v = rand(B, H, N, d), rand(B, H, N, d), rand(B, H, N, d)
    perm = rng.permutation(N)
    o1, L1 = oracle.attn_fwd(q, k, v, 0.4, 0)
    o2, L2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, 0)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(L2, L1, atol=1e-13)
    # the output rows follow the query order
    o3, _ = oracle.attn_fwd(q[:, :, perm], k, v, 0.4, 0)
    np.testing.assert_allclose(o3, o1[:, :, perm], atol=1e-13)


@pytest.mark.parametrize("causal", [0, 1])
def test_masked_positions_contribute_nothing(causal):
    B, H, N, d = 1, 1, 12, 4
    length = 8
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    kl = np.array([length])
    o1, L1 = oracle.attn_fwd(q, k, v, 0.5, causal, kv_len=kl)
    dq1, dk1, dv1 = oracle.attn_bwd(q, k, v, do, 0.5, causal, kv_len=kl)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, length:] += 10 * rand(N - length, d)
    v2[:, :, length:] -= 10 * rand(N - length, d)
    o2, L2 = oracle.attn_fwd(q, k2, v2, 0.5, causal, kv_len=kl)
    dq2, dk2, dv2 = oracle.attn_bwd(q, k2, v2, do, 0.5, causal, kv_len=kl)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(L1, L2)
    np.testing.assert_array_equal(dq1, dq2)
    assert np.all(dk1[:, :, length:] == 0) and np.all(dv1[:, :, length:] == 0)
    assert np.all(dk2[:, :, length:] == 0) and np.all(dv2[:, :, length:] == 0)


def test_causal_rows_ignore_later_keys():
    N, d = 10, 4
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    o1, L1 = oracle.attn_fwd(q, k, v, 0.5, 1)
    j = 6
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, j] += 3.0
    v2[0, 0, j] -= 3.0
    o2, L2 = oracle.attn_fwd(q, k2, v2, 0.5, 1)
    np.testing.assert_array_equal(o1[0, 0, :j], o2[0, 0, :j])
    np.testing.assert_array_equal(L1[0, 0, :j], L2[0, 0, :j])
    assert np.all(np.abs(o1[0, 0, j:] - o2[0, 0, j:]).max(axis=1) > 0)
    # row 0 sees key 0 only
    np.testing.assert_array_equal(o1[0, 0, 0], v[0, 0, 0])


def test_empty_rows_give_zero_output_and_minus_inf():
    q, k, v, do = (rand(1, 1, 4, 3) for _ in range(4))
    o, L = oracle.attn_fwd(q, k, v, 1.0, 0, kv_len=np.array([0]))
    assert np.all(o == 0) and np.all(np.isneginf(L))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 1.0, 0, kv_len=np.array([0]))
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


# --- backward: finite differences and row sums of dS --------------------------

@pytest.mark.parametrize("causal,length", [(0, 7), (1, 7), (0, 5), (1, 4)])
def test_backward_matches_central_differences(causal, length):
    N, d, scale, h = 7, 3, 0.8, 1e-6
    q, k, v, do = (rand(1, 1, N, d) for _ in range(4))
    kl = np.array([length])

    def f(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, scale, causal, kv_len=kl, nthreads=1)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.attn_bwd(q, k, v, do, scale, causal, kv_len=kl, nthreads=1)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        err = np.abs(num - grad).max() / max(np.abs(grad).max(), 1e-300)
        assert err <= 1e-6, (which, err)


@pytest.mark.parametrize("causal", [0, 1])
def test_dk_columns_sum_to_zero(causal):
    # sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0 because each row of dS sums to 0
    q, k, v, do = (rand(2, 2, 16, 8) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.35, causal)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-13)
    # sum_j dV_j = sum_i (sum_j p_ij) dO_i = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


# --- the tiled online-softmax method reaches the same numbers ------------------

def tiled_online_attention(q, k, v, scale, causal, length, Br, Bc):
    """Test-only fp64 restatement of the tiled method: query blocks of Br rows,
    key/value blocks of Bc rows, a running row max m and row sum l that rescale
    the output accumulator as blocks arrive (fmread.com summary section 三.2
    "增量Softmax计算"; apxml.com chapter, "在线Softmax"; study notes
    "分块计算整体流程(Tiling)")."""
    N, d = q.shape
    O = np.zeros((N, d))
    L = np.zeros(N)
    for i0 in range(0, N, Br):
        rows = np.arange(i0, min(i0 + Br, N))
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        acc = np.zeros((len(rows), d))
        for j0 in range(0, N, Bc):
            cols = np.arange(j0, min(j0 + Bc, N))
            S = scale * q[rows] @ k[cols].T
            vis = cols[None, :] < length
            if causal:
                vis = vis & (cols[None, :] <= rows[:, None])
            S = np.where(vis, S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            safe = np.where(np.isneginf(m_new), 0.0, m_new)
            Pt = np.exp(S - safe[:, None])
            alpha = np.exp(np.where(np.isneginf(m), -np.inf, m - safe))
            l = alpha * l + Pt.sum(axis=1)
            acc = alpha[:, None] * acc + Pt @ v[cols]
            m = m_new
        with np.errstate(invalid="ignore", divide="ignore"):
            O[rows] = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1)[:, None], 0.0)
            L[rows] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1)), -np.inf)
    return O, L


@pytest.mark.parametrize("Br,Bc", [(1, 1), (3, 3), (16, 3), (3, 16), (128, 128), (16, 128)])
@pytest.mark.parametrize("causal,length", [(0, 37), (1, 37), (0, 20), (1, 29)])
def test_tiled_online_softmax_equals_untiled(Br, Bc, causal, length):
    N, d = 37, 8
    q, k, v = rand(N, d), rand(N, d), rand(N, d)
    o, L = oracle.attn_fwd(q[None, None], k[None, None], v[None, None], 0.4, causal,
                           kv_len=np.array([length]))
    ot, Lt = tiled_online_attention(q, k, v, 0.4, causal, length, Br, Bc)
    np.testing.assert_allclose(ot, o[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lt, L[0, 0], rtol=0, atol=1e-12)


# --- special case handled by an independent library routine ------------------

@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_fp64_sdpa_with_autograd(causal):
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 2, 13, 8
    lens = np.array([13, 9])
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    o, L = oracle.attn_fwd(q, k, v, 0.3, causal, kv_len=lens)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.3, causal, kv_len=lens)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = torch.zeros(B, 1, N, N, dtype=torch.bool)
    for b in range(B):
        mask[b, 0] = torch.tensor(visible_mask(N, causal, lens[b]))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.3)
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
    s = 0.3 * np.einsum("bhic,bhjc->bhij", q, k)
    s = np.where(mask.numpy(), s, -np.inf)
    np.testing.assert_allclose(L, np.logaddexp.reduce(s, axis=-1), atol=1e-12)


# --- the sampled entry points follow the same definition ---------------------

@pytest.mark.parametrize("causal,length", [(0, 40), (1, 40), (0, 23), (1, 31)])
def test_sampled_rows_and_columns_match_whole_tensor_results(causal, length):
    N, d = 40, 8
    q, k, v, do = (rand(1, 1, N, d) for _ in range(4))
    kl = np.array([length])
    o, L = oracle.attn_fwd(q, k, v, 0.5, causal, kv_len=kl)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, causal, kv_len=kl)
    rows = np.array([0, 1, 17, 39])
    o_r, L_r = oracle.fwd_rows(q[0, 0], k[0, 0], v[0, 0], 0.5, causal, length, rows)
    np.testing.assert_allclose(o_r, o[0, 0, rows], atol=1e-14)
    np.testing.assert_allclose(L_r, L[0, 0, rows], atol=1e-14)
    dq_r = oracle.bwd_dq_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.5, causal, length, rows)
    np.testing.assert_allclose(dq_r, dq[0, 0, rows], atol=1e-13)
    cols = np.array([0, 5, 22, 39])
    dk_c, dv_c = oracle.bwd_dkdv_cols(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.5, causal, length, cols)
    np.testing.assert_allclose(dk_c, dk[0, 0, cols], atol=1e-13)
    np.testing.assert_allclose(dv_c, dv[0, 0, cols], atol=1e-13)


# --- sliding window and block-sparse mask terms --------------------------------

def band_mask(N, window):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (j <= i) & (j >= i - window)


def block_to_pos(bm, N, bs):
    """Expand a (query block, key block) mask to positions."""
    blk = np.arange(N) // bs
    return bm[blk[:, None], blk[None, :]].astype(bool)


def test_window_zero_attends_to_own_position_only():
    # With w = 0 every row keeps exactly one key (itself): P is the identity,
    # so O = V, L = scale q_i.k_i, dV = dO and dS = 0 (dQ = dK = 0).
    B, H, N, d = 1, 2, 9, 5
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    o, L = oracle.attn_fwd(q, k, v, 0.7, False, window=0)
    np.testing.assert_allclose(o, v, atol=1e-14)
    np.testing.assert_allclose(L, 0.7 * np.einsum("bhic,bhic->bhi", q, k), atol=1e-13)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.7, False, window=0)
    np.testing.assert_allclose(dv, do, atol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)


def test_window_rows_ignore_keys_outside_the_band():
    # Perturbing K, V outside row i's band [i - w, i] leaves row i unchanged.
    N, d, w = 12, 4, 3
    q, k, v = (rand(1, 1, N, d) for _ in range(3))
    o, L = oracle.attn_fwd(q, k, v, 0.5, False, window=w)
    i = 7
    k2, v2 = k.copy(), v.copy()
    outside = [j for j in range(N) if not (i - w <= j <= i)]
    k2[0, 0, outside] += rand(len(outside), d)
    v2[0, 0, outside] += rand(len(outside), d)
    o2, L2 = oracle.attn_fwd(q, k2, v2, 0.5, False, window=w)
    np.testing.assert_allclose(o2[0, 0, i], o[0, 0, i], atol=1e-14)
    np.testing.assert_allclose(L2[0, 0, i], L[0, 0, i], atol=1e-14)


def test_block_diagonal_mask_equals_independent_blocks():
    # A block mask that keeps only the diagonal pairs splits the sequence into
    # independent attention problems, one per block: each must equal the
    # unmasked oracle run on that block alone.
    N, d, bs = 11, 6, 4
    q, k, v, do = (rand(1, 2, N, d) for _ in range(4))
    nb = (N + bs - 1) // bs
    bm = np.eye(nb, dtype=np.uint8)
    o, L = oracle.attn_fwd(q, k, v, 0.4, False, block_mask=bm, block=bs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.4, False, block_mask=bm, block=bs)
    for t in range(nb):
        sl = slice(t * bs, min(N, (t + 1) * bs))
        ob, Lb = oracle.attn_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.4, False)
        gq, gk, gv = oracle.attn_bwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], 0.4, False)
        np.testing.assert_allclose(o[:, :, sl], ob, atol=1e-14)
        np.testing.assert_allclose(L[:, :, sl], Lb, atol=1e-14)
        np.testing.assert_allclose(dq[:, :, sl], gq, atol=1e-13)
        np.testing.assert_allclose(dk[:, :, sl], gk, atol=1e-13)
        np.testing.assert_allclose(dv[:, :, sl], gv, atol=1e-13)


def test_all_ones_block_mask_changes_nothing_and_empty_block_rows_are_zero():
    N, d, bs = 10, 4, 4
    q, k, v, do = (rand(1, 1, N, d) for _ in range(4))
    nb = 3
    o0, L0 = oracle.attn_fwd(q, k, v, 0.5, True)
    o1, L1 = oracle.attn_fwd(q, k, v, 0.5, True, block_mask=np.ones((nb, nb), np.uint8), block=bs)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(L0, L1)
    # query block 1 keeps no key block: its rows are empty (O = 0, L = -inf,
    # zero gradients), and keys are only reached from the other blocks
    bm = np.ones((nb, nb), np.uint8)
    bm[1, :] = 0
    o, L = oracle.attn_fwd(q, k, v, 0.5, False, block_mask=bm, block=bs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, False, block_mask=bm, block=bs)
    np.testing.assert_array_equal(o[0, 0, 4:8], 0.0)
    assert np.all(np.isneginf(L[0, 0, 4:8]))
    np.testing.assert_array_equal(dq[0, 0, 4:8], 0.0)


@pytest.mark.parametrize("causal,window,use_bm", [(False, 2, False), (True, 5, True),
                                                  (False, -1, True), (True, -1, True)])
def test_window_and_block_mask_match_torch_fp64_sdpa(causal, window, use_bm):
    torch = pytest.importorskip("torch")
    B, H, N, d, bs = 2, 2, 14, 8, 4
    lens = np.array([14, 10])
    nb = (N + bs - 1) // bs
    bm = (np.random.default_rng(7).random((nb, nb)) < 0.6).astype(np.uint8)
    np.fill_diagonal(bm, 1)   # every query keeps its own position: no empty rows
    bm_arg = bm if use_bm else None
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    o, L = oracle.attn_fwd(q, k, v, 0.3, causal, kv_len=lens, window=window,
                           block_mask=bm_arg, block=bs)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.3, causal, kv_len=lens, window=window,
                                 block_mask=bm_arg, block=bs)
    mask = np.zeros((B, 1, N, N), bool)
    for b in range(B):
        m = visible_mask(N, causal, lens[b])
        if window >= 0:
            m = m & band_mask(N, window)
        if use_bm:
            m = m & block_to_pos(bm, N, bs)
        mask[b, 0] = m
    # Rows that keep no key (a query block whose kept pairs all lie past
    # kv_len) are NaN in the library; compare the others, and check the empty
    # ones against the empty-row convention (O = 0, L = -inf, no gradient).
    keep = np.broadcast_to(mask.any(-1), (B, H, N))
    kp = np.broadcast_to(keep[..., None], o.shape)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(mask),
                                                          scale=0.3)
    to = torch.where(torch.tensor(kp), to, torch.zeros_like(to))
    to.backward(torch.tensor(np.where(kp, do, 0.0)))
    np.testing.assert_allclose(o[kp], to.detach().numpy()[kp], atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)
    assert np.all(o[~kp] == 0.0) and np.all(np.isneginf(L[~keep])) and np.all(dq[~kp] == 0.0)
    s = 0.3 * np.einsum("bhic,bhjc->bhij", q, k)
    s = np.where(mask, s, -np.inf)
    with np.errstate(invalid="ignore"):
        ref_L = np.logaddexp.reduce(s, axis=-1)
    np.testing.assert_allclose(L[keep], ref_L[keep], atol=1e-12)


@pytest.mark.parametrize("causal,length,window,use_bm", [(0, 40, 7, False), (1, 33, -1, True),
                                                         (0, 40, -1, True), (1, 40, 20, True)])
def test_sampled_entry_points_follow_window_and_block_mask(causal, length, window, use_bm):
    N, d, bs = 40, 8, 8
    nb = N // bs
    bm = (np.random.default_rng(3).random((nb, nb)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm_arg = bm if use_bm else None
    q, k, v, do = (rand(1, 1, N, d) for _ in range(4))
    kl = np.array([length])
    kw = dict(window=window, block_mask=bm_arg, block=bs)
    o, L = oracle.attn_fwd(q, k, v, 0.5, causal, kv_len=kl, **kw)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, causal, kv_len=kl, **kw)
    rows = np.array([0, 1, 17, 39])
    o_r, L_r = oracle.fwd_rows(q[0, 0], k[0, 0], v[0, 0], 0.5, causal, length, rows, **kw)
    np.testing.assert_allclose(o_r, o[0, 0, rows], atol=1e-14)
    np.testing.assert_allclose(L_r, L[0, 0, rows], atol=1e-14)
    dq_r = oracle.bwd_dq_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.5, causal, length, rows, **kw)
    np.testing.assert_allclose(dq_r, dq[0, 0, rows], atol=1e-13)
    cols = np.array([0, 5, 22, 39])
    dk_c, dv_c = oracle.bwd_dkdv_cols(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.5, causal, length,
                                      cols, **kw)
    np.testing.assert_allclose(dk_c, dk[0, 0, cols], atol=1e-13)
    np.testing.assert_allclose(dv_c, dv[0, 0, cols], atol=1e-13)


# --- dropout ------------------------------------------------------------------

def test_philox4x32_10_known_answers():
    # Known-answer vectors published with the generator's reference
    # implementation (Random123): zero counter and key, all-ones counter and
    # key, and counter/key taken from the hexadecimal digits of pi.
    assert oracle.philox4x32_10([0, 0, 0, 0], [0, 0]) == [
        0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    ones = 0xFFFFFFFF
    assert oracle.philox4x32_10([ones] * 4, [ones] * 2) == [
        0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert oracle.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                                [0xA4093822, 0x299F31D0]) == [
        0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_dropout_decisions_follow_the_counter_layout():
    # Z_ij comes from Philox at counter (j // 8, i, h, b), key (seed low, high),
    # 16-bit value j % 8 (low half of word (j % 8) // 2 first), kept iff
    # u >= floor(p * 65536).  Spot-check against direct generator calls.
    p, seed, b, h, N = 0.3, 0x0123456789ABCDEF, 1, 2, 40
    m = oracle.dropout_mult(b, h, N, p, seed)
    thr = int(math.floor(p * 65536))
    inv_q = 65536.0 / (65536 - thr)
    for (i, j) in [(0, 0), (0, 7), (3, 8), (17, 33), (39, 39), (5, 22)]:
        w = oracle.philox4x32_10([j // 8, i, h, b], [seed & 0xFFFFFFFF, seed >> 32])[(j % 8) // 2]
        u = (w >> 16) if (j % 8) % 2 else (w & 0xFFFF)
        assert m[i, j] == (inv_q if u >= thr else 0.0)


def test_dropout_keep_rate_and_unbiased_scale():
    p, N = 0.25, 1024
    ms = [oracle.dropout_mult(b, h, N, p, 777) for b in (0, 1) for h in (0, 3)]
    keep = np.mean([(m > 0).mean() for m in ms])
    q = (65536 - math.floor(p * 65536)) / 65536
    sigma = math.sqrt(q * (1 - q) / (4 * N * N))
    assert abs(keep - q) < 5 * sigma
    assert abs(np.mean([m.mean() for m in ms]) - 1.0) < 5 * sigma / q
    # different heads, batches and rows draw different decisions
    assert not np.array_equal(ms[0], ms[1]) and not np.array_equal(ms[0], ms[2])
    assert not np.array_equal(ms[0][0], ms[0][1])


def test_dropout_zero_is_no_dropout_and_single_key_closed_form():
    q, k, v, do = (rand(2, 2, 33, 8) for _ in range(4))
    o0, L0 = oracle.attn_fwd(q, k, v, 0.5, True)
    o1, L1 = oracle.attn_fwd(q, k, v, 0.5, True, dropout_p=0.0, seed=99)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(L0, L1)
    g0 = oracle.attn_bwd(q, k, v, do, 0.5, True)
    g1 = oracle.attn_bwd(q, k, v, do, 0.5, True, dropout_p=0.0, seed=99)
    for a, b in zip(g0, g1):
        np.testing.assert_array_equal(a, b)
    # one key: P = 1, so O = v * Z/q and L = scale q.k whatever the drop
    q1, k1, v1 = (rand(1, 3, 1, 6) for _ in range(3))
    o, L = oracle.attn_fwd(q1, k1, v1, 0.7, False, dropout_p=0.4, seed=5)
    for h in range(3):
        mult = oracle.dropout_mult(0, h, 1, 0.4, 5)[0, 0]
        np.testing.assert_allclose(o[0, h, 0], v1[0, h, 0] * mult, atol=1e-15)
    np.testing.assert_allclose(L, 0.7 * np.einsum("bhic,bhic->bhi", q1, k1), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_matches_torch_fp64_autograd_with_the_same_multipliers(causal):
    # The attention arithmetic with dropout, restated with library operations
    # (softmax, matmul, autograd) around the oracle's own multiplier matrix.
    torch = pytest.importorskip("torch")
    B, H, N, d, p, seed = 2, 2, 21, 8, 0.35, 2024
    lens = np.array([21, 14])
    q, k, v, do = (rand(B, H, N, d) for _ in range(4))
    o, L = oracle.attn_fwd(q, k, v, 0.4, causal, kv_len=lens, dropout_p=p, seed=seed)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.4, causal, kv_len=lens, dropout_p=p, seed=seed)
    mult = np.stack([np.stack([oracle.dropout_mult(b, h, N, p, seed) for h in range(H)])
                     for b in range(B)])
    mask = np.zeros((B, 1, N, N), bool)
    for b in range(B):
        mask[b, 0] = visible_mask(N, causal, lens[b])
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    s = 0.4 * tq @ tk.transpose(-1, -2)
    s = s.masked_fill(~torch.tensor(mask), float("-inf"))
    P = torch.softmax(s, dim=-1)
    to = (P * torch.tensor(mult)) @ tv
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_dropout_backward_matches_central_differences():
    # With the seed fixed the dropout decisions are fixed, so <dO, O> is a
    # smooth function of Q, K, V and its gradient is the backward pass.
    N, d, p, seed = 9, 4, 0.3, 31
    q, k, v, do = (rand(1, 1, N, d) for _ in range(4))
    f = lambda q_, k_, v_: float((oracle.attn_fwd(q_, k_, v_, 0.6, True, dropout_p=p,
                                                  seed=seed)[0] * do).sum())
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.6, True, dropout_p=p, seed=seed)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            args_m = [xm if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_dropout_sampled_entry_points_match_whole_tensor_results():
    N, d, p, seed = 40, 8, 0.2, 77
    q, k, v, do = (rand(2, 3, N, d) for _ in range(4))
    kl = np.array([40, 29])
    kw = dict(window=11, dropout_p=p, seed=seed)
    o, L = oracle.attn_fwd(q, k, v, 0.5, True, kv_len=kl, **kw)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, True, kv_len=kl, **kw)
    rows = np.array([0, 1, 17, 39])
    cols = np.array([0, 5, 22, 39])
    for b, h in ((0, 0), (1, 2)):
        qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
        ln = int(kl[b])
        o_r, L_r = oracle.fwd_rows(qh, kh, vh, 0.5, True, ln, rows, b=b, h=h, **kw)
        np.testing.assert_allclose(o_r, o[b, h, rows], atol=1e-14)
        np.testing.assert_allclose(L_r, L[b, h, rows], atol=1e-14)
        dq_r = oracle.bwd_dq_rows(qh, kh, vh, doh, 0.5, True, ln, rows, b=b, h=h, **kw)
        np.testing.assert_allclose(dq_r, dq[b, h, rows], atol=1e-13)
        dk_c, dv_c = oracle.bwd_dkdv_cols(qh, kh, vh, doh, 0.5, True, ln, cols, b=b, h=h, **kw)
        np.testing.assert_allclose(dk_c, dk[b, h, cols], atol=1e-13)
        np.testing.assert_allclose(dv_c, dv[b, h, cols], atol=1e-13)
