"""Shared helpers of the GPU parity tests: seeded inputs on the device, the
same inputs widened to fp64 for the oracle, and the error measures."""
import json
import math
import os

import numpy as np

from exact_io_aware_40_gb300 import inputs

# Tolerances fixed by the problem statement for bf16 inputs.
TOL_O_ABS = 1e-2      # max |O - O_ref|
TOL_L_ABS = 1e-3      # max |L - L_ref| over finite entries
TOL_GRAD_REL = 5e-2   # max |g - g_ref| / max |g_ref| for dQ, dK, dV


class Case:
    """One seeded workload: bf16 device tensors plus their exact fp64 values."""

    def __init__(self, seed, B, H, N, d, kv_range=None, with_dout=True, device="cuda:0",
                 bits=None, scale=None):
        import torch
        self.B, self.H, self.N, self.d = B, H, N, d
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        if bits is None:
            bits = inputs.attention_inputs(seed, B, H, N, d, with_dout=with_dout)
        self.f64 = {n: inputs.bf16_bits_to_f64(b) for n, b in bits.items()}
        self.dev = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)
                    for n, b in bits.items()}
        self.kv_len = None
        self.kv_len_dev = None
        if kv_range is not None:
            lo, hi = kv_range
            self.kv_len = inputs.kv_lengths(seed, B, lo, hi)
            self.kv_len_dev = torch.from_numpy(self.kv_len).to(device)

    def set_kv_len(self, lens, device="cuda:0"):
        import torch
        self.kv_len = np.asarray(lens, np.int32)
        self.kv_len_dev = torch.from_numpy(self.kv_len).to(device)

    def length(self, b):
        return self.N if self.kv_len is None else int(min(max(self.kv_len[b], 0), self.N))


def to_f64(t):
    return t.double().cpu().numpy()


def err_o(o, o_ref):
    return float(np.abs(o - o_ref).max()) if o.size else 0.0


def err_l(L, L_ref):
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isneginf(L), np.isneginf(L_ref)), "-inf pattern of L differs"
    return float(np.abs(L[fin] - L_ref[fin]).max()) if fin.any() else 0.0


def err_rel(g, g_ref):
    den = float(np.abs(g_ref).max())
    num = float(np.abs(g - g_ref).max())
    if den == 0.0:
        return num
    return num / den


def report(kind, case, causal, **errs):
    """Append the measured errors of one check as a JSON line to the file named
    by FA_PARITY_REPORT (no-op when unset); used to tabulate parity results."""
    path = os.environ.get("FA_PARITY_REPORT")
    if not path:
        return
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "kind": kind,
           "B": case.B, "H": case.H, "N": case.N, "d": case.d, "causal": int(bool(causal)),
           "kv_len": None if case.kv_len is None else [int(x) for x in case.kv_len]}
    rec.update({k: float(v) for k, v in errs.items()})
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


# --- inputs whose row maximum rises across key blocks ------------------------
#
# The forward keeps a running row maximum m and rescales its output
# accumulator when a later key block raises m (the online softmax of the
# apxml.com chapter, section "在线Softmax", and of the fmread.com summary,
# section 三.2 "增量Softmax计算").  iid N(0,1) inputs at scale 1/sqrt(d) raise
# m by 2-3 log2 units over a whole row; the kernels skip a rescale below 8
# log2 units, so these shapes make m jump by more.

LOG2E = 1.0 / math.log(2.0)
RESCALE_SCENARIOS = ("ramp", "mid", "last")


def scenario_bits(kind, seed, B, H, N, d, scale, fmt="bf16", with_dout=True):
    """Seeded inputs of one rising-score scenario (scores are `scale` times Q K^T):
      ramp      key row j scaled by a gain rising linearly from 1 to 6;
      mid       flat scores (noise 0.25) with keys at N/2 raised by 10 log2
                units -- one key per 1024 earlier keys, so the earlier keys
                still carry about half of the weight after the rescale;
                V has mean 1, so that half of the weight moves O;
      last      flat scores with the last keys raised by 10 log2 units (one
                per 1024 earlier keys, at least one), all in the final block;
                V has mean 1."""
    unit = math.log(2.0) / scale  # one log2 unit of scaled score, unscaled
    kw = dict(fmt=fmt, with_dout=with_dout)
    if kind == "ramp":
        gain = 1.0 + 5.0 * np.arange(N) / max(N - 1, 1)
        return inputs.shaped_key_inputs(seed, B, H, N, d, gain=gain, **kw)
    lv = np.zeros(N)
    if kind == "mid":
        c = max(1, (N // 2) >> 10)
        lv[N // 2:N // 2 + c] = 10.0 * unit
    elif kind == "last":
        c = min(64, max(1, N >> 10))
        lv[N - c:] = 10.0 * unit
    else:
        raise ValueError(kind)
    return inputs.shaped_key_inputs(seed, B, H, N, d, levels=lv, noise=0.25, v_shift=1.0, **kw)


def visible(N, rows, causal, length=None, window=-1, block_mask=None, block=128):
    """[len(rows), N] bool: key j visible to query i under every mask term."""
    i = np.asarray(rows)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((len(rows), N), bool)
    if length is not None:
        vis &= j < length
    if causal or window >= 0:
        vis &= j <= i
    if window >= 0:
        vis &= j >= i - window
    if block_mask is not None:
        vis &= np.asarray(block_mask)[i // block, j // block] != 0
    return vis


def rescaled_rows(q, k, scale, vis, rows, margin=0.25):
    """Number of rows (of one head; q, k fp64 [N, d]) whose largest visible
    scaled score, in log2 units, exceeds the largest one in the 128-key block
    that holds the row's first visible key by more than 8 + margin.  The
    kernels visit keys in blocks of 64 or 128 from that block on and rescale
    only when the row maximum grows by more than 8 log2 units, so every such
    row rescales an accumulator that already holds that first block's
    weights (a nonzero output)."""
    t = scale * LOG2E * (q[rows] @ k.T)
    t = np.where(vis, t, -np.inf)
    has = vis.any(axis=1)
    first = np.argmax(vis, axis=1)
    blk = np.arange(k.shape[0])[None, :] // 128 == (first // 128)[:, None]
    m_first = np.where(blk, t, -np.inf).max(axis=1)
    m_all = t.max(axis=1)
    grow = np.where(has, m_all - np.where(has, m_first, 0.0), 0.0)
    return int((grow > 8.0 + margin).sum())


def o_bound_bf16(o_ref, a_ref):
    """Per-element O tolerance where |O| can exceed 4 (dropout, or inputs whose
    weights concentrate on few keys): the two bf16 roundings (the weights fed
    to the product and O itself), each at most 2^-9 relative, with a factor two
    of margin, or 1e-2 where larger; a_ref = sum_j w_ij |v_jc| with the weights
    w the product applies (the oracle run on |V|)."""
    return np.maximum(TOL_O_ABS, 2.0 ** -8 * (np.abs(o_ref) + a_ref))
