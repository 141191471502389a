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

    def __init__(self, seed, B, H, N, d, kv_range=None, with_dout=True, device="cuda:0"):
        import torch
        self.B, self.H, self.N, self.d = B, H, N, d
        self.scale = 1.0 / math.sqrt(d)
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
