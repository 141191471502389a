"""Seeded, platform-independent synthetic inputs for attention workloads.

This module only draws random numbers; it holds none of the attention
arithmetic, so the CUDA path and the fp64 oracle can both be fed from it.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based stream -- output
``e`` of stream ``(seed, tensor)`` is the SplitMix64 finaliser applied to
``key + (e + 1) * GAMMA`` -- then the Box-Muller transform in fp64, rounded to
fp32 and then to bf16 with round-to-nearest-even.  Only 64-bit integer
arithmetic and IEEE fp64 are used, so an x86 host and an Arm host draw the
same bits (up to a last-ulp libm difference in log/cos/sin that the fp32 and
bf16 roundings almost always absorb).

Streams: tensor ids Q=0, K=1, V=2, dO=3, key-padding lengths=4, block masks=5.  A workload
with index ``k`` in the configuration list uses seed ``1000 + k``.
"""
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM = {"Q": 0, "K": 1, "V": 2, "dO": 3, "kv_len": 4, "block_mask": 5}
SEED_BASE = 1000


def _mix64(z):
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed, stream):
    with np.errstate(over="ignore"):
        k = _mix64(np.array([np.uint64(seed) * GAMMA], dtype=np.uint64))
        k = _mix64(k + np.uint64(stream) * _M2 + GAMMA)
    return k[0]


def uint64_stream(seed, stream, n, start=0):
    """Outputs start .. start+n-1 of the counter-based stream (seed, stream)."""
    key = _stream_key(seed, stream)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(key + ctr * GAMMA)


def normal_f64(seed, stream, n):
    """n iid N(0,1) fp64 draws (Box-Muller on pairs of 53-bit uniforms)."""
    npairs = (n + 1) // 2
    u = uint64_stream(seed, stream, 2 * npairs)
    scale = 1.0 / 9007199254740992.0  # 2^-53
    u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale  # (0, 1]
    u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * scale          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def f32_to_bf16_bits(x):
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def normal_bf16_bits(seed, stream, shape):
    """iid N(0,1) values rounded fp64 -> fp32 -> bf16, as uint16 bit patterns."""
    n = int(np.prod(shape))
    return f32_to_bf16_bits(normal_f64(seed, stream, n).astype(np.float32)).reshape(shape)


def e4m3_bits_to_f64(bits):
    """Exact values of e4m3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal; 0x7F/0xFF are NaN, no infinities)."""
    c = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


_E4M3_POS = e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))  # codes 0 .. 0x7E, ascending


def f32_to_e4m3_bits(x):
    """Round values to e4m3 codes: nearest, ties to the even code, saturating at
    +-448 (the largest finite value)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(a - _E4M3_POS[lo])
    d_hi = np.abs(_E4M3_POS[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def normal_e4m3_bits(seed, stream, shape):
    """iid N(0,1) values rounded fp64 -> e4m3 codes (uint8)."""
    n = int(np.prod(shape))
    return f32_to_e4m3_bits(normal_f64(seed, stream, n)).reshape(shape)


def kv_lengths(seed, B, lo, hi):
    """Per-sequence key lengths, uniform integers in [lo, hi] (int32 [B])."""
    u = uint64_stream(seed, STREAM["kv_len"], B)
    return (np.uint64(lo) + u % np.uint64(hi - lo + 1)).astype(np.int32)


def block_mask(seed, nb, density, diagonal=True):
    """Random [nb, nb] uint8 block mask: each (query block, key block) pair is
    kept with probability `density`; `diagonal` keeps every diagonal pair."""
    u = uint64_stream(seed, STREAM["block_mask"], nb * nb)
    uni = (u >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    m = (uni < density).astype(np.uint8).reshape(nb, nb)
    if diagonal:
        np.fill_diagonal(m, 1)
    return m


def attention_inputs(seed, B, H, N, d, with_dout=True):
    """bf16 bit patterns of Q, K, V (and dO) for one workload, each [B,H,N,d]."""
    names = ("Q", "K", "V", "dO") if with_dout else ("Q", "K", "V")
    return {nm: normal_bf16_bits(seed, STREAM[nm], (B, H, N, d)) for nm in names}


def _round_to(x, fmt):
    if fmt == "bf16":
        return f32_to_bf16_bits(np.asarray(x, np.float64).astype(np.float32))
    if fmt == "e4m3":
        return f32_to_e4m3_bits(x)
    raise ValueError("fmt must be 'bf16' or 'e4m3'")


def shaped_key_inputs(seed, B, H, N, d, gain=None, levels=None, noise=1.0, v_shift=0.0,
                      fmt="bf16", with_dout=True):
    """Inputs whose attention scores rise along the key axis, so that a row's
    running maximum grows by many units after the first key blocks.

    The draws are those of `attention_inputs` (same seed and streams); only
    their shape changes:
      - `gain` (fp64 [N] or None): key row j is multiplied by gain[j];
      - `levels` (fp64 [N] or None): column 0 of every query row is set to 1,
        column 0 of key row j to levels[j], and the other key columns are
        multiplied by `noise`; the score of any query with key j is then
        levels[j] plus a term of spread `noise * sqrt(d - 1)` (before the
        caller's scale);
      - `v_shift`: added to every value of V (a nonzero mean makes any
        weighted average of V rows differ from zero).
    Values are rounded to bf16 (uint16 bits) or to e4m3 codes (uint8; fmt =
    "e4m3": Q, K, V only)."""
    names = ("Q", "K", "V", "dO") if (with_dout and fmt == "bf16") else ("Q", "K", "V")
    shape = (B, H, N, d)
    x = {nm: normal_f64(seed, STREAM[nm], B * H * N * d).reshape(shape) for nm in names}
    if gain is not None:
        x["K"] = x["K"] * np.asarray(gain, np.float64).reshape(1, 1, N, 1)
    if levels is not None:
        x["K"] = x["K"] * noise
        x["K"][..., 0] = np.asarray(levels, np.float64).reshape(1, 1, N)
        x["Q"][..., 0] = 1.0
    x["V"] = x["V"] + v_shift
    return {nm: _round_to(v, fmt) for nm, v in x.items()}
