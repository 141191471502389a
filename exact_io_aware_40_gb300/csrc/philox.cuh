// philox.cuh -- dropout decisions from the counter-based generator
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11), written here from the paper's definition.
//
// Dropout on the attention weights (the study notes list it among the steps
// fused into the kernel, section "Kernel融合"): P_ij is kept with probability
// q and scaled by 1/q.  The decision for (batch b, head h, query i, key j)
// reads the generator at counter (j / 8, i, h, b) with the 64-bit seed as key;
// the call's 128 bits are eight 16-bit values, value j % 8 (the low half of
// word (j % 8) / 2 first) deciding key j: kept iff value >= thr, with the
// integer threshold thr = floor(p * 65536) and q = (65536 - thr) / 65536.
#pragma once
#include <cstdint>

namespace fa {

// One Philox4x32-10 call: ten rounds of two 32 x 32 -> 64-bit products whose
// high halves are XORed into the other two counter words together with the
// round key; the key advances by two Weyl constants per round.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t m0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t m1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(m1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(m0 >> 32) ^ c3 ^ k1;
    c1 = static_cast<uint32_t>(m1);
    c3 = static_cast<uint32_t>(m0);
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep bits of 8 consecutive keys j0 .. j0 + 7 (j0 a multiple of 8) of query
// i: bit t <-> key j0 + t.
__device__ __forceinline__ uint32_t keep8(uint32_t j0, uint32_t i, uint32_t h, uint32_t b,
                                          uint32_t seed_lo, uint32_t seed_hi, uint32_t thr) {
  const uint4 r = philox4x32_10(j0 >> 3, i, h, b, seed_lo, seed_hi);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  uint32_t m = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    m |= static_cast<uint32_t>((w[t] & 0xffffu) >= thr) << (2 * t);
    m |= static_cast<uint32_t>((w[t] >> 16) >= thr) << (2 * t + 1);
  }
  return m;
}

// Keep bits of 32 consecutive keys j0 .. j0 + 31 (j0 a multiple of 8) of
// query i: bit t <-> key j0 + t.
__device__ __forceinline__ uint32_t keep32(uint32_t j0, uint32_t i, uint32_t h, uint32_t b,
                                           uint32_t seed_lo, uint32_t seed_hi, uint32_t thr) {
  uint32_t m = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) m |= keep8(j0 + 8 * g, i, h, b, seed_lo, seed_hi, thr) << (8 * g);
  return m;
}

// The transposed case: a warp whose lane l holds key kw0 + l (kw0 a multiple
// of 32) and needs the keep bits of 64 consecutive queries i0 .. i0 + 63.
// Returns, in every lane, the 64 bits of its own key (bit c <-> query i0 + c).
// Each lane makes 8 generator calls -- key group g = l % 4 (8 keys) for the
// queries i0 + l / 4 + 8 t, t = 0..7 -- and the bits are exchanged with 16
// shuffles; all 32 lanes must call this together.
__device__ __forceinline__ uint64_t keep64_transposed(uint32_t kw0, uint32_t i0, uint32_t h,
                                                      uint32_t b, uint32_t seed_lo,
                                                      uint32_t seed_hi, uint32_t thr) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t g = lane & 3u, cl = lane >> 2;
  uint32_t word[2] = {0u, 0u};  // byte t % 4 of word t / 4: keys 8g..8g+7 for query cl + 8t
#pragma unroll
  for (int t = 0; t < 8; ++t)
    word[t >> 2] |= keep8(kw0 + 8 * g, i0 + cl + 8 * t, h, b, seed_lo, seed_hi, thr)
                    << (8 * (t & 3));
  const uint32_t my_g = lane >> 3, my_bit = lane & 7u;
  uint64_t m = 0;
#pragma unroll
  for (int c7 = 0; c7 < 8; ++c7) {
    const int src = (c7 << 2) | static_cast<int>(my_g);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const uint32_t v = __shfl_sync(0xffffffffu, word[w], src);
#pragma unroll
      for (int byte = 0; byte < 4; ++byte) {
        const int c = c7 + 8 * (4 * w + byte);  // query column
        m |= static_cast<uint64_t>((v >> (8 * byte + my_bit)) & 1u) << c;
      }
    }
  }
  return m;
}

// The same for 32 consecutive queries i0 .. i0 + 31: every lane gets the 32
// bits of its own key kw0 + lane (bit c <-> query i0 + c).  Lane l makes 4
// generator calls -- key group l % 4 for the queries i0 + l / 4 + 8 t,
// t = 0..3 -- and the bits are exchanged with 8 shuffles; all 32 lanes must
// call this together.
__device__ __forceinline__ uint32_t keep32_transposed(uint32_t kw0, uint32_t i0, uint32_t h,
                                                      uint32_t b, uint32_t seed_lo,
                                                      uint32_t seed_hi, uint32_t thr) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t g = lane & 3u, cl = lane >> 2;
  uint32_t word = 0u;  // byte t: keys 8g..8g+7 for query cl + 8t
#pragma unroll
  for (int t = 0; t < 4; ++t)
    word |= keep8(kw0 + 8 * g, i0 + cl + 8 * t, h, b, seed_lo, seed_hi, thr) << (8 * t);
  const uint32_t my_g = lane >> 3, my_bit = lane & 7u;
  uint32_t m = 0;
#pragma unroll
  for (int c7 = 0; c7 < 8; ++c7) {
    const uint32_t v = __shfl_sync(0xffffffffu, word, (c7 << 2) | static_cast<int>(my_g));
#pragma unroll
    for (int t = 0; t < 4; ++t) m |= ((v >> (8 * t + my_bit)) & 1u) << (c7 + 8 * t);
  }
  return m;
}

}  // namespace fa
