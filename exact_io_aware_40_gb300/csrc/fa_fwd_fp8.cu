// fa_fwd_fp8.cu -- forward pass of exact attention with 8-bit floating-point
// (e4m3) Q, K and V, d = 128, on sm_103a.
//
// The method is unchanged (tiling, masked online softmax, O accumulated on
// chip; study notes "FlashAttention学习笔记", section "分块计算整体流程
// (Tiling)"); the pages name FP8 as the direction the method takes next
// (bxzpzcl.cn article, section "量化技术深度融合").  Inputs are e4m3 codes
// with one fp32 dequantisation factor per tensor (value = factor * code), so
// S = scale * (dq Q8)(dk K8)^T and O = softmax(S) (dv V8); the products run on
// the tensor cores in kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate), at twice
// the bf16 rate.  P enters the PV product rounded to e4m3, and O is divided
// by the row sum of the unrounded P (the sum L uses as well): the weights
// applied to V then differ from P by the e4m3 rounding alone, at most 2^-4 of
// each, so |O - O_exact| <= 2^-4 sum_j p_j |v_j|.  (Summing the rounded
// weights instead would take three more conversions per pair of elements, and
// the softmax, not the tensor pipe, bounds this kernel.)  O is written in
// bf16.
// e4m3 holds normal values from 2^-6 to 448 only: weights taken relative to
// the row maximum alone would fall into its subnormal range, or to zero, once
// they are 2^-7 of the maximum or less, and hundreds of such keys can carry
// much of a row's weight after its maximum has jumped.  So P is computed as
// 2^(s - m + 6) (s, m in log2 units): weights down to 2^-12 of the maximum
// stay normal, and with the rescale threshold at 2 the largest weight is at
// most 2^8 = 256 < 448.  The common factor 2^6 cancels in O and is taken out
// of L.
//
// GB300 mapping: one 128-row query block per CTA, 128-key blocks.  With d =
// 128 one row of Q, K or V^T is 128 bytes, one 128-byte swizzle atom, and
// every operand is K-major: S = Q K_j^T reads Q and K_j along d; PV reads P
// (queries x keys) along the keys and V_j^T (d x keys, from a transposed copy
// of V that fa_fwd_fp8 writes into its workspace first) along the keys too.
//   warp 0     TMA producer (Q once; K_j and V_j^T through 2-stage rings)
//   warp 1     tcgen05 issuer: S_j into one of two TMEM buffers (columns 0,
//              128), then O += P_{j-1} V_{j-1} (O at column 256)
//   warps 2-5  softmax (thread = query row = TMEM lane): P as e4m3 into one
//              of two shared-memory tiles, conditional O rescale, epilogue.
#include <type_traits>

#include "kernels.h"
#include "masks.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBR = 128;      // query rows per CTA (MMA M)
constexpr int kBC = 128;      // keys per block (MMA N of S, K of PV)
constexpr int kD = 128;       // head dimension
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 2.0f;  // log2 units: rescale O only if m grows by > 2
constexpr float kPOffset = 6.0f;           // P = 2^(s - m + kPOffset), at most 2^8
constexpr float kLn2 = 0.693147180559945309f;

constexpr int kTile8 = 128 * 128;  // 128 rows x 128 one-byte elements
constexpr int kSt = 2;             // K and V^T ring depth
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile8;
constexpr int kOffV = kOffK + kSt * kTile8;  // V^T tiles: d rows x 128 keys
constexpr int kOffP = kOffV + kSt * kTile8;  // P as e4m3, two buffers
constexpr int kOffO = kOffP + 2 * kTile8;    // O staging: two 64-column bf16 atoms
constexpr int kOffBar = kOffO + 2 * kBR * 128;
// q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], o_done, drain
constexpr int kNumBar = 1 + 4 * kSt + 2 + 2 + 1 + 1;
constexpr int kOffMisc = kOffBar + kNumBar * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColO = 256;

__device__ __forceinline__ uint32_t s_col(int b) { return b ? 128u : 0u; }

__device__ __forceinline__ bool bar_and_128(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id)
      : "memory");
  return r != 0;
}

// Descriptors of the four k-steps of a K-major 8-bit operand with 128-byte
// rows: step k covers elements [32k, 32k+32) of the row, byte offset 32 k
// inside the swizzled row.
__device__ __forceinline__ void kmaj8_steps(uint32_t base, uint64_t (&d)[4]) {
  const uint64_t d0 = sdesc_sw128(base, 16, 1024);
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = sdesc_add(d0, 32u * k);
}

__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt,
                      const __grid_constant__ CUtensorMap tmO, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sQ = sb + kOffQ, sK = sb + kOffK, sV = sb + kOffV, sP = sb + kOffP;
  const uint32_t sO = sb + kOffO;
  const uint32_t bar0 = sb + kOffBar;
  const uint32_t bar_q = bar0;
  auto bar_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (1 + kSt + s); };
  auto bar_vfull = [&](int s) { return bar0 + 8u * (1 + 2 * kSt + s); };
  auto bar_vempty = [&](int s) { return bar0 + 8u * (1 + 3 * kSt + s); };
  const uint32_t bar_sfull0 = bar0 + 8u * (1 + 4 * kSt);
  const uint32_t bar_pfull0 = bar_sfull0 + 16u;
  const uint32_t bar_odone = bar_pfull0 + 16u;
  const uint32_t bar_drain = bar_odone + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Longest query blocks (causal) first, in groups of ranks, head-major inside
  // a group.
  int bh, qt;
  cta_tile(static_cast<int>(blockIdx.x), a.n_qtiles, a.BH, a.tile_group, &bh, &qt);
  qt = a.n_qtiles - 1 - qt;
  const int q0 = qt * kBR;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  int T = (kv_limit + kBC - 1) / kBC;
  if (a.causal) T = min(T, qt + 1);

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kSt; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), 1);
    }
    mbar_init(bar_sfull0, 1);
    mbar_init(bar_sfull0 + 8, 1);
    mbar_init(bar_pfull0, 4);
    mbar_init(bar_pfull0 + 8, 4);
    mbar_init(bar_odone, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{a.err, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar_q, kTile8);
      tma_load_3d(sQ, &tmQ, 0, q0, bh, bar_q, pol_q);
      int last_k[kSt], last_v[kSt];
      for (int s = 0; s < kSt; ++s) last_k[s] = last_v[s] = -1;
      for (int j = 0; j < T; ++j) {
        const int st = j % kSt;
        if (j >= kSt && !mbar_wait(bar_kempty(st), ((j / kSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_kfull(st), kTile8);
        tma_load_3d(sK + st * kTile8, &tmK, 0, j * kBC, bh, bar_kfull(st), pol_kv);
        last_k[st] = j;
        if (j >= kSt && !mbar_wait(bar_vempty(st), ((j / kSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_vfull(st), kTile8);
        // V_j^T: the 128 keys of block j (inner coordinate) for all d rows.
        tma_load_3d(sV + st * kTile8, &tmVt, j * kBC, 0, bh, bar_vfull(st), pol_kv);
        last_v[st] = j;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar_q, 0);
        for (int s = 0; s < kSt; ++s) {
          if (last_k[s] >= 0) mbar_wait_drain(bar_kfull(s), (last_k[s] / kSt) & 1);
          if (last_v[s] >= 0) mbar_wait_drain(bar_vfull(s), (last_v[s] / kSt) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idS = idesc_e4m3(kBR, kBC);
      constexpr uint32_t idO = idesc_e4m3(kBR, kD);
      static_assert(kD == 128 && kBC == 128, "four 32-element k-steps per product");
      uint64_t aQ[4];  // the resident Q tile's descriptors, built once
      kmaj8_steps(sQ, aQ);
      bool ok = mbar_wait(bar_q, 0, ab);
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1, vs = jj % kSt;
        if (!mbar_wait(bar_pfull0 + 8u * bb, (jj >> 1) & 1, ab)) return false;
        if (!mbar_wait(bar_vfull(vs), (jj / kSt) & 1, ab)) return false;
        tc_fence_after();
        uint64_t a[4], b[4];
        kmaj8_steps(sP + bb * kTile8, a);
        kmaj8_steps(sV + vs * kTile8, b);
        mma_ss_f8_x4(tmem + kColO, a, b, idO, jj > 0 ? 1u : 0u);
        mma_commit(bar_odone);
        mma_commit(bar_vempty(vs));
        return true;
      };
      for (int j = 0; ok && j < T; ++j) {
        const int bb = j & 1, ks = j % kSt;
        // S_j overwrites S_{j-2}'s buffer, and the softmax then overwrites
        // P_{j-2}'s tile: both are free once PV_{j-2} has completed.
        if (j >= 2 && !mbar_wait(bar_odone, (j - 2) & 1, ab)) { ok = false; break; }
        if (!mbar_wait(bar_kfull(ks), (j / kSt) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        {
          uint64_t b[4];
          kmaj8_steps(sK + ks * kTile8, b);
          mma_ss_f8_x4(tmem + s_col(bb), aQ, b, idS, 0u);
        }
        mma_commit(bar_sfull0 + 8u * bb);
        mma_commit(bar_kempty(ks));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(T - 1);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;           // TMEM lanes [32*quarter, +32)
    const int row = quarter * 32 + lane;    // row of the tile = TMEM lane
    const int grow = q0 + row;              // query index
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_run = -INFINITY;                // running max, log2 units (scaled)
    float l_run = 0.f;                      // row sum of P
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int bb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull0 + 8u * bb, (j >> 1) & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + s_col(bb) + 32 * c, sr[c]);
      tmem_wait_ld();
      const int key0 = j * kBC;
      const bool need_mask = (key0 + kBC > kv_limit) || (a.causal && key0 + kBC - 1 > q0);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = key0 + 32 * c + e;
            const bool keep = (key < kv_limit) & !((a.causal != 0) & (key > grow));
            sr[c][e] = keep ? sr[c][e] : __float_as_uint(-INFINITY);
          }
      }
      float mxp[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mxp[t] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mxp[e & 7] = fmaxf(mxp[e & 7], __uint_as_float(sr[c][e]));
      const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                             fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      const float m_cand = fmaxf(m_run, mx * a.scale_log2);
      const bool grow_max = m_cand > m_run + kRescaleThreshold;
      const float m_new = grow_max ? m_cand : m_run;
      const float alpha = grow_max ? ex2(m_run - m_new) : 1.f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new - kPOffset;
      // P = 2^(s * scale * log2e - m + 6), rounded to e4m3 into this row of P's
      // shared-memory tile (the 128-byte swizzle TMA and the tensor core use:
      // 16-byte chunk t of row r at chunk t ^ (r % 8)).
      const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2);
      const uint64_t nm2 = f2_pack(-m_use, -m_use);
      uint64_t se[2] = {0ull, 0ull};
      uint8_t* prow = smem + kOffP + bb * kTile8 + row * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[8];  // 32 keys = 32 bytes = two 16-byte chunks
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])),
                           scl2, nm2),
                    t0, t1);
          const float p0 = ex2(t0), p1 = ex2(t1);
          const uint32_t q8 = pack_e4m3(p0, p1);
          if (e & 1)
            w[e >> 1] |= q8 << 16;
          else
            w[e >> 1] = q8;
          se[e & 1] = f2_add(se[e & 1], f2_pack(p0, p1));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int chunk = 2 * c + h;
          const int phys = chunk ^ (row & 7);
          *reinterpret_cast<uint4*>(prow + phys * 16) =
              make_uint4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
        }
      }
      // The tensor core reads P through the async proxy.
      fence_proxy_async_smem();
      float u0, u1;
      f2_unpack(f2_add(se[0], se[1]), u0, u1);
      l_run = l_run * alpha + (u0 + u1);
      m_run = m_new;
      if (j > 0 && __any_sync(0xffffffffu, grow_max)) {
        // O holds P_0..P_{j-1} V; rescale it once PV_{j-1} has landed (only
        // PV_{j-1} can be pending: S_j was issued after PV_{j-2} completed).
        if (!__all_sync(0xffffffffu, mbar_wait(bar_odone, (j - 1) & 1, ab))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + kColO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tl + kColO + 32 * c, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull0 + 8u * bb);
    }
    if (ok && T > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_odone, (T - 1) & 1, ab));
      tc_fence_after();
    }
    ok = bar_and_128(1, ok && *abort_flag == 0);
    if (ok) {
      // ---------------------------------------------------------- epilogue
      const float inv_l = l_run > 0.f ? a.out_scale / l_run : 0.f;
      if (grow < a.N) {
        const float Lv = l_run > 0.f ? (m_run - kPOffset + log2f(l_run)) * kLn2 : -INFINITY;
        a.L[static_cast<long long>(bh) * a.N + grow] = Lv;
      }
      // O * dv / lh -> bf16 -> staging tile (128-byte swizzle, two 64-column
      // atoms) -> TMA store (rows >= N are clipped).
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        if (T > 0) {
          tmem_ld32(tl + kColO + 32 * c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        const int atom = (32 * c) / 64;
        const int chunk0 = ((32 * c) % 64) / 8;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * t + 0]) * inv_l, __uint_as_float(o[8 * t + 1]) * inv_l);
          v.y = pack_bf16(__uint_as_float(o[8 * t + 2]) * inv_l, __uint_as_float(o[8 * t + 3]) * inv_l);
          v.z = pack_bf16(__uint_as_float(o[8 * t + 4]) * inv_l, __uint_as_float(o[8 * t + 5]) * inv_l);
          v.w = pack_bf16(__uint_as_float(o[8 * t + 6]) * inv_l, __uint_as_float(o[8 * t + 7]) * inv_l);
          const int phys = (chunk0 + t) ^ (row & 7);
          *reinterpret_cast<uint4*>(smem + kOffO + atom * (kBR * 128) + row * 128 + phys * 16) = v;
        }
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (warp == 2 && lane == 0) {
        for (int c = 0; c < 2; ++c) tma_store_3d(&tmO, sO + c * (kBR * 128), c * 64, q0, bh);
        bulk_commit();
        bulk_wait0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// V [BH, N, 128] e4m3 -> V^T [BH, 128, Npad]; keys in [N, Npad) are zero.
// One CTA per 128 keys of one head, 256 threads, through a shared tile.
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint8_t* __restrict__ V,
                                                          uint8_t* __restrict__ Vt, int N, int Npad) {
  __shared__ uint8_t t[128][132];  // [key][d], padded rows
  const int k0 = static_cast<int>(blockIdx.x) * 128;
  const long long bh = blockIdx.y;
  const uint8_t* src = V + bh * static_cast<long long>(N) * kD;
  for (int w = threadIdx.x; w < 128 * 32; w += 256) {
    const int key = w >> 5, c4 = (w & 31) * 4;
    uint32_t v = 0u;
    if (k0 + key < N) v = *reinterpret_cast<const uint32_t*>(src + static_cast<long long>(k0 + key) * kD + c4);
    *reinterpret_cast<uint32_t*>(&t[key][c4]) = v;
  }
  __syncthreads();
  uint8_t* dst = Vt + bh * static_cast<long long>(kD) * Npad;
  for (int w = threadIdx.x; w < 128 * 32; w += 256) {
    const int dd = w >> 5, k4 = (w & 31) * 4;
    if (k0 + k4 >= Npad) continue;
    const uint32_t v = static_cast<uint32_t>(t[k4][dd]) | (static_cast<uint32_t>(t[k4 + 1][dd]) << 8) |
                       (static_cast<uint32_t>(t[k4 + 2][dd]) << 16) |
                       (static_cast<uint32_t>(t[k4 + 3][dd]) << 24);
    *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(dd) * Npad + k0 + k4) = v;
  }
}

}  // namespace

cudaError_t launch_transpose_v8(const void* V, void* Vt, int BH, int N, int Npad,
                                cudaStream_t stream) {
  const dim3 grid((Npad + 127) / 128, BH);
  if (grid.x == 0 || BH <= 0) return cudaSuccess;
  if (BH > 65535) return cudaErrorInvalidConfiguration;
  transpose_v_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(V),
                                               static_cast<uint8_t*>(Vt), N, Npad);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVt,
                           const CUtensorMap& tmO, const FwdArgs& a, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = static_cast<long long>(a.n_qtiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdArgs ag = a;
  // 512 TMEM columns: one CTA per SM; K and V^T of a head, e4m3
  ag.tile_group = tile_group(a.causal != 0, a.n_qtiles, a.BH, 1, 2ll * a.N * 128);
  fa_fwd_fp8_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tmQ, tmK, tmVt,
                                                                                 tmO, ag);
  return cudaGetLastError();
}

}  // namespace fa
