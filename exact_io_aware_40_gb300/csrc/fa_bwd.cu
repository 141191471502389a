// fa_bwd.cu -- backward pass of exact attention on sm_103a.
//
// Method: the forward pass keeps only O and the row logsumexp L; the backward
// pass recomputes the attention matrix tile by tile from L instead of reading
// a stored N x N matrix (fmread.com summary, section 三.2 "反向传播优化";
// abstract of "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness").  The pages state no gradient formulas; the ones used are the
// textbook gradient of softmax attention:
//   P = exp(scale * Q K^T - L),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D) with D_i = dO_i . O_i,  dQ = scale dS K,  dK = scale dS^T Q.
//
// GB300 mapping: one CTA per 128-key block j of one (batch, head); the loop
// runs over 128-row query blocks i (the study notes' K/V-outer loop order,
// section "分块计算整体流程(Tiling)"), so dK_j and dV_j accumulate in TMEM:
//   warp 0      producer: K_j, V_j once; Q_i, dO_i per step through a 2-stage
//               TMA ring; L_i (pre-multiplied by log2 e) and D_i into smem.
//   warp 1      tcgen05 issuer: S^T = K_j Q_i^T and dP^T = V_j dO_i^T (keys on
//               TMEM lanes), dV += P^T dO_i and dK += dS^T Q_i (A from TMEM),
//               dQ_i = dS K_j (A from smem).
//   warps 4-7   compute: thread = key row; P^T = exp2(S^T scale log2e - L log2e)
//               -> bf16 into TMEM; dS^T = P^T o (dP^T - D) -> bf16 into TMEM
//               (for dK) and into swizzled smem (for dQ); final dK, dV stores.
//   warps 8-11  dQ drain: thread = query row; TMEM -> fp32 vector reductions
//               into the dQ accumulator in global memory.
// TMEM (512 columns): S^T 0-127 (P^T over 0-63), dP^T 128-255 (dS^T over
// 128-191), dV 256.., dK 256+d..; dQ_i lives in 384-447 for d = 64 and reuses
// the dP^T columns for d = 128 (the dK product has read dS^T by then).
#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBK = 128;       // keys per CTA (MMA M of the key-row products)
constexpr int kBQ = 128;       // query rows per step
constexpr int kThreads = 384;
constexpr int kQSt = 2;        // Q/dO ring depth
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kErrLayout = 3;  // device error code: shared-memory base misaligned

template <int HD>
struct BCfg {
  static constexpr int kAtoms = HD / 64;
  static constexpr int kAtomBytes = 128 * 128;            // 128 rows x 128 B
  static constexpr int kTileBytes = kAtoms * kAtomBytes;  // 128 rows x d bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // kQSt stages
  static constexpr int kOffdO = kOffQ + kQSt * kTileBytes;         // kQSt stages
  static constexpr int kOffdS = kOffdO + kQSt * kTileBytes;        // 128 x 128 bf16
  static constexpr int kOffLD = kOffdS + 2 * kAtomBytes;           // kQSt x (L2[128], D[128])
  static constexpr int kOffBar = kOffLD + kQSt * 1024;
  // kv_full, qdo_full[2], qdo_empty[2], ld_full[2], s_full, dp_full, p_full,
  // ds_full, dq_full, dq_empty, dsm_empty, final, drain
  static constexpr int kNumBar = 1 + 3 * kQSt + 9;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 16;
  static constexpr int kSlack = (kUsed + 1024 <= 232448) ? 1024 : 0;
  static constexpr int kSmemBytes = kUsed + kSlack;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 256 + HD;
  static constexpr uint32_t kColdQ = HD == 64 ? 384 : 128;
  static constexpr bool kDqInDp = HD != 64;
};

__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const BwdArgs a) {
  using C = BCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  if (pad > static_cast<uint32_t>(C::kSlack)) {  // cannot happen with a 1 KB-aligned window
    if (threadIdx.x == 0) atomicCAS(a.err, 0, kErrLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sK = sb + C::kOffK, sV = sb + C::kOffV;
  const uint32_t sQ = sb + C::kOffQ, sdO = sb + C::kOffdO, sdS = sb + C::kOffdS;
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  const uint32_t bar0 = sb + C::kOffBar;
  const uint32_t bar_kv = bar0;
  auto bar_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (1 + kQSt + s); };
  auto bar_ld_full = [&](int s) { return bar0 + 8u * (1 + 2 * kQSt + s); };
  const uint32_t bar_s = bar0 + 8u * (1 + 3 * kQSt);
  const uint32_t bar_dp = bar_s + 8, bar_p = bar_s + 16, bar_ds = bar_s + 24;
  const uint32_t bar_dq_full = bar_s + 32, bar_dq_empty = bar_s + 40, bar_dsm_empty = bar_s + 48;
  const uint32_t bar_final = bar_s + 56, bar_drain = bar_s + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Head-major order (the CTAs in flight share one head's Q/dO in L2); small kt
  // (most work under causal) first.
  const int bh = static_cast<int>(blockIdx.x / a.n_ktiles);
  const int kt = static_cast<int>(blockIdx.x % a.n_ktiles);
  const int k0 = kt * kBK;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  const int i_start = a.causal ? kt : 0;
  const int n_iter = (k0 >= kv_limit) ? 0 : a.n_qtiles - i_start;

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < kQSt; ++s) {
      mbar_init(bar_qdo_full(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
      mbar_init(bar_ld_full(s), 32);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 4);
    mbar_init(bar_ds, 4);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_empty, 4);
    mbar_init(bar_dsm_empty, 1);
    mbar_init(bar_final, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
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
    // -------------------------------------------------------------- producer
    if (n_iter > 0) {
      uint64_t pol_kv = 0, pol_q = 0;
      if (lane == 0) {
        pol_kv = policy_evict_first();
        pol_q = policy_evict_last();  // Q_i, dO_i are re-read by every key block
        mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c) {
          tma_load_3d(sK + c * C::kAtomBytes, &tmK, c * 64, k0, bh, bar_kv, pol_kv);
          tma_load_3d(sV + c * C::kAtomBytes, &tmV, c * 64, k0, bh, bar_kv, pol_kv);
        }
      }
      int last[kQSt] = {-1, -1};
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % kQSt;
        const int q0 = (i_start + it) * kBQ;
        if (it >= kQSt &&
            !__all_sync(0xffffffffu, mbar_wait(bar_qdo_empty(st), ((it / kQSt) & 1) ^ 1, ab)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_qdo_full(st), 2 * C::kTileBytes);
          for (int c = 0; c < C::kAtoms; ++c) {
            tma_load_3d(sQ + st * C::kTileBytes + c * C::kAtomBytes, &tmQ, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
            tma_load_3d(sdO + st * C::kTileBytes + c * C::kAtomBytes, &tmdO, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
          }
        }
        last[st] = it;
        float* L2 = sLD + st * 256;
        float* Dv = L2 + 128;
        const long long rbase = static_cast<long long>(bh) * a.N;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = lane * 4 + e;
          const int q = q0 + r;
          L2[r] = q < a.N ? a.L[rbase + q] * kLog2e : 0.f;
          Dv[r] = q < a.N ? a.D[rbase + q] : 0.f;
        }
        mbar_arrive(bar_ld_full(st));
      }
      if (lane == 0 && *abort_flag) {
        mbar_wait_drain(bar_kv, 0);
        for (int s = 0; s < kQSt; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar_qdo_full(s), (last[s] / kQSt) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);   // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(128, HD, false, true);    // dV, dK (B MN-major)
      constexpr uint32_t idQ = idesc_bf16(128, HD, true, true);      // dQ (A, B MN-major)
      auto kmaj = [](uint32_t base, int k) {  // K-major operand, step k of 16 columns
        return sdesc_sw128(base + (k >> 2) * C::kAtomBytes + (k & 3) * 32, 16, 1024);
      };
      auto mnmaj = [](uint32_t base, int k) {  // MN-major operand, step k of 16 rows
        return sdesc_sw128(base + k * 2048, C::kAtomBytes, 1024);
      };
      auto issue_s = [&](int it) {
        const uint32_t q = sQ + (it % kQSt) * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tmem + C::kColS, kmaj(sK, k), kmaj(q, k), idS, k > 0 ? 1u : 0u);
        mma_commit(bar_s);
      };
      auto issue_dp = [&](int it) {
        const uint32_t g = sdO + (it % kQSt) * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tmem + C::kColdP, kmaj(sV, k), kmaj(g, k), idS, k > 0 ? 1u : 0u);
        mma_commit(bar_dp);
      };
      bool ok = mbar_wait(bar_kv, 0, ab) && mbar_wait(bar_qdo_full(0), 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int st = it % kQSt;
        const bool more = it + 1 < n_iter;
        // dV += P^T dO_i
        if (!(ok = mbar_wait(bar_p, it & 1, ab))) break;
        tc_fence_after();
        {
          const uint32_t g = sdO + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < kBQ / 16; ++k)
            mma_ts(tmem + C::kColdV, tmem + C::kColS + k * 8, mnmaj(g, k), idKV,
                   (it > 0 || k > 0) ? 1u : 0u);
        }
        // S^T of the next step can overwrite P^T: the product above read it first.
        if (more) {
          const int st1 = (it + 1) % kQSt;
          if (!(ok = mbar_wait(bar_qdo_full(st1), ((it + 1) / kQSt) & 1, ab))) break;
          tc_fence_after();
          issue_s(it + 1);
        }
        // dK += dS^T Q_i
        if (!(ok = mbar_wait(bar_ds, it & 1, ab))) break;
        tc_fence_after();
        {
          const uint32_t q = sQ + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < kBQ / 16; ++k)
            mma_ts(tmem + C::kColdK, tmem + C::kColdP + k * 8, mnmaj(q, k), idKV,
                   (it > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar_qdo_empty(st));
        // dQ_i = dS K_j
        if (!C::kDqInDp && it > 0) {
          if (!(ok = mbar_wait(bar_dq_empty, (it - 1) & 1, ab))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_ss(tmem + C::kColdQ, mnmaj(sdS, k), mnmaj(sK, k), idQ, k > 0 ? 1u : 0u);
        mma_commit(bar_dq_full);
        mma_commit(bar_dsm_empty);
        if (more) {
          if (C::kDqInDp) {
            if (!(ok = mbar_wait(bar_dq_empty, it & 1, ab))) break;
            tc_fence_after();
          }
          issue_dp(it + 1);
        }
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // -------------------------------------------------------------- compute
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row = TMEM lane
    const int key = k0 + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool key_ok = key < kv_limit;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int st = it % kQSt;
      const int q0 = (i_start + it) * kBQ;
      const float* L2 = sLD + st * 256;
      const float* Dv = L2 + 128;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_ld_full(st), (it / kQSt) & 1, ab) &&
                                       mbar_wait(bar_s, it & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = !key_ok || (q0 + kBQ > a.N) || (a.causal && q0 < k0 + kBK - 1);
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32];
        tmem_ld32(tl + C::kColS + 32 * c, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          float p0 = ex2(fmaf(__uint_as_float(sr[2 * e]), a.scale_log2, -L2[qa]));
          float p1 = ex2(fmaf(__uint_as_float(sr[2 * e + 1]), a.scale_log2, -L2[qa + 1]));
          if (need_mask) {
            const int qg = q0 + qa;
            if (!key_ok || qg >= a.N || (a.causal && key > qg)) p0 = 0.f;
            if (!key_ok || qg + 1 >= a.N || (a.causal && key > qg + 1)) p1 = 0.f;
          }
          pk[16 * c + e] = pack_bf16(p0, p1);
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pk[16 * c + e];
        tmem_st16(tl + C::kColS + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);

      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp, it & 1, ab) &&
                                       (it == 0 || mbar_wait(bar_dsm_empty, (it - 1) & 1, ab)))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t dr[32];
        tmem_ld32(tl + C::kColdP + 32 * c, dr);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          const uint32_t pw = pk[16 * c + e];
          const float d0 = bf16lo(pw) * (__uint_as_float(dr[2 * e]) - Dv[qa]);
          const float d1 = bf16hi(pw) * (__uint_as_float(dr[2 * e + 1]) - Dv[qa + 1]);
          w[e] = pack_bf16(d0, d1);
        }
        // dS^T columns [16c, 16c+16) overwrite dP^T columns this thread has read.
        tmem_st16(tl + C::kColdP + 16 * c, w);
        // dS for the dQ product: A operand, MN-major (queries contiguous),
        // 128-byte swizzle; key row kr, queries 32c..32c+31 = 4 pieces of 16 B.
        const int atom = c >> 1;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int piece = ((c & 1) * 4 + t) ^ (kr & 7);
          uint4 v = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          *reinterpret_cast<uint4*>(smem + C::kOffdS + atom * C::kAtomBytes + kr * 128 +
                                    piece * 16) = v;
        }
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
    if (ok && n_iter > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, ab));
      tc_fence_after();
    }
    ok = bar_and(1, 128, ok && *abort_flag == 0);
    if (ok) {
      // ------------------------------------------------------------ dK, dV rows
      // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
      const bool store = key < a.N;
      const long long row = static_cast<long long>(bh) * a.N + (store ? key : 0);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint16_t* dst = (which == 0 ? a.dV : a.dK) + row * HD;
        const uint32_t col = which == 0 ? C::kColdV : C::kColdK;
        const float mul = which == 0 ? 1.f : a.scale;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t r[32];
          if (n_iter > 0) {
            tmem_ld32(tl + col + 32 * c, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * t + 0]) * mul, __uint_as_float(r[8 * t + 1]) * mul);
            v.y = pack_bf16(__uint_as_float(r[8 * t + 2]) * mul, __uint_as_float(r[8 * t + 3]) * mul);
            v.z = pack_bf16(__uint_as_float(r[8 * t + 4]) * mul, __uint_as_float(r[8 * t + 5]) * mul);
            v.w = pack_bf16(__uint_as_float(r[8 * t + 6]) * mul, __uint_as_float(r[8 * t + 7]) * mul);
            if (store) *reinterpret_cast<uint4*>(dst + 32 * c + 8 * t) = v;
          }
        }
      }
    }
  } else if (warp >= 8) {
    // -------------------------------------------------------------- dQ drain
    const int quarter = warp & 3;
    const int qr = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int it = 0; it < n_iter; ++it) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dq_full, it & 1, ab))) break;
      tc_fence_after();
      const int q = (i_start + it) * kBQ + qr;
      float* dst = a.dq_acc + (static_cast<long long>(bh) * a.N + q) * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + C::kColdQ + 32 * c, r);
        tmem_wait_ld();
        if (q < a.N) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            red_add_v4(dst + 32 * c + 4 * t, __uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                       __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// d = 128: 64-query steps.  Halving the query step frees TMEM for separate
// dS^T and dQ regions, so no product waits for the dQ drain:
//   TMEM  S^T 0-63 (P^T over 0-31) | dP^T 64-127 | dS^T 128-159 |
//         dQ^T 192-255 | dV 256-383 | dK 384-511
// dQ is produced transposed, dQ_i^T = K_j^T dS^T (M = d = 128 on TMEM lanes,
// N = 64 queries); the drain warps (lane t = column t of dQ) write the tile
// row-major into shared memory and one thread adds it into the fp32
// accumulator with a single TMA bulk reduce-add.
// Per step i the issue order is
//   dV += P^T dO_i;  S^T(i+1);  dP^T(i+1);  dK += dS^T Q_i;  dQ_i^T
// so the exponentials of step i+1 overlap dK_i and dQ_i.
constexpr int kQ64 = 64;   // query rows per step
constexpr int kQ64St = 2;  // Q/dO ring depth

struct B128 {
  static constexpr int kKVAtom = 128 * 128;         // 128 rows x 128 B
  static constexpr int kKVTile = 2 * kKVAtom;       // 128 rows x 128 bf16
  static constexpr int kQAtom = kQ64 * 128;         // 64 rows x 128 B
  static constexpr int kQTile = 2 * kQAtom;         // 64 rows x 128 bf16
  static constexpr int kDsBuf = 128 * kQ64 * 2;     // 128 keys x 64 queries bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kKVTile;
  static constexpr int kOffQ = 2 * kKVTile;
  static constexpr int kOffdO = kOffQ + kQ64St * kQTile;
  static constexpr int kOffdS = kOffdO + kQ64St * kQTile;  // 2 buffers
  static constexpr int kOffLD = kOffdS + 2 * kDsBuf;       // kQ64St x (L2[64], D[64])
  static constexpr int kOffStage = (kOffLD + kQ64St * 512 + 1023) / 1024 * 1024;  // dQ tile, fp32
  static constexpr int kStageBytes = kQ64 * 128 * 4;
  static constexpr int kOffBar = kOffStage + kStageBytes;
  // kv, qdo_full[], qdo_empty[], ld_full[], s, dp, p, ds, dst_empty, dq_full,
  // dq_empty, dsm_empty[2], final, drain
  static constexpr int kNumBar = 1 + 3 * kQ64St + 7 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColdP = 64, kColdS = 128, kColdQ = 192, kColdV = 256,
                            kColdK = 384;
};

__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel_q64(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                      const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using C = B128;
  constexpr int HD = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sK = sb + C::kOffK, sV = sb + C::kOffV;
  const uint32_t sQ = sb + C::kOffQ, sdO = sb + C::kOffdO, sdS = sb + C::kOffdS;
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  const uint32_t bar0 = sb + C::kOffBar;
  const uint32_t bar_kv = bar0;
  auto bar_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (1 + kQ64St + s); };
  auto bar_ld_full = [&](int s) { return bar0 + 8u * (1 + 2 * kQ64St + s); };
  const uint32_t bar_s = bar0 + 8u * (1 + 3 * kQ64St);
  const uint32_t bar_dp = bar_s + 8, bar_p = bar_s + 16, bar_ds = bar_s + 24;
  const uint32_t bar_dst_empty = bar_s + 32, bar_dq_full = bar_s + 40, bar_dq_empty = bar_s + 48;
  auto bar_dsm_empty = [&](int b) { return bar_s + 56u + 8u * b; };
  const uint32_t bar_final = bar_s + 72, bar_drain = bar_s + 80;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Head-major order; small kt (most work under causal) first.
  const int bh = static_cast<int>(blockIdx.x / a.n_ktiles);
  const int kt = static_cast<int>(blockIdx.x % a.n_ktiles);
  const int k0 = kt * kBK;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  const int i_start = a.causal ? k0 / kQ64 : 0;
  const int n_iter = (k0 >= kv_limit) ? 0 : a.n_qtiles - i_start;

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < kQ64St; ++s) {
      mbar_init(bar_qdo_full(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
      mbar_init(bar_ld_full(s), 32);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 4);
    mbar_init(bar_ds, 4);
    mbar_init(bar_dst_empty, 1);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_empty, 4);
    mbar_init(bar_dsm_empty(0), 1);
    mbar_init(bar_dsm_empty(1), 1);
    mbar_init(bar_final, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
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
    // -------------------------------------------------------------- producer
    if (n_iter > 0) {
      uint64_t pol_kv = 0, pol_q = 0;
      if (lane == 0) {
        pol_kv = policy_evict_first();
        pol_q = policy_evict_last();  // Q_i, dO_i are re-read by every key block
        mbar_arrive_expect_tx(bar_kv, 2 * C::kKVTile);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sK + c * C::kKVAtom, &tmK, c * 64, k0, bh, bar_kv, pol_kv);
          tma_load_3d(sV + c * C::kKVAtom, &tmV, c * 64, k0, bh, bar_kv, pol_kv);
        }
      }
      int last[kQ64St];
      for (int t = 0; t < kQ64St; ++t) last[t] = -1;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % kQ64St;
        const int q0 = (i_start + it) * kQ64;
        if (it >= kQ64St &&
            !__all_sync(0xffffffffu, mbar_wait(bar_qdo_empty(st), ((it / kQ64St) & 1) ^ 1, ab)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_qdo_full(st), 2 * C::kQTile);
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(sQ + st * C::kQTile + c * C::kQAtom, &tmQ, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
            tma_load_3d(sdO + st * C::kQTile + c * C::kQAtom, &tmdO, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
          }
        }
        last[st] = it;
        float* L2 = sLD + st * 128;
        float* Dv = L2 + 64;
        const long long rbase = static_cast<long long>(bh) * a.N;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = lane * 2 + e;
          const int q = q0 + r;
          L2[r] = q < a.N ? a.L[rbase + q] * kLog2e : 0.f;
          Dv[r] = q < a.N ? a.D[rbase + q] : 0.f;
        }
        mbar_arrive(bar_ld_full(st));
      }
      if (lane == 0 && *abort_flag) {
        mbar_wait_drain(bar_kv, 0);
        for (int s = 0; s < kQ64St; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar_qdo_full(s), (last[s] / kQ64St) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = idesc_bf16(128, kQ64, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(128, HD, false, true);    // dV, dK
      constexpr uint32_t idQ = idesc_bf16(HD, kQ64, true, true);     // dQ^T
      // K-major operands, step k of 16 columns of d (atom k/4, 32 B per step)
      auto kmaj_kv = [](uint32_t base, int k) {
        return sdesc_sw128(base + (k >> 2) * C::kKVAtom + (k & 3) * 32, 16, 1024);
      };
      auto kmaj_q = [](uint32_t base, int k) {
        return sdesc_sw128(base + (k >> 2) * C::kQAtom + (k & 3) * 32, 16, 1024);
      };
      // MN-major operands, step k of 16 rows (two 8-row groups)
      auto mn_q = [](uint32_t base, int k) { return sdesc_sw128(base + k * 2048, C::kQAtom, 1024); };
      auto mn_kv = [](uint32_t base, int k) { return sdesc_sw128(base + k * 2048, C::kKVAtom, 1024); };
      auto issue_s = [&](int it) {
        const uint32_t q = sQ + (it % kQ64St) * C::kQTile;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tmem + C::kColS, kmaj_kv(sK, k), kmaj_q(q, k), idS, k > 0 ? 1u : 0u);
        mma_commit(bar_s);
      };
      auto issue_dp = [&](int it) {
        const uint32_t g = sdO + (it % kQ64St) * C::kQTile;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tmem + C::kColdP, kmaj_kv(sV, k), kmaj_q(g, k), idS, k > 0 ? 1u : 0u);
        mma_commit(bar_dp);
      };
      bool ok = mbar_wait(bar_kv, 0, ab) && mbar_wait(bar_qdo_full(0), 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int st = it % kQ64St;
        const bool more = it + 1 < n_iter;
        // dV += P^T dO_i
        if (!(ok = mbar_wait(bar_p, it & 1, ab))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kQ64 / 16; ++k)
          mma_ts(tmem + C::kColdV, tmem + C::kColS + k * 8, mn_q(sdO + st * C::kQTile, k), idKV,
                 (it > 0 || k > 0) ? 1u : 0u);
        // S^T(i+1) overwrites P^T(i): the product above reads it first.
        if (more) {
          if (!(ok = mbar_wait(bar_qdo_full((it + 1) % kQ64St), ((it + 1) / kQ64St) & 1, ab))) break;
          tc_fence_after();
          issue_s(it + 1);
        }
        if (!(ok = mbar_wait(bar_ds, it & 1, ab))) break;
        tc_fence_after();
        // dP^T(i+1): dS^T(i) lives in its own columns, so this need not wait for dK.
        if (more) issue_dp(it + 1);
        // dK += dS^T Q_i
#pragma unroll
        for (int k = 0; k < kQ64 / 16; ++k)
          mma_ts(tmem + C::kColdK, tmem + C::kColdS + k * 8, mn_q(sQ + st * C::kQTile, k), idKV,
                 (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar_dst_empty);
        mma_commit(bar_qdo_empty(st));
        // dQ_i^T = K_j^T dS^T into the dQ columns once the previous tile is drained
        if (it > 0) {
          if (!(ok = mbar_wait(bar_dq_empty, (it - 1) & 1, ab))) break;
          tc_fence_after();
        }
        const uint32_t ds = sdS + (it & 1) * C::kDsBuf;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_ss(tmem + C::kColdQ, mn_kv(sK, k), sdesc_sw128(ds + k * 2048, 16, 1024), idQ,
                 k > 0 ? 1u : 0u);
        mma_commit(bar_dq_full);
        mma_commit(bar_dsm_empty(it & 1));
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // -------------------------------------------------------------- compute
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row = TMEM lane
    const int key = k0 + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool key_ok = key < kv_limit;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int st = it % kQ64St;
      const int q0 = (i_start + it) * kQ64;
      const float* L2 = sLD + st * 128;
      const float* Dv = L2 + 64;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_ld_full(st), (it / kQ64St) & 1, ab) &&
                                       mbar_wait(bar_s, it & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool need_mask = !key_ok || (q0 + kQ64 > a.N) || (a.causal && q0 < k0 + kBK - 1);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sr[32];
        tmem_ld32(tl + C::kColS + 32 * c, sr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          float p0 = ex2(fmaf(__uint_as_float(sr[2 * e]), a.scale_log2, -L2[qa]));
          float p1 = ex2(fmaf(__uint_as_float(sr[2 * e + 1]), a.scale_log2, -L2[qa + 1]));
          if (need_mask) {
            const int qg = q0 + qa;
            if (!key_ok || qg >= a.N || (a.causal && key > qg)) p0 = 0.f;
            if (!key_ok || qg + 1 >= a.N || (a.causal && key > qg + 1)) p1 = 0.f;
          }
          pk[16 * c + e] = pack_bf16(p0, p1);
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pk[16 * c + e];
        tmem_st16(tl + C::kColS + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);

      const int buf = it & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar_dp, it & 1, ab) &&
                          (it < 1 || mbar_wait(bar_dst_empty, (it - 1) & 1, ab)) &&
                          (it < 2 || mbar_wait(bar_dsm_empty(buf), ((it >> 1) & 1) ^ 1, ab)))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dr[32];
        tmem_ld32(tl + C::kColdP + 32 * c, dr);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          const uint32_t pw = pk[16 * c + e];
          const float d0 = bf16lo(pw) * (__uint_as_float(dr[2 * e]) - Dv[qa]);
          const float d1 = bf16hi(pw) * (__uint_as_float(dr[2 * e + 1]) - Dv[qa + 1]);
          w[e] = pack_bf16(d0, d1);
        }
        tmem_st16(tl + C::kColdS + 16 * c, w);
        // dS^T for the dQ product: B operand, MN-major (queries contiguous),
        // 128-byte swizzle; key row kr, queries 32c..32c+31 = 4 pieces of 16 B.
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int piece = (c * 4 + t) ^ (kr & 7);
          *reinterpret_cast<uint4*>(smem + C::kOffdS + buf * C::kDsBuf + kr * 128 + piece * 16) =
              make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
    if (ok && n_iter > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, ab));
      tc_fence_after();
    }
    ok = bar_and(1, 128, ok && *abort_flag == 0);
    if (ok) {
      // ------------------------------------------------------------ dK, dV rows
      // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
      const bool store = key < a.N;
      const long long row = static_cast<long long>(bh) * a.N + (store ? key : 0);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint16_t* dst = (which == 0 ? a.dV : a.dK) + row * HD;
        const uint32_t col = which == 0 ? C::kColdV : C::kColdK;
        const float mul = which == 0 ? 1.f : a.scale;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t r[32];
          if (n_iter > 0) {
            tmem_ld32(tl + col + 32 * c, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * t + 0]) * mul, __uint_as_float(r[8 * t + 1]) * mul);
            v.y = pack_bf16(__uint_as_float(r[8 * t + 2]) * mul, __uint_as_float(r[8 * t + 3]) * mul);
            v.z = pack_bf16(__uint_as_float(r[8 * t + 4]) * mul, __uint_as_float(r[8 * t + 5]) * mul);
            v.w = pack_bf16(__uint_as_float(r[8 * t + 6]) * mul, __uint_as_float(r[8 * t + 7]) * mul);
            if (store) *reinterpret_cast<uint4*>(dst + 32 * c + 8 * t) = v;
          }
        }
      }
    }
  } else if (warp >= 8) {
    // -------------------------------------------------------------- dQ drain
    // Thread t holds column t of dQ_i (TMEM lane t of dQ^T) for the 64 query
    // rows; it writes that column of the row-major fp32 staging tile, and one
    // thread then adds the tile into the accumulator (rows >= N are clipped).
    const int quarter = warp & 3;
    const int dd = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* stage = reinterpret_cast<float*>(smem + C::kOffStage);
    const uint32_t sstage = sb + C::kOffStage;
    for (int it = 0; it < n_iter; ++it) {
      // One decision for all four drain warps (they share named barrier 2).
      // Passing this barrier also means the previous reduce has finished
      // reading the staging tile: its issuer waited before arriving here.
      if (!bar_and(2, 128, mbar_wait(bar_dq_full, it & 1, ab))) break;
      tc_fence_after();
      const int q0 = (i_start + it) * kQ64;
      uint32_t r0[32], r1[32];
      tmem_ld32(tl + C::kColdQ, r0);
      tmem_ld32(tl + C::kColdQ + 32, r1);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_empty);
#pragma unroll
      for (int q = 0; q < 32; ++q) stage[q * HD + dd] = __uint_as_float(r0[q]);
#pragma unroll
      for (int q = 0; q < 32; ++q) stage[(32 + q) * HD + dd] = __uint_as_float(r1[q]);
      fence_proxy_async_smem();
      bar_sync_n(2, 128);
      if (dd == 0) {
        tma_reduce_add_3d(&tmdQ, sstage, 0, q0, bh);
        bulk_commit();
        bulk_wait_read0();
      }
    }
    if (dd == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_bwd_q64(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmdO, const CUtensorMap& tmdQ, const BwdArgs& a,
                           cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_bwd_kernel_q64, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             B128::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = static_cast<long long>(a.n_ktiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_kernel_q64<<<static_cast<unsigned>(grid), kThreads, B128::kSmemBytes, stream>>>(
      tmQ, tmK, tmV, tmdO, tmdQ, a);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_bwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         const CUtensorMap& tmdO, const BwdArgs& a, cudaStream_t stream) {
  using C = BCfg<HD>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = static_cast<long long>(a.n_ktiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_kernel<HD><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV,
                                                                                     tmdO, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                       const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_bwd_t<64>(tmQ, tmK, tmV, tmdO, a, stream);
    case 128: return launch_bwd_q64(tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
