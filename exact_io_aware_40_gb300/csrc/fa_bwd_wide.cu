// fa_bwd_wide.cu -- backward pass of exact attention for d = 64 and d = 128.
//
// Same method and formulas as fa_bwd.cu (P recomputed from L; dV = P^T dO,
// dP = dO V^T, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q; fmread.com
// summary, section 三.2 "反向传播优化"), organised so that every tcgen05 product
// is 128 wide (M = 128, N = 128): an M = 128 product instruction takes at
// least about 45 clocks, so one with N = 64 runs at two thirds of the tensor
// rate whatever its operands' source, while N = 128 runs at the full rate
// (64 clocks per 16-deep k-step).  Each 128-wide step is split by columns
// between two softmax warpgroups, so both work on every step in parallel:
//
// fa_bwd_dkdv_wide_kernel -- one CTA per 128-key block j, 128-row query steps
//   i.  TMEM: S^T 0-127, dP^T 128-255 (keys on lanes, queries on columns), dV
//   256.., dK 256+d.  Warpgroup A handles query columns 0-63 of the step,
//   warpgroup B 64-127; each writes its P^T (bf16) over the first half of its
//   own S^T columns and its dS^T over the first half of its own dP^T columns,
//   and the dV and dK products address those halves k-step by k-step.
//   Issue order per step: dV_i, S^T_{i+1} (after dV_i has read P^T_i),
//   dK_i, dP^T_{i+1} (after dK_i has read dS^T_i).
// fa_bwd_dq_wide_kernel -- one CTA per 128-row query block, 128-key steps j.
//   TMEM: two S buffers 0-127 and 128-255 (S_{j+1} is computed while the
//   warpgroups work on S_j), dP 256-383, dQ 384...  Warpgroup A handles key
//   columns 0-63, B 64-127.  dS_j goes over the first half of each
//   warpgroup's columns of S_j's buffer (read before), so the dP buffer is
//   free once the warpgroups have loaded dP_j: dP_{j+1} is issued then, and
//   the products overlap the warpgroups' work instead of waiting on it.
//   Issue order per step: dP_{j+1} (after dP_j is read), dQ_j (after dS_j),
//   S_{j+2} (into S_j's buffer, after dQ_j has read dS_j).
#include "kernels.h"
#include <type_traits>

#include "masks.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kT = 128;  // keys per block = query rows per step (and vice versa)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool bar_and_w(int id, int nthreads, bool pred) {
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
__device__ __forceinline__ void bar_sync_w(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Descriptors of the K k-steps of a K-major operand (128-row tile, 64-column
// atoms of 16 KB): step k covers columns [16k, 16k+16) of d.
template <int K>
__device__ __forceinline__ void kmaj128_steps(uint32_t base, uint64_t (&d)[K]) {
  const uint64_t d0 = sdesc_sw128(base, 16, 1024);
#pragma unroll
  for (int k = 0; k < K; ++k) d[k] = sdesc_add(d0, (k >> 2) * 16384 + (k & 3) * 32);
}
// The same for an MN-major operand (128-row tile; rows = reduction dim):
// step k covers rows [16k, 16k+16).
template <int K>
__device__ __forceinline__ void mnmaj128_steps(uint32_t base, uint64_t (&d)[K]) {
  const uint64_t d0 = sdesc_sw128(base, 16384, 1024);
#pragma unroll
  for (int k = 0; k < K; ++k) d[k] = sdesc_add(d0, k * 2048);
}
// TMEM column of k-step k (16 rows of the reduction dim) of a bf16 A operand
// whose two 64-row halves sit at `lo` and `hi`.
__device__ __forceinline__ uint32_t split_col(uint32_t lo, uint32_t hi, int k) {
  return k < 4 ? lo + 8u * k : hi + 8u * (k - 4);
}

template <int HD>
struct WCfg {
  static constexpr int kAtoms = HD / 64;
  static constexpr int kTile = kAtoms * 16384;          // 128 rows x d bf16
  static constexpr int kSt = HD == 64 ? 3 : 2;          // ring depth
};

// ===========================================================================
// dK, dV
// ===========================================================================
template <int HD>
struct KvW {
  using W = WCfg<HD>;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = W::kTile;
  static constexpr int kOffQ = 2 * W::kTile;                    // kSt stages
  static constexpr int kOffdO = kOffQ + W::kSt * W::kTile;      // kSt stages
  static constexpr int kLdSt = 4;                               // L, D ring depth
  static constexpr int kOffLD = kOffdO + W::kSt * W::kTile;     // kLdSt x (L2[128], D[128])
  static constexpr int kOffBar = kOffLD + kLdSt * 1024;
  // k, qdo_full[], qdo_empty[], ld_full[4], ld_empty[4], s, dp, p, ds, final, drain, v
  static constexpr int kNumBar = 1 + 2 * W::kSt + 2 * kLdSt + 7;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 256 + HD;
};

// DROP: dropout on P (a separate instantiation, as in the forward).
template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmdO, const BwdArgs a) {
  using C = KvW<HD>;
  using W = WCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sK = sb + C::kOffK, sV = sb + C::kOffV, sQ = sb + C::kOffQ, sdO = sb + C::kOffdO;
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  const uint32_t bar0 = sb + C::kOffBar;
  const uint32_t bar_kv = bar0;
  auto bar_qdo_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (1 + W::kSt + s); };
  auto bar_ld_full = [&](int s) { return bar0 + 8u * (1 + 2 * W::kSt + s); };
  auto bar_ld_empty = [&](int s) { return bar0 + 8u * (1 + 2 * W::kSt + C::kLdSt + s); };
  const uint32_t bar_s = bar0 + 8u * (1 + 2 * W::kSt + 2 * C::kLdSt);
  const uint32_t bar_dp = bar_s + 8, bar_p = bar_s + 16, bar_ds = bar_s + 24;
  const uint32_t bar_final = bar_s + 32, bar_drain = bar_s + 40;
  // K_j and V_j land on separate barriers: the first S^T needs K_j and Q_0
  // only, so those are loaded first and V_j after them.
  const uint32_t bar_v = bar_s + 48;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Small kt (most work under causal) first, in groups of ranks, head-major
  // inside a group.
  int bh, kt;
  cta_tile(static_cast<int>(blockIdx.x), a.n_ktiles, a.BH, a.tile_group, &bh, &kt);
  const int k0 = kt * kT;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  // Query blocks that see this key block: a range from the masks, thinned by
  // column kt of the block mask; every role walks it in the same order.
  int ilo, ihi;
  query_block_range(kt, a.n_qtiles, kv_limit, a.causal, a.window, &ilo, &ihi);
  const uint8_t* bmc = a.bmask ? a.bmask + kt : nullptr;  // column kt, stride nb
  volatile int* n_steps = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  if (warp == 3) {
    const int n = count_blocks(bmc, a.nb, ilo, ihi);
    if (lane == 0) *n_steps = n;
  }

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    mbar_init(bar_v, 1);
    for (int s = 0; s < W::kSt; ++s) {
      mbar_init(bar_qdo_full(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
    }
    for (int s = 0; s < C::kLdSt; ++s) {
      mbar_init(bar_ld_full(s), 32);
      mbar_init(bar_ld_empty(s), 8);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 8);
    mbar_init(bar_ds, 8);
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
  const int n_iter = *n_steps;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (n_iter > 0) {
      uint64_t pol_kv = 0, pol_q = 0;
      if (lane == 0) {
        pol_kv = policy_evict_first();
        pol_q = policy_evict_last();  // Q_i, dO_i are re-read by every key block
        mbar_arrive_expect_tx(bar_kv, W::kTile);
        for (int c = 0; c < W::kAtoms; ++c)
          tma_load_3d(sK + c * 16384, &tmK, c * 64, k0, bh, bar_kv, pol_kv);
      }
      int last[W::kSt];
      for (int t = 0; t < W::kSt; ++t) last[t] = -1;
      int qb = next_block(bmc, a.nb, ilo, ihi);
      for (int it = 0; it < n_iter; ++it, qb = next_block(bmc, a.nb, qb + 1, ihi)) {
        const int st = it % W::kSt;
        const int q0 = qb * kT;
        if (it >= W::kSt &&
            !__all_sync(0xffffffffu, mbar_wait(bar_qdo_empty(st), ((it / W::kSt) & 1) ^ 1, ab)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_qdo_full(st), 2 * W::kTile);
          for (int c = 0; c < W::kAtoms; ++c) {
            tma_load_3d(sQ + st * W::kTile + c * 16384, &tmQ, c * 64, q0, bh, bar_qdo_full(st),
                        pol_q);
            tma_load_3d(sdO + st * W::kTile + c * 16384, &tmdO, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
          }
          if (it == 0) {
            mbar_arrive_expect_tx(bar_v, W::kTile);
            for (int c = 0; c < W::kAtoms; ++c)
              tma_load_3d(sV + c * 16384, &tmV, c * 64, k0, bh, bar_v, pol_kv);
          }
        }
        last[st] = it;
      }
      if (lane == 0 && *abort_flag) {
        mbar_wait_drain(bar_kv, 0);
        mbar_wait_drain(bar_v, 0);
        for (int s = 0; s < W::kSt; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar_qdo_full(s), (last[s] / W::kSt) & 1);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------ row terms L, D
    // Off the Q/dO ring, up to kLdSt steps ahead of the softmax warpgroups.
    const long long rbase = static_cast<long long>(bh) * a.N;
    int qb = next_block(bmc, a.nb, ilo, ihi);
    for (int it = 0; it < n_iter; ++it, qb = next_block(bmc, a.nb, qb + 1, ihi)) {
      const int st = it % C::kLdSt;
      const int q0 = qb * kT;
      if (it >= C::kLdSt &&
          !__all_sync(0xffffffffu, mbar_wait(bar_ld_empty(st), ((it / C::kLdSt) & 1) ^ 1, ab)))
        break;
      float* L2 = sLD + st * 256;
      float* Dv = L2 + 128;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = lane * 4 + e;
        const int q = q0 + r;
        L2[r] = q < a.N ? -(a.L[rbase + q] * kLog2e) : 0.f;  // negated: the FMA adds it
        Dv[r] = q < a.N ? a.D[rbase + q] : 0.f;
      }
      mbar_arrive(bar_ld_full(st));
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = idesc_bf16(kT, kT, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(kT, HD, false, true);  // dV, dK
      constexpr int kD = HD / 16, kQ = kT / 16;  // k-steps over d, over a query step
      // Built once: descriptors of the resident K_j and V_j, TMEM addresses
      // of the P^T and dS^T halves (A operands of dV and dK).
      uint64_t aK[kD], aV[kD];
      kmaj128_steps(sK, aK);
      kmaj128_steps(sV, aV);
      uint32_t tP[kQ], tdS[kQ];
#pragma unroll
      for (int k = 0; k < kQ; ++k) {
        tP[k] = tmem + split_col(C::kColS, C::kColS + 64, k);
        tdS[k] = tmem + split_col(C::kColdP, C::kColdP + 64, k);
      }
      // Q/dO stage of step it (cur) and of step it + 1 (nxt)
      RingPos<W::kSt> cur, nxt;
      auto issue_s = [&](int st) {
        uint64_t b[kD];
        kmaj128_steps(sQ + st * W::kTile, b);
        mma_ss_k(tmem + C::kColS, aK, b, idS, 0u);
        mma_commit(bar_s);
      };
      auto issue_dp = [&](int st) {
        uint64_t b[kD];
        kmaj128_steps(sdO + st * W::kTile, b);
        mma_ss_k(tmem + C::kColdP, aV, b, idS, 0u);
        mma_commit(bar_dp);
      };
      bool ok = mbar_wait(bar_kv, 0, ab) && mbar_wait(bar_qdo_full(0), 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      if (ok && (ok = mbar_wait(bar_v, 0, ab))) {
        tc_fence_after();
        issue_dp(0);
      }
      nxt.next();
      for (int it = 0; ok && it < n_iter; ++it) {
        const int st = cur.stage;
        const bool more = it + 1 < n_iter;
        // dV += P^T dO_i (P^T halves at columns 0 and 64)
        if (!(ok = mbar_wait(bar_p, it & 1, ab))) break;
        tc_fence_after();
        {
          uint64_t b[kQ];
          mnmaj128_steps(sdO + st * W::kTile, b);
          mma_ts_k(tmem + C::kColdV, tP, b, idKV, it > 0 ? 1u : 0u);
        }
        // S^T(i+1) overwrites P^T(i): the product above reads it first.
        if (more) {
          if (!(ok = mbar_wait(bar_qdo_full(nxt.stage), nxt.phase, ab))) break;
          tc_fence_after();
          issue_s(nxt.stage);
        }
        // dK += dS^T Q_i (dS^T halves at columns 128 and 192)
        if (!(ok = mbar_wait(bar_ds, it & 1, ab))) break;
        tc_fence_after();
        {
          uint64_t b[kQ];
          mnmaj128_steps(sQ + st * W::kTile, b);
          mma_ts_k(tmem + C::kColdK, tdS, b, idKV, it > 0 ? 1u : 0u);
        }
        mma_commit(bar_qdo_empty(st));
        // dP^T(i+1) overwrites dS^T(i): dK above reads it first.
        if (more) issue_dp(nxt.stage);
        cur.next();
        nxt.next();
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int x = (warp >> 2) - 1;        // 0: query columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;   // key row = TMEM lane
    const int key = k0 + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t cs = C::kColS + 64u * x, cdp = C::kColdP + 64u * x;
    const bool key_ok = key < kv_limit;
    bool ok = true;
    int qb = next_block(bmc, a.nb, ilo, ihi);
    for (int it = 0; it < n_iter; ++it, qb = next_block(bmc, a.nb, qb + 1, ihi)) {
      const int lst = it % C::kLdSt;
      const int q0 = qb * kT + 64 * x;  // first query column of this half
      const float* L2 = sLD + lst * 256 + 64 * x;
      const float* Dv = sLD + lst * 256 + 128 + 64 * x;
      // Dropout keep bits of this thread's key for the step's 64 queries of
      // this half (the warp draws them together), before S^T arrives.
      uint64_t km = 0;
      if constexpr (DROP)
        if (ok)
          km = keep64_transposed(static_cast<uint32_t>(k0 + quarter * 32), static_cast<uint32_t>(q0),
                               static_cast<uint32_t>(bh % a.H), static_cast<uint32_t>(b),
                               a.seed_lo, a.seed_hi, a.drop_thr);
      // ---- P^T: on the critical path (S^T -> P^T -> dV -> next S^T)
      const bool ok1 = ok && __all_sync(0xffffffffu,
                                        mbar_wait(bar_ld_full(lst), (it / C::kLdSt) & 1, ab) &&
                                            mbar_wait(bar_s, it & 1, ab));
      float p[64];
      if (ok1) {
        tc_fence_after();
        const bool band = (a.causal != 0) | (a.window >= 0);
        const bool need_mask = !key_ok || (q0 + 64 > a.N) || (band && q0 < k0 + kT - 1) ||
                               (a.window >= 0 && k0 < q0 + 63 - a.window);
        uint32_t sr[2][32];
        tmem_ld32(tl + cs, sr[0]);
        tmem_ld32(tl + cs + 32, sr[1]);
        tmem_wait_ld();
        // p = 2^(s^T scale log2e - L log2e) on packed fp32 pairs (the ring
        // holds -L log2e).
        const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2);
        const uint64_t* nL2 = reinterpret_cast<const uint64_t*>(L2);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e >> 4][(2 * e) & 31]),
                                   __uint_as_float(sr[e >> 4][(2 * e + 1) & 31])),
                           scl2, nL2[e]),
                    t0, t1);
          p[2 * e] = ex2(t0);
          p[2 * e + 1] = ex2(t1);
        }
        // One branch per step; inside, selects only (a branch per element in
        // the loop above costs more than the exponentials).
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int qg = q0 + e;
            const bool keep = (qg < a.N) & visible(qg, key, kv_limit, a.causal, a.window);
            p[e] = keep ? p[e] : 0.f;
          }
        }
        uint32_t w[32];
        if constexpr (DROP) {
          // dV takes the dropped weights P Z / q; p itself stays for dS^T.
#pragma unroll
          for (int e = 0; e < 32; ++e)
            w[e] = pack_bf16((km >> (2 * e)) & 1u ? p[2 * e] * a.drop_scale : 0.f,
                             (km >> (2 * e + 1)) & 1u ? p[2 * e + 1] * a.drop_scale : 0.f);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = pack_bf16(p[2 * e], p[2 * e + 1]);
        }
        // P^T over the first half of this warpgroup's S^T columns (read above)
        tmem_st32(tl + cs, w);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);
      }
      // Both warpgroups finish P^T before either starts dS^T.  dS^T feeds dK,
      // which the MMA warp issues only after dV and the next S^T, so it has
      // slack; P^T has none, and running the two side by side slowed P^T.
      // Every exit of the loop passes through this barrier, so a warpgroup
      // that stops early cannot leave the other waiting.
      ok = bar_and_w(3, 256, ok1);
      if (!ok) break;
      // ---- dS^T
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dp, it & 1, ab));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dr[32];
          tmem_ld32(tl + cdp + 32 * c, dr);
          tmem_wait_ld();
          uint32_t w[16];
          // dS^T = P^T o (dP^T - D); with dropout dP^T = (V dO^T) Z / q.
          auto ds_chunk = [&](auto drop) {
            const uint64_t* Dv2 = reinterpret_cast<const uint64_t*>(Dv);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int qa = 32 * c + 2 * e;
              float g0 = __uint_as_float(dr[2 * e]), g1 = __uint_as_float(dr[2 * e + 1]);
              if constexpr (decltype(drop)::value) {
                g0 = (km >> qa) & 1u ? g0 * a.drop_scale : 0.f;
                g1 = (km >> (qa + 1)) & 1u ? g1 * a.drop_scale : 0.f;
              }
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(p[qa], p[qa + 1]), f2_sub(f2_pack(g0, g1), Dv2[qa >> 1])),
                        d0, d1);
              w[e] = pack_bf16(d0, d1);
            }
          };
          if constexpr (DROP)
            ds_chunk(std::true_type{});
          else
            ds_chunk(std::false_type{});
          tmem_st16(tl + cdp + 16 * c, w);  // dS^T over columns this thread has read
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_ds);
          mbar_arrive(bar_ld_empty(lst));  // this step's L, D have been read
        }
      }
      // A failed wait here reaches the barrier above in the next step (its
      // waits fail at once) or ends the loop.
    }
    if (ok && n_iter > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, ab));
      tc_fence_after();
    }
    ok = bar_and_w(1 + x, 128, ok && *abort_flag == 0);
    if (ok) {
      // ------------------------------------------------------------ dV (A), dK (B)
      // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
      const bool store = key < a.N;
      const long long row = static_cast<long long>(bh) * a.N + (store ? key : 0);
      uint16_t* dst = (x == 0 ? a.dV : a.dK) + row * HD;
      const uint32_t col = x == 0 ? C::kColdV : C::kColdK;
      const float mul = x == 0 ? 1.f : a.scale;
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

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ
// ===========================================================================
template <int HD>
struct QW {
  using W = WCfg<HD>;
  // Separate K and V rings.  V_j is free once dP_j has completed, K_j only
  // after dQ_j; K_{j+2} must arrive before S_{j+2}, which is issued right
  // after dQ_j, so K needs one stage more than V.
  static constexpr int kKSt = HD == 64 ? 4 : 3;
  static constexpr int kVSt = HD == 64 ? 3 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffdO = W::kTile;
  static constexpr int kOffK = 2 * W::kTile;
  static constexpr int kOffV = kOffK + kKSt * W::kTile;
  static constexpr int kOffBar = kOffV + kVSt * W::kTile;
  // q_full, k_full[], k_empty[], v_full[], v_empty[], s[2], dp, ds, final, drain, dp_free,
  // do_full
  static constexpr int kNumBar = 1 + 2 * kKSt + 2 * kVSt + 8;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColdP = 256, kColdQ = 384;
};

template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmdO,
                          const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using C = QW<HD>;
  using W = WCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sQ = sb + C::kOffQ, sdO = sb + C::kOffdO, sK = sb + C::kOffK, sV = sb + C::kOffV;
  const uint32_t bar0 = sb + C::kOffBar;
  const uint32_t bar_q = bar0;
  auto bar_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (1 + C::kKSt + s); };
  auto bar_vfull = [&](int s) { return bar0 + 8u * (1 + 2 * C::kKSt + s); };
  auto bar_vempty = [&](int s) { return bar0 + 8u * (1 + 2 * C::kKSt + C::kVSt + s); };
  const uint32_t barx = bar0 + 8u * (1 + 2 * C::kKSt + 2 * C::kVSt);
  auto bar_s = [&](int b2) { return barx + 8u * b2; };
  const uint32_t bar_dp = barx + 16, bar_ds = barx + 24, bar_final = barx + 32, bar_drain = barx + 40;
  const uint32_t bar_dpfree = barx + 48;
  // Q and dO land on separate barriers: the first S needs Q and K_0 only, so
  // those are loaded first and dO, V_0 after them.
  const uint32_t bar_do = barx + 56;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Longest query blocks (causal) first, in groups of ranks, head-major inside
  // a group.
  int bh, qt;
  cta_tile(static_cast<int>(blockIdx.x), a.n_qtiles, a.BH, a.tile_group, &bh, &qt);
  qt = a.n_qtiles - 1 - qt;
  const int q0 = qt * kT;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  // Key blocks this query block sees: a range from the masks, thinned by row
  // qt of the block mask; every role walks it in the same order.
  int jlo, jhi;
  key_block_range(qt, kv_limit, a.causal, a.window, &jlo, &jhi);
  const uint8_t* bmr = a.bmask ? a.bmask + static_cast<long long>(qt) * a.nb : nullptr;
  volatile int* n_steps = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  if (warp == 3) {
    const int n = count_blocks(bmr, 1, jlo, jhi);
    if (lane == 0) *n_steps = n;
  }

  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_do, 1);
    for (int s = 0; s < C::kKSt; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int s = 0; s < C::kVSt; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), 1);
    }
    mbar_init(bar_s(0), 1);
    mbar_init(bar_s(1), 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_ds, 8);
    mbar_init(bar_final, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_dpfree, 8);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdQ);
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
  const int T = *n_steps;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0 && T > 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar_q, W::kTile);
      for (int c = 0; c < W::kAtoms; ++c)
        tma_load_3d(sQ + c * 16384, &tmQ, c * 64, q0, bh, bar_q, pol_q);
      int lastk[C::kKSt], lastv[C::kVSt];
      for (int s = 0; s < C::kKSt; ++s) lastk[s] = -1;
      for (int s = 0; s < C::kVSt; ++s) lastv[s] = -1;
      int kb = next_block(bmr, 1, jlo, jhi);
      for (int j = 0; j < T; ++j, kb = next_block(bmr, 1, kb + 1, jhi)) {
        const int sk = j % C::kKSt, sv = j % C::kVSt;
        if (j >= C::kKSt && !mbar_wait(bar_kempty(sk), ((j / C::kKSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_kfull(sk), W::kTile);
        for (int c = 0; c < W::kAtoms; ++c)
          tma_load_3d(sK + sk * W::kTile + c * 16384, &tmK, c * 64, kb * kT, bh, bar_kfull(sk),
                      pol_kv);
        lastk[sk] = j;
        if (j == 0) {
          mbar_arrive_expect_tx(bar_do, W::kTile);
          for (int c = 0; c < W::kAtoms; ++c)
            tma_load_3d(sdO + c * 16384, &tmdO, c * 64, q0, bh, bar_do, pol_q);
        }
        if (j >= C::kVSt && !mbar_wait(bar_vempty(sv), ((j / C::kVSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_vfull(sv), W::kTile);
        for (int c = 0; c < W::kAtoms; ++c)
          tma_load_3d(sV + sv * W::kTile + c * 16384, &tmV, c * 64, kb * kT, bh, bar_vfull(sv),
                      pol_kv);
        lastv[sv] = j;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar_q, 0);
        mbar_wait_drain(bar_do, 0);
        for (int s = 0; s < C::kKSt; ++s)
          if (lastk[s] >= 0) mbar_wait_drain(bar_kfull(s), (lastk[s] / C::kKSt) & 1);
        for (int s = 0; s < C::kVSt; ++s)
          if (lastv[s] >= 0) mbar_wait_drain(bar_vfull(s), (lastv[s] / C::kVSt) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idS = idesc_bf16(kT, kT, false, false);  // S, dP
      constexpr uint32_t idQ = idesc_bf16(kT, HD, false, true);   // dQ
      constexpr int kD = HD / 16, kK = kT / 16;  // k-steps over d, over a key step
      // Built once: descriptors of the resident Q and dO tiles.
      uint64_t aQ[kD], adO[kD];
      kmaj128_steps(sQ, aQ);
      kmaj128_steps(sdO, adO);
      RingPos<C::kKSt> ks, kq;  // K stages of the next S product and of dQ_j
      RingPos<C::kVSt> vs;      // V stage of the next dP product
      // S_j = Q K_j^T into buffer j & 1
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(bar_kfull(ks.stage), ks.phase, ab)) return false;
        tc_fence_after();
        uint64_t b[kD];
        kmaj128_steps(sK + ks.stage * W::kTile, b);
        mma_ss_k(tmem + C::kColS + 128u * (j & 1), aQ, b, idS, 0u);
        mma_commit(bar_s(j & 1));
        ks.next();
        return true;
      };
      // dP_j = dO V_j^T; V_j's stage is free again once it completes.
      auto issue_dp = [&]() -> bool {
        if (!mbar_wait(bar_vfull(vs.stage), vs.phase, ab)) return false;
        tc_fence_after();
        uint64_t b[kD];
        kmaj128_steps(sV + vs.stage * W::kTile, b);
        mma_ss_k(tmem + C::kColdP, adO, b, idS, 0u);
        mma_commit(bar_dp);
        mma_commit(bar_vempty(vs.stage));
        vs.next();
        return true;
      };
      bool ok = mbar_wait(bar_q, 0, ab);
      if (ok) ok = issue_s(0);
      if (ok) ok = mbar_wait(bar_do, 0, ab) && issue_dp();
      if (ok && T > 1) ok = issue_s(1);
      for (int j = 0; ok && j < T; ++j) {
        // dP_{j+1} as soon as the warpgroups hold dP_j in registers.
        if (j + 1 < T) {
          if (!(ok = mbar_wait(bar_dpfree, j & 1, ab))) break;
          tc_fence_after();
          if (!(ok = issue_dp())) break;
        }
        if (!(ok = mbar_wait(bar_ds, j & 1, ab))) break;
        tc_fence_after();
        // dQ += dS_j K_j (dS_j halves at columns 0 and 64 of S_j's buffer;
        // B = K_j MN-major)
        {
          const uint32_t sb = tmem + C::kColS + 128u * (j & 1);
          uint32_t a[kK];
#pragma unroll
          for (int k = 0; k < kK; ++k) a[k] = split_col(sb, sb + 64, k);
          uint64_t b[kK];
          mnmaj128_steps(sK + kq.stage * W::kTile, b);
          mma_ts_k(tmem + C::kColdQ, a, b, idQ, j > 0 ? 1u : 0u);
        }
        if (j == T - 1) mma_commit(bar_final);
        mma_commit(bar_kempty(kq.stage));
        kq.next();
        // S_{j+2} overwrites dS_j: the product above reads it first (in order).
        if (j + 2 < T && !(ok = issue_s(j + 2))) break;
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int x = (warp >> 2) - 1;        // 0: key columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row = TMEM lane
    const int grow = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t cdp = C::kColdP + 64u * x;
    const long long ridx = static_cast<long long>(bh) * a.N + grow;
    const float L2 = grow < a.N ? a.L[ridx] * kLog2e : 0.f;
    const float Dr = grow < a.N ? a.D[ridx] : 0.f;
    bool ok = true;
    const uint32_t hh = static_cast<uint32_t>(bh % a.H), bb = static_cast<uint32_t>(b);
    int kb = next_block(bmr, 1, jlo, jhi);
    for (int j = 0; j < T; ++j, kb = next_block(bmr, 1, kb + 1, jhi)) {
      const int key0 = kb * kT + 64 * x;  // first key column of this half
      // Dropout keep bits of this row's 64 keys, drawn before S arrives.
      uint64_t km = 0;
      if constexpr (DROP)
        km = keep32(static_cast<uint32_t>(key0), static_cast<uint32_t>(grow), hh, bb, a.seed_lo,
                    a.seed_hi, a.drop_thr) |
             static_cast<uint64_t>(keep32(static_cast<uint32_t>(key0 + 32),
                                          static_cast<uint32_t>(grow), hh, bb, a.seed_lo,
                                          a.seed_hi, a.drop_thr))
                 << 32;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s(j & 1), (j >> 1) & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool band = (a.causal != 0) | (a.window >= 0);
      const bool need_mask = (key0 + 64 > kv_limit) || (band && key0 + 63 > q0) ||
                             (a.window >= 0 && key0 < q0 + kT - 1 - a.window);
      uint32_t sr[2][32];
      tmem_ld32(tl + C::kColS + 128u * (j & 1) + 64u * x, sr[0]);
      tmem_ld32(tl + C::kColS + 128u * (j & 1) + 64u * x + 32, sr[1]);
      tmem_wait_ld();
      float p[64];
      {
        // p = 2^(s scale log2e - L log2e) on packed fp32 pairs
        const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2), nL2 = f2_pack(-L2, -L2);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])),
                             scl2, nL2),
                      t0, t1);
            p[32 * c + 2 * e] = ex2(t0);
            p[32 * c + 2 * e + 1] = ex2(t1);
          }
        }
      }
      // One branch per step; inside, selects only.
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int key = key0 + e;
          const bool keep = visible(grow, key, kv_limit, a.causal, a.window);
          p[e] = keep ? p[e] : 0.f;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp, j & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld32(tl + cdp, dr[0]);
      tmem_ld32(tl + cdp + 32, dr[1]);
      tmem_wait_ld();
      // dP_j is in registers: the MMA warp may overwrite the dP buffer.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dpfree);
      uint32_t w[32];
      // dS = P o (dP - D); with dropout dP = (dO V^T) Z / q.
      const uint64_t Dr2 = f2_pack(Dr, Dr);
      auto ds_step = [&](auto drop) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float g0 = __uint_as_float(dr[e >> 4][(2 * e) & 31]);
          float g1 = __uint_as_float(dr[e >> 4][(2 * e + 1) & 31]);
          if constexpr (decltype(drop)::value) {
            g0 = (km >> (2 * e)) & 1u ? g0 * a.drop_scale : 0.f;
            g1 = (km >> (2 * e + 1)) & 1u ? g1 * a.drop_scale : 0.f;
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[2 * e], p[2 * e + 1]), f2_sub(f2_pack(g0, g1), Dr2)), d0, d1);
          w[e] = pack_bf16(d0, d1);
        }
      };
      if constexpr (DROP)
        ds_step(std::true_type{});
      else
        ds_step(std::false_type{});
      // dS over the first half of this warpgroup's columns of S_j's buffer
      tmem_st32(tl + C::kColS + 128u * (j & 1) + 64u * x, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
    if (ok && T > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, ab));
      tc_fence_after();
    }
    // Both warpgroups agree (named barrier 1 over all 256 softmax threads).
    ok = bar_and_w(1, 256, ok && *abort_flag == 0);
    if (ok && x == 0) {
      // ------------------------------------------------------------ epilogue
      // dQ * scale -> bf16 -> the idle Q tile (swizzled like TMA) -> TMA store
      // (rows >= N are clipped).  Every lane takes part in the loads.
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        if (T > 0) {
          tmem_ld32(tl + C::kColdQ + 32 * c, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        const int atom = (32 * c) / 64;
        const int chunk0 = ((32 * c) % 64) / 8;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(r[8 * t + 0]) * a.scale, __uint_as_float(r[8 * t + 1]) * a.scale);
          v.y = pack_bf16(__uint_as_float(r[8 * t + 2]) * a.scale, __uint_as_float(r[8 * t + 3]) * a.scale);
          v.z = pack_bf16(__uint_as_float(r[8 * t + 4]) * a.scale, __uint_as_float(r[8 * t + 5]) * a.scale);
          v.w = pack_bf16(__uint_as_float(r[8 * t + 6]) * a.scale, __uint_as_float(r[8 * t + 7]) * a.scale);
          const int phys = (chunk0 + t) ^ (row & 7);
          *reinterpret_cast<uint4*>(smem + C::kOffQ + atom * 16384 + row * 128 + phys * 16) = v;
        }
      }
      fence_proxy_async_smem();
      bar_sync_w(2, 128);
      if (quarter == 0 && lane == 0) {
        for (int c = 0; c < W::kAtoms; ++c) tma_store_3d(&tmdQ, sQ + c * 16384, c * 64, q0, bh);
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

template <typename Kern>
cudaError_t set_smem_w(Kern k, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !done[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

template <int HD, bool DROP>
cudaError_t launch_dkdv_w(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdArgs& a, cudaStream_t stream) {
  static bool done[64] = {};
  cudaError_t e = set_smem_w(fa_bwd_dkdv_wide_kernel<HD, DROP>, KvW<HD>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(a.n_ktiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdArgs ag = a;
  ag.tile_group = tile_group(a.causal != 0 && a.window < 0, a.n_ktiles, a.BH, 1,
                             4ll * a.N * HD);  // Q and dO of a head, bf16
  fa_bwd_dkdv_wide_kernel<HD, DROP><<<static_cast<unsigned>(grid), kThreads, KvW<HD>::kSmemBytes,
                                stream>>>(tmQ, tmK, tmV, tmdO, ag);
  return cudaGetLastError();
}

template <int HD, bool DROP>
cudaError_t launch_dq_w(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const CUtensorMap& tmdQ, const BwdArgs& a,
                        cudaStream_t stream) {
  static bool done[64] = {};
  cudaError_t e = set_smem_w(fa_bwd_dq_wide_kernel<HD, DROP>, QW<HD>::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(a.n_qtiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdArgs ag = a;
  ag.tile_group = tile_group(a.causal != 0 && a.window < 0, a.n_qtiles, a.BH, 1,
                             4ll * a.N * HD);  // K and V of a head, bf16
  fa_bwd_dq_wide_kernel<HD, DROP><<<static_cast<unsigned>(grid), kThreads, QW<HD>::kSmemBytes,
                              stream>>>(tmQ, tmK, tmV, tmdO, tmdQ, ag);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_wide(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                 const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
      return a.drop_thr ? launch_dkdv_w<64, true>(tmQ, tmK, tmV, tmdO, a, stream)
                        : launch_dkdv_w<64, false>(tmQ, tmK, tmV, tmdO, a, stream);
    case 128:
      return a.drop_thr ? launch_dkdv_w<128, true>(tmQ, tmK, tmV, tmdO, a, stream)
                        : launch_dkdv_w<128, false>(tmQ, tmK, tmV, tmdO, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq_wide(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                               const CUtensorMap& tmV, const CUtensorMap& tmdO,
                               const CUtensorMap& tmdQ, const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
      return a.drop_thr ? launch_dq_w<64, true>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream)
                        : launch_dq_w<64, false>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
    case 128:
      return a.drop_thr ? launch_dq_w<128, true>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream)
                        : launch_dq_w<128, false>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
