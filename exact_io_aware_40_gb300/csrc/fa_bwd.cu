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
// Two kernels, neither with atomics, both with two softmax warpgroups that
// alternate so one warpgroup's exponentials overlap the other's products:
//
// fa_bwd_dkdv_kernel -- one CTA per 128-key block j (the study notes' K/V-outer
// loop order, section "分块计算整体流程(Tiling)"); dK_j and dV_j accumulate in
// TMEM while the CTA walks 64-row query steps i, even steps in warpgroup A,
// odd steps in warpgroup B:
//   S^T = K_j Q_i^T, dP^T = V_j dO_i^T (keys on TMEM lanes); P^T = exp2(S^T
//   scale log2e - L log2e) -> bf16 into TMEM; dS^T = P^T o (dP^T - D) -> bf16
//   into TMEM; dV += P^T dO_i, dK += dS^T Q_i (A operands from TMEM).
// fa_bwd_dq_kernel -- one CTA per pair of 128-row query blocks (like the
// forward); dQ accumulates in TMEM over 64-key steps j:
//   S = Q K_j^T, dP = dO V_j^T (queries on TMEM lanes, so L_i and D_i are
//   per-thread constants); dS = P o (dP - D) -> bf16 into TMEM;
//   dQ += dS K_j; finally dQ * scale -> bf16 -> TMA store.
// The cost is that S and dP are computed twice (7 products per tile pair
// instead of 5); in exchange dQ needs no fp32 accumulator, no reductions, and
// is deterministic.
#include "kernels.h"
#include <type_traits>

#include "masks.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

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
__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Descriptors of the K k-steps of a K-major operand whose 64-column atoms
// are `atom` bytes apart: step k covers columns [16k, 16k+16) of d (atom k/4,
// 32 B per step).
template <int K>
__device__ __forceinline__ void kmaj_steps(uint32_t base, uint32_t atom, uint64_t (&d)[K]) {
  const uint64_t d0 = sdesc_sw128(base, 16, 1024);
#pragma unroll
  for (int k = 0; k < K; ++k) d[k] = sdesc_add(d0, (k >> 2) * atom + (k & 3) * 32);
}
// The same for an MN-major operand (rows = reduction dim): step k covers rows
// [16k, 16k+16) (two 8-row groups, SBO 1024 B); 64-column atoms are `atom`
// bytes apart (LBO).
template <int K>
__device__ __forceinline__ void mnmaj_steps(uint32_t base, uint32_t atom, uint64_t (&d)[K]) {
  const uint64_t d0 = sdesc_sw128(base, atom, 1024);
#pragma unroll
  for (int k = 0; k < K; ++k) d[k] = sdesc_add(d0, k * 2048);
}

// The steps of S rows (or keys) a CTA visits: the 128-blocks of a range from
// the mask terms, thinned by a block-mask row or column (`m`, consecutive
// blocks `stride` bytes apart; nullptr keeps all), each cut into steps of S,
// and those of the block holding `limit` only up to it.  Every role walks the
// same steps with its own cursor.
template <int S>
struct StepWalk {
  const uint8_t* m;
  int stride, hi, limit, blk, sub;
  __device__ __forceinline__ void init(const uint8_t* m_, int stride_, int lo, int hi_,
                                       int limit_) {
    m = m_;
    stride = stride_;
    hi = hi_;
    limit = limit_;
    sub = 0;
    blk = next_block(m, stride, lo, hi);
  }
  __device__ __forceinline__ int pos() const { return blk * kMaskBlock + sub * S; }
  __device__ __forceinline__ void next() {
    ++sub;
    if (sub * S == kMaskBlock || pos() >= limit) {
      sub = 0;
      blk = next_block(m, stride, blk + 1, hi);
    }
  }
};
// Number of steps of such a walk; called by a whole warp.
template <int S>
__device__ __forceinline__ int count_steps(const uint8_t* m, int stride, int lo, int hi,
                                           int limit) {
  int n = count_blocks(m, stride, lo, hi) * (kMaskBlock / S);
  const int lb = (limit - 1) / kMaskBlock;  // the block holding the last position
  if (limit > 0 && lb >= lo && lb < hi && block_on(m, stride, lb)) {
    const int in_last = (limit - lb * kMaskBlock + S - 1) / S;
    n -= kMaskBlock / S - in_last;
  }
  return n;
}

// ===========================================================================
// dK, dV
// ===========================================================================
constexpr int kKeys = 128;  // keys per CTA (MMA M)

// HD: head dim; DH: columns of dK/dV this CTA accumulates (HD, or HD/2 when
// d = 256 and the two halves go to two CTAs); QS: query rows per step.
template <int HD, int DH, int QS>
struct KvCfg {
  static constexpr int kAtoms = HD / 64;
  static constexpr int kHalves = HD / DH;
  static constexpr int kKVAtom = 128 * 128;          // 128 rows x 128 B
  static constexpr int kKVTile = kAtoms * kKVAtom;
  static constexpr int kQAtom = QS * 128;            // QS rows x 128 B
  static constexpr int kQTile = kAtoms * kQAtom;
  static constexpr int kSt = HD == 256 ? 3 : 4;      // Q/dO ring depth
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kKVTile;
  static constexpr int kOffQ = 2 * kKVTile;
  static constexpr int kOffdO = kOffQ + kSt * kQTile;
  static constexpr int kOffLD = kOffdO + kSt * kQTile;   // kSt x (L2[QS], D[QS])
  static constexpr int kOffBar = kOffLD + kSt * 8 * QS;
  // kv, qdo_full[kSt], qdo_empty[kSt], ld_full[kSt], s[2], dp[2], p[2], ds[2],
  // final, drain
  static constexpr int kNumBar = 1 + 3 * kSt + 8 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: warpgroup x owns S^T at 2 QS x (P^T over its first QS/2 columns)
  // and dP^T at 2 QS x + QS (dS^T over its first QS/2 columns); dV, dK at 256.
  static constexpr uint32_t kColdV = 256, kColdK = 256 + DH;
  static_assert(4 * QS <= 256 && 256 + 2 * DH <= 512, "TMEM budget");
};

// DROP: dropout on P; MASKX: a sliding window or a block mask (separate
// instantiations, as in the other kernels).
template <int HD, int DH, int QS, bool DROP, bool MASKX>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdArgs a) {
  using C = KvCfg<HD, DH, QS>;
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
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (1 + C::kSt + s); };
  auto bar_ld_full = [&](int s) { return bar0 + 8u * (1 + 2 * C::kSt + s); };
  const uint32_t barx = bar0 + 8u * (1 + 3 * C::kSt);
  auto bar_s = [&](int x) { return barx + 8u * x; };
  auto bar_dp = [&](int x) { return barx + 16u + 8u * x; };
  auto bar_p = [&](int x) { return barx + 32u + 8u * x; };
  auto bar_ds = [&](int x) { return barx + 48u + 8u * x; };
  const uint32_t bar_final = barx + 64u, bar_drain = barx + 72u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Head-major order; small kt (most work under causal) first; the column
  // halves of one key block (d = 256) are neighbours.
  const int half = static_cast<int>(blockIdx.x % C::kHalves);
  const int blk = static_cast<int>(blockIdx.x / C::kHalves);
  const int bh = blk / a.n_ktiles;
  const int kt = blk % a.n_ktiles;
  const int k0 = kt * kKeys;
  const int b = bh / a.H;
  const int hatom = half * (DH / 64);  // first 64-column atom of this CTA's half
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  // Query steps of QS rows: the visible 128-row query blocks (a range from the
  // key padding, causal and window terms, thinned by column kt of the block
  // mask), each cut into steps, the last one up to row N.
  const int window = MASKX ? a.window : -1;
  int ilo, ihi;
  query_block_range(kt, a.nb, kv_limit, a.causal, window, &ilo, &ihi);
  const uint8_t* bmc = (MASKX && a.bmask) ? a.bmask + kt : nullptr;  // column kt, stride nb
  const int n_iter = count_steps<QS>(bmc, a.nb, ilo, ihi, a.N);

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < C::kSt; ++s) {
      mbar_init(bar_qdo_full(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
      mbar_init(bar_ld_full(s), 32);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_s(x), 1);
      mbar_init(bar_dp(x), 1);
      mbar_init(bar_p(x), 4);
      mbar_init(bar_ds(x), 4);
    }
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
        for (int c = 0; c < C::kAtoms; ++c) {
          tma_load_3d(sK + c * C::kKVAtom, &tmK, c * 64, k0, bh, bar_kv, pol_kv);
          tma_load_3d(sV + c * C::kKVAtom, &tmV, c * 64, k0, bh, bar_kv, pol_kv);
        }
      }
      int last[C::kSt];
      for (int t = 0; t < C::kSt; ++t) last[t] = -1;
      StepWalk<QS> walk;
      walk.init(bmc, a.nb, ilo, ihi, a.N);
      for (int it = 0; it < n_iter; ++it, walk.next()) {
        const int st = it % C::kSt;
        const int q0 = walk.pos();
        if (it >= C::kSt &&
            !__all_sync(0xffffffffu, mbar_wait(bar_qdo_empty(st), ((it / C::kSt) & 1) ^ 1, ab)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_qdo_full(st), 2 * C::kQTile);
          for (int c = 0; c < C::kAtoms; ++c) {
            tma_load_3d(sQ + st * C::kQTile + c * C::kQAtom, &tmQ, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
            tma_load_3d(sdO + st * C::kQTile + c * C::kQAtom, &tmdO, c * 64, q0, bh,
                        bar_qdo_full(st), pol_q);
          }
        }
        last[st] = it;
        float* L2 = sLD + st * 2 * QS;
        float* Dv = L2 + QS;
        const long long rbase = static_cast<long long>(bh) * a.N;
#pragma unroll
        for (int e = 0; e < QS / 32; ++e) {
          const int r = lane * (QS / 32) + e;
          const int q = q0 + r;
          L2[r] = q < a.N ? -(a.L[rbase + q] * kLog2e) : 0.f;  // negated: the FMA adds it
          Dv[r] = q < a.N ? a.D[rbase + q] : 0.f;
        }
        mbar_arrive(bar_ld_full(st));
      }
      if (lane == 0 && *abort_flag) {
        mbar_wait_drain(bar_kv, 0);
        for (int s = 0; s < C::kSt; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar_qdo_full(s), (last[s] / C::kSt) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = idesc_bf16(kKeys, QS, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(kKeys, DH, false, true);  // dV, dK
      constexpr int kD = HD / 16, kQ = QS / 16;  // k-steps over d, over a query step
      // Built once: descriptors of the resident K and V tiles.
      uint64_t aK[kD], aV[kD];
      kmaj_steps(sK, C::kKVAtom, aK);
      kmaj_steps(sV, C::kKVAtom, aV);
      // S^T(i), dP^T(i) into warpgroup (i & 1)'s columns; sp is the Q/dO
      // stage of the next step issued (one call per step, in order).
      RingPos<C::kSt> sp;
      auto issue_s_dp = [&](int it) -> bool {
        const int st = sp.stage, x = it & 1;
        if (!mbar_wait(bar_qdo_full(st), sp.phase, ab)) return false;
        sp.next();
        tc_fence_after();
        uint64_t b[kD];
        kmaj_steps(sQ + st * C::kQTile, C::kQAtom, b);
        mma_ss_k(tmem + 2u * QS * x, aK, b, idS, 0u);
        mma_commit(bar_s(x));
        kmaj_steps(sdO + st * C::kQTile, C::kQAtom, b);
        mma_ss_k(tmem + 2u * QS * x + QS, aV, b, idS, 0u);
        mma_commit(bar_dp(x));
        return true;
      };
      bool ok = mbar_wait(bar_kv, 0, ab);
      if (ok) ok = issue_s_dp(0);
      if (ok && n_iter > 1) ok = issue_s_dp(1);
      // Step it: dK(it-1), then S^T/dP^T(it+1) into the columns step it-1 has
      // released, then dV(it).
      int st_cur = 0, st_prev = 0;  // Q/dO stages of steps it and it - 1
      for (int it = 0; ok && it <= n_iter; ++it) {
        if (it >= 1) {
          const int pv = it - 1, y = pv & 1, st = st_prev;
          if (!(ok = mbar_wait(bar_ds(y), (pv >> 1) & 1, ab))) break;
          tc_fence_after();
          {
            uint32_t a[kQ];
            uint64_t b[kQ];
#pragma unroll
            for (int k = 0; k < kQ; ++k) a[k] = tmem + 2u * QS * y + QS + k * 8;
            mnmaj_steps(sQ + st * C::kQTile + hatom * C::kQAtom, C::kQAtom, b);
            mma_ts_k(tmem + C::kColdK, a, b, idKV, pv > 0 ? 1u : 0u);
          }
          mma_commit(bar_qdo_empty(st));
          // S^T(it+1) overwrites P^T(it-1) and dP^T(it+1) overwrites dS^T(it-1):
          // dV(it-1) and dK(it-1) were issued first (MMAs execute in order).
          if (it + 1 < n_iter && !(ok = issue_s_dp(it + 1))) break;
        }
        if (it < n_iter) {
          const int x = it & 1, st = st_cur;
          if (!(ok = mbar_wait(bar_p(x), (it >> 1) & 1, ab))) break;
          tc_fence_after();
          uint32_t a[kQ];
          uint64_t b[kQ];
#pragma unroll
          for (int k = 0; k < kQ; ++k) a[k] = tmem + 2u * QS * x + k * 8;
          mnmaj_steps(sdO + st * C::kQTile + hatom * C::kQAtom, C::kQAtom, b);
          mma_ts_k(tmem + C::kColdV, a, b, idKV, it > 0 ? 1u : 0u);
        }
        st_prev = st_cur;
        st_cur = st_cur + 1 == C::kSt ? 0 : st_cur + 1;
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int x = (warp >> 2) - 1;        // warpgroup: 0 = even steps, 1 = odd steps
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;   // key row = TMEM lane
    const int key = k0 + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t cs = 2u * QS * x, cdp = 2u * QS * x + QS;
    const bool key_ok = key < kv_limit;
    bool ok = true;
    StepWalk<QS> walk;  // this warpgroup's steps: x, x + 2, ...
    walk.init(bmc, a.nb, ilo, ihi, a.N);
    if (x) walk.next();
    for (int it = x, n = 0; it < n_iter; it += 2, ++n, walk.next(), walk.next()) {
      const int st = it % C::kSt;
      const int q0 = walk.pos();
      const float* L2 = sLD + st * 2 * QS;
      const float* Dv = L2 + QS;
      // Dropout keep bits of this thread's key for the step's QS queries (the
      // warp draws them together).
      uint32_t km = 0;
      if constexpr (DROP) {
        static_assert(QS == 32, "keep bits for 32-query steps");
        km = keep32_transposed(static_cast<uint32_t>(k0 + quarter * 32), static_cast<uint32_t>(q0),
                               static_cast<uint32_t>(bh % a.H), static_cast<uint32_t>(b), a.seed_lo,
                               a.seed_hi, a.drop_thr);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_ld_full(st), (it / C::kSt) & 1, ab) &&
                                       mbar_wait(bar_s(x), n & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool band = (a.causal != 0) | (window >= 0);
      const bool need_mask = !key_ok || (q0 + QS > a.N) || (band && q0 < k0 + kKeys - 1) ||
                             (window >= 0 && k0 < q0 + QS - 1 - window);
      float p[QS];
#pragma unroll
      for (int c = 0; c < QS / 32; ++c) {
        uint32_t sr[32];
        tmem_ld32(tl + cs + 32 * c, sr);
        tmem_wait_ld();
        uint32_t w[16];
        // p = 2^(s^T scale log2e - L log2e) on packed fp32 pairs (the ring
        // holds -L log2e)
        const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2);
        const uint64_t* nL2 = reinterpret_cast<const uint64_t*>(L2 + 32 * c);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                           scl2, nL2[e]),
                    t0, t1);
          p[32 * c + 2 * e] = ex2(t0);
          p[32 * c + 2 * e + 1] = ex2(t1);
        }
        // One branch per chunk; inside, selects only (a branch per element
        // in the loop above costs more than the exponentials).
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int qg = q0 + 32 * c + e;
            const bool keep = (qg < a.N) & visible(qg, key, kv_limit, a.causal, window);
            p[32 * c + e] = keep ? p[32 * c + e] : 0.f;
          }
        }
        // dV takes the dropped weights P Z / q; p itself stays for dS^T.
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          if constexpr (DROP)
            w[e] = pack_bf16((km >> qa) & 1u ? p[qa] * a.drop_scale : 0.f,
                             (km >> (qa + 1)) & 1u ? p[qa + 1] * a.drop_scale : 0.f);
          else
            w[e] = pack_bf16(p[qa], p[qa + 1]);
        }
        tmem_st16(tl + cs + 16 * c, w);  // P^T: first 32 columns of the S^T buffer
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(x));

      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp(x), n & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < QS / 32; ++c) {
        uint32_t dr[32];
        tmem_ld32(tl + cdp + 32 * c, dr);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qa = 32 * c + 2 * e;
          // dS^T = P^T o (dP^T - D); with dropout dP^T = (V dO^T) Z / q.
          float g0 = __uint_as_float(dr[2 * e]), g1 = __uint_as_float(dr[2 * e + 1]);
          if constexpr (DROP) {
            g0 = (km >> qa) & 1u ? g0 * a.drop_scale : 0.f;
            g1 = (km >> (qa + 1)) & 1u ? g1 * a.drop_scale : 0.f;
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[qa], p[qa + 1]),
                           f2_sub(f2_pack(g0, g1), reinterpret_cast<const uint64_t*>(Dv)[qa >> 1])),
                    d0, d1);
          w[e] = pack_bf16(d0, d1);
        }
        // dS^T columns [16c, 16c+16) overwrite dP^T columns this thread has read.
        tmem_st16(tl + cdp + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds(x));
    }
    if (ok && n_iter > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final, 0, ab));
      tc_fence_after();
    }
    ok = bar_and(1 + x, 128, ok && *abort_flag == 0);
    if (ok) {
      // ------------------------------------------------------------ dV (A), dK (B)
      // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
      const bool store = key < a.N;
      const long long row = static_cast<long long>(bh) * a.N + (store ? key : 0);
      uint16_t* dst = (x == 0 ? a.dV : a.dK) + row * HD + half * DH;
      const uint32_t col = x == 0 ? C::kColdV : C::kColdK;
      const float mul = x == 0 ? 1.f : a.scale;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
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
constexpr int kQRows = 128;  // query rows per block (MMA M)

// QT: query blocks per CTA (2, or 1 for d = 256); KS: keys per step.
template <int HD, int QT, int KS>
struct QCfg {
  static constexpr int kAtoms = HD / 64;
  static constexpr int kQAtom = kQRows * 128;       // 128 rows x 128 B
  static constexpr int kQTile = kAtoms * kQAtom;
  static constexpr int kKAtom = KS * 128;           // KS rows x 128 B
  static constexpr int kKTile = kAtoms * kKAtom;
  static constexpr int kSt = 3;                     // K/V ring depth
  static constexpr int kOffQ = 0;                   // Q_A (, Q_B)
  static constexpr int kOffdO = QT * kQTile;        // dO_A (, dO_B)
  static constexpr int kOffK = 2 * QT * kQTile;
  static constexpr int kOffV = kOffK + kSt * kKTile;
  static constexpr int kOffBar = kOffV + kSt * kKTile;
  // q_full[2], kv_full[kSt], kv_empty[kSt], s[2], dp[2], ds[2], final[2], drain
  static constexpr int kNumBar = 2 + 2 * kSt + 8 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: block x owns S at 2 KS x and dP at 2 KS x + KS (dS over its first
  // KS/2 columns); dQ_A (, dQ_B) at 256 (and 256 + d).
  static constexpr uint32_t kColdQ = 256;
  static_assert(4 * KS <= 256 && 256 + QT * HD <= 512, "TMEM budget");
};

template <int HD, int QT, int KS, bool DROP, bool MASKX>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using C = QCfg<HD, QT, KS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sQ = sb + C::kOffQ, sdO = sb + C::kOffdO, sK = sb + C::kOffK, sV = sb + C::kOffV;
  const uint32_t bar0 = sb + C::kOffBar;
  auto bar_qfull = [&](int x) { return bar0 + 8u * x; };
  auto bar_kvfull = [&](int s) { return bar0 + 8u * (2 + s); };
  auto bar_kvempty = [&](int s) { return bar0 + 8u * (2 + C::kSt + s); };
  const uint32_t barx = bar0 + 8u * (2 + 2 * C::kSt);
  auto bar_s = [&](int x) { return barx + 8u * x; };
  auto bar_dp = [&](int x) { return barx + 16u + 8u * x; };
  auto bar_ds = [&](int x) { return barx + 32u + 8u * x; };
  auto bar_final = [&](int x) { return barx + 48u + 8u * x; };
  const uint32_t bar_drain = barx + 64u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Head-major order with the longest query blocks (causal) of a head first.
  const int n_pairs = (a.n_qtiles + QT - 1) / QT;
  const int bh = static_cast<int>(blockIdx.x / n_pairs);
  const int pr = n_pairs - 1 - static_cast<int>(blockIdx.x % n_pairs);
  const int qtA = QT * pr;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  static_assert(QT == 1, "one query block per CTA");
  constexpr bool hasB = false;
  // Key steps of KS keys: the visible 128-key blocks (a range from the key
  // padding, causal and window terms, thinned by row qtA of the block mask),
  // each cut into steps, the last one up to kv_len.
  const int window = MASKX ? a.window : -1;
  int jlo, jhi;
  key_block_range(qtA, kv_limit, a.causal, window, &jlo, &jhi);
  const uint8_t* bmr = (MASKX && a.bmask) ? a.bmask + static_cast<long long>(qtA) * a.nb : nullptr;
  const int TA = count_steps<KS>(bmr, 1, jlo, jhi, kv_limit);
  constexpr int TB = 0;
  const int T = TA;

  if (tid == 0) {
    mbar_init(bar_qfull(0), 1);
    mbar_init(bar_qfull(1), 1);
    for (int s = 0; s < C::kSt; ++s) {
      mbar_init(bar_kvfull(s), 1);
      mbar_init(bar_kvempty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_s(x), 1);
      mbar_init(bar_dp(x), 1);
      mbar_init(bar_ds(x), 4);
      mbar_init(bar_final(x), 1);
    }
    mbar_init(bar_drain, 1);
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

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0 && T > 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      for (int x = 0; x < (hasB ? 2 : 1); ++x) {
        mbar_arrive_expect_tx(bar_qfull(x), 2 * C::kQTile);
        for (int c = 0; c < C::kAtoms; ++c) {
          tma_load_3d(sQ + x * C::kQTile + c * C::kQAtom, &tmQ, c * 64, (qtA + x) * kQRows, bh,
                      bar_qfull(x), pol_q);
          tma_load_3d(sdO + x * C::kQTile + c * C::kQAtom, &tmdO, c * 64, (qtA + x) * kQRows, bh,
                      bar_qfull(x), pol_q);
        }
      }
      int last[C::kSt];
      for (int s = 0; s < C::kSt; ++s) last[s] = -1;
      StepWalk<KS> walk;
      walk.init(bmr, 1, jlo, jhi, kv_limit);
      for (int j = 0; j < T; ++j, walk.next()) {
        const int st = j % C::kSt;
        if (j >= C::kSt && !mbar_wait(bar_kvempty(st), ((j / C::kSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_kvfull(st), 2 * C::kKTile);
        for (int c = 0; c < C::kAtoms; ++c) {
          tma_load_3d(sK + st * C::kKTile + c * C::kKAtom, &tmK, c * 64, walk.pos(), bh,
                      bar_kvfull(st), pol_kv);
          tma_load_3d(sV + st * C::kKTile + c * C::kKAtom, &tmV, c * 64, walk.pos(), bh,
                      bar_kvfull(st), pol_kv);
        }
        last[st] = j;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar_qfull(0), 0);
        if (hasB) mbar_wait_drain(bar_qfull(1), 0);
        for (int s = 0; s < C::kSt; ++s)
          if (last[s] >= 0) mbar_wait_drain(bar_kvfull(s), (last[s] / C::kSt) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idS = idesc_bf16(kQRows, KS, false, false);  // S, dP
      constexpr uint32_t idQ = idesc_bf16(kQRows, HD, false, true);       // dQ
      constexpr int kD = HD / 16, kK = KS / 16;  // k-steps over d, over a key step
      // S_x(j), dP_x(j) into block x's columns
      // The K/V stage and phase of step j come with the call.
      auto issue_s_dp = [&](int x, int j, int st, uint32_t ph) -> bool {
        if (j == 0 && !mbar_wait(bar_qfull(x), 0, ab)) return false;
        if (!mbar_wait(bar_kvfull(st), ph, ab)) return false;
        tc_fence_after();
        uint64_t a[kD], b[kD];
        kmaj_steps(sQ + x * C::kQTile, C::kQAtom, a);
        kmaj_steps(sK + st * C::kKTile, C::kKAtom, b);
        mma_ss_k(tmem + 2u * KS * x, a, b, idS, 0u);
        mma_commit(bar_s(x));
        kmaj_steps(sdO + x * C::kQTile, C::kQAtom, a);
        kmaj_steps(sV + st * C::kKTile, C::kKAtom, b);
        mma_ss_k(tmem + 2u * KS * x + KS, a, b, idS, 0u);
        mma_commit(bar_dp(x));
        return true;
      };
      bool ok = true;
      if (TA > 0) ok = issue_s_dp(0, 0, 0, 0u);
      if (ok && TB > 0) ok = issue_s_dp(1, 0, 0, 0u);
      RingPos<C::kSt> cur, nxt;  // K/V stages of steps j and j + 1
      nxt.next();
      for (int j = 0; ok && j < T; ++j, cur.next(), nxt.next()) {
        const int st = cur.stage;
        for (int x = 0; x < 2 && ok; ++x) {
          const int Tx = x == 0 ? TA : TB;
          if (j >= Tx) continue;
          if (!(ok = mbar_wait(bar_ds(x), j & 1, ab))) break;
          tc_fence_after();
          // dQ_x += dS_x K_j (A = dS from TMEM, B = K_j MN-major)
          {
            uint32_t a[kK];
            uint64_t b[kK];
#pragma unroll
            for (int s = 0; s < kK; ++s) a[s] = tmem + 2u * KS * x + KS + s * 8;
            mnmaj_steps(sK + st * C::kKTile, C::kKAtom, b);
            mma_ts_k(tmem + C::kColdQ + static_cast<uint32_t>(HD) * x, a, b, idQ, j > 0 ? 1u : 0u);
          }
          if (j == Tx - 1) mma_commit(bar_final(x));
          // the last reader of K_j, V_j releases the stage
          if (x == 1 || j >= TB) mma_commit(bar_kvempty(st));
          // S_x(j+1) and dP_x(j+1) overwrite S_x(j) (read) and dS_x(j) (read by
          // the product just issued: MMAs execute in order).
          if (j + 1 < Tx) ok = issue_s_dp(x, j + 1, nxt.stage, nxt.phase);
        }
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int x = (warp >> 2) - 1;        // 0: block A (warps 4-7), 1: block B (warps 8-11)
    const int Tn = x == 0 ? TA : TB;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row = TMEM lane
    const int q0 = (qtA + x) * kQRows;
    const int grow = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t cs = 2u * KS * x, cdp = 2u * KS * x + KS;
    const uint32_t cq = C::kColdQ + static_cast<uint32_t>(HD) * x;
    const long long ridx = static_cast<long long>(bh) * a.N + grow;
    const float L2 = grow < a.N ? a.L[ridx] * kLog2e : 0.f;
    const float Dr = grow < a.N ? a.D[ridx] : 0.f;
    bool ok = true;
    StepWalk<KS> walk;
    walk.init(bmr, 1, jlo, jhi, kv_limit);
    for (int j = 0; j < Tn; ++j, walk.next()) {
      const int key0 = walk.pos();
      // Dropout keep bits of this row's KS keys, drawn before S arrives.
      uint32_t km = 0;
      if constexpr (DROP) {
        static_assert(KS == 32, "keep bits for 32-key steps");
        km = keep32(static_cast<uint32_t>(key0), static_cast<uint32_t>(grow),
                    static_cast<uint32_t>(bh % a.H), static_cast<uint32_t>(b), a.seed_lo,
                    a.seed_hi, a.drop_thr);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s(x), j & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool band = (a.causal != 0) | (window >= 0);
      const bool need_mask = (key0 + KS > kv_limit) || (band && key0 + KS - 1 > q0) ||
                             (window >= 0 && key0 < q0 + kQRows - 1 - window);
      uint32_t sr[KS / 32][32];
#pragma unroll
      for (int c = 0; c < KS / 32; ++c) tmem_ld32(tl + cs + 32 * c, sr[c]);
      tmem_wait_ld();
      float p[KS];
      {
        // p = 2^(s scale log2e - L log2e) on packed fp32 pairs
        const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2), nL2 = f2_pack(-L2, -L2);
#pragma unroll
        for (int c = 0; c < KS / 32; ++c) {
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
        for (int e = 0; e < KS; ++e) {
          const bool keep = visible(grow, key0 + e, kv_limit, a.causal, window);
          p[e] = keep ? p[e] : 0.f;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dp(x), j & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < KS / 32; ++c) {
        uint32_t dr[32];
        tmem_ld32(tl + cdp + 32 * c, dr);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // dS = P o (dP - D); with dropout dP = (dO V^T) Z / q.
          const int ka = 32 * c + 2 * e;
          float g0 = __uint_as_float(dr[2 * e]), g1 = __uint_as_float(dr[2 * e + 1]);
          if constexpr (DROP) {
            g0 = (km >> ka) & 1u ? g0 * a.drop_scale : 0.f;
            g1 = (km >> (ka + 1)) & 1u ? g1 * a.drop_scale : 0.f;
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[ka], p[ka + 1]), f2_sub(f2_pack(g0, g1), f2_pack(Dr, Dr))),
                    d0, d1);
          w[e] = pack_bf16(d0, d1);
        }
        // dS columns [16c, 16c+16) overwrite dP columns this thread has read.
        tmem_st16(tl + cdp + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds(x));
    }
    if (ok && Tn > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_final(x), 0, ab));
      tc_fence_after();
    }
    ok = bar_and(1 + x, 128, ok && *abort_flag == 0);
    if (ok && (x == 0 || hasB)) {
      // ------------------------------------------------------------ epilogue
      // dQ * scale -> bf16 -> the idle Q_x tile (swizzled like TMA) -> TMA
      // store (rows >= N are clipped).  Every lane takes part in the loads.
      const int qoff = C::kOffQ + x * C::kQTile;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        if (Tn > 0) {
          tmem_ld32(tl + cq + 32 * c, r);
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
          *reinterpret_cast<uint4*>(smem + qoff + atom * C::kQAtom + row * 128 + phys * 16) = v;
        }
      }
      fence_proxy_async_smem();
      bar_sync_n(1 + x, 128);
      if (quarter == 0 && lane == 0) {
        for (int c = 0; c < C::kAtoms; ++c)
          tma_store_3d(&tmdQ, sQ + x * C::kQTile + c * C::kQAtom, c * 64, q0, bh);
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
cudaError_t set_smem(Kern k, int bytes, bool (&done)[64]) {
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

template <int HD, int DH, int QS, bool DROP, bool MASKX>
cudaError_t launch_dkdv_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdArgs& a, cudaStream_t stream) {
  using C = KvCfg<HD, DH, QS>;
  static bool done[64] = {};
  cudaError_t e = set_smem(fa_bwd_dkdv_kernel<HD, DH, QS, DROP, MASKX>, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(a.n_ktiles) * a.BH * C::kHalves;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_dkdv_kernel<HD, DH, QS, DROP, MASKX>
      <<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmdO, a);
  return cudaGetLastError();
}

template <int HD, int QT, int KS, bool DROP, bool MASKX>
cudaError_t launch_dq_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const CUtensorMap& tmdQ, const BwdArgs& a,
                        cudaStream_t stream) {
  using C = QCfg<HD, QT, KS>;
  static bool done[64] = {};
  cudaError_t e = set_smem(fa_bwd_dq_kernel<HD, QT, KS, DROP, MASKX>, C::kSmemBytes, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((a.n_qtiles + QT - 1) / QT) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_bwd_dq_kernel<HD, QT, KS, DROP, MASKX>
      <<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmdO,
                                                                        tmdQ, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const BwdArgs& a,
                            cudaStream_t stream) {
  switch (d) {
    case 64:
    case 128: return launch_bwd_dkdv_wide(d, tmQ, tmK, tmV, tmdO, a, stream);
    case 256: {
      const bool maskx = a.window >= 0 || a.bmask != nullptr;
      if (a.drop_thr)
        return maskx ? launch_dkdv_t<256, 128, 32, true, true>(tmQ, tmK, tmV, tmdO, a, stream)
                     : launch_dkdv_t<256, 128, 32, true, false>(tmQ, tmK, tmV, tmdO, a, stream);
      return maskx ? launch_dkdv_t<256, 128, 32, false, true>(tmQ, tmK, tmV, tmdO, a, stream)
                   : launch_dkdv_t<256, 128, 32, false, false>(tmQ, tmK, tmV, tmdO, a, stream);
    }
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                          const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
    case 128: return launch_bwd_dq_wide(d, tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
    case 256: {
      const bool maskx = a.window >= 0 || a.bmask != nullptr;
      if (a.drop_thr)
        return maskx ? launch_dq_t<256, 1, 32, true, true>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream)
                     : launch_dq_t<256, 1, 32, true, false>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
      return maskx ? launch_dq_t<256, 1, 32, false, true>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream)
                   : launch_dq_t<256, 1, 32, false, false>(tmQ, tmK, tmV, tmdO, tmdQ, a, stream);
    }
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
