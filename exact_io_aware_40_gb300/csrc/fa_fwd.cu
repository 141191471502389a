// fa_fwd.cu -- forward pass of exact attention on sm_103a.
//
// Method (the pages' statement of it): Q is cut into row blocks Q_i and K, V
// into row blocks K_j, V_j (study notes "FlashAttention学习笔记", section
// "分块计算整体流程(Tiling)"); for each block pair S_ij = Q_i K_j^T is computed,
// masked and pushed through a safe softmax whose running row maximum and row
// sum are updated as blocks arrive (apxml.com chapter "高效注意力算法实现
// (FlashAttention)", section "在线Softmax"; fmread.com summary section 三.2
// "增量Softmax计算"), and O_ij = P_ij V_j is accumulated.  Everything between
// the loads of Q, K, V and the store of O and L stays on chip (study notes,
// section "Kernel融合").
//
// GB300 mapping: one 128-row query block per CTA, key blocks of 64 rows.
//   - TMEM: two S buffers of 64 columns (S_j = Q K_j^T double-buffered so the
//     product for block j+1 overlaps the softmax of block j) and O (d
//     columns) -- 256 columns for d <= 128, so with under 100 KB of shared
//     memory two CTAs share an SM and one CTA's set-up, pipeline fill and
//     epilogue overlap the other's products (d = 256: 512 columns, one CTA);
//   - warp 0: TMA producer (Q once; K_j, V_j through 2-stage rings, 128-byte
//     swizzle, 64-column atoms); warp 1: tcgen05 issuer (one thread) and TMEM
//     owner; warps 2-5: softmax (thread = query row = TMEM lane): reads its S
//     row, masks, updates (m, l), writes P (bf16) back to TMEM for the PV
//     product, rescales its O row only when the row maximum grew by more than
//     2^8, and finally writes O / l (TMA store) and L.
// The commit that announces S(j+1) also covers every earlier product of the
// issuing thread, PV(j) included, so O is stable whenever the softmax holds a
// fresh S: the rescale needs no extra wait.
// Key blocks are visited in the order of the tile walk of masks.cuh: the
// contiguous range that kv_len, causal and window leave, thinned by the block
// mask; elements are masked only in blocks that cross a boundary.
// Loop order: query block outer (per CTA), key block inner, so O stays in TMEM
// for the whole loop; the study notes' K/V-outer order computes the same
// result (they only differ in which operand is reused on chip).
#include <type_traits>

#include "kernels.h"
#include "masks.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBR = 128;      // query rows per CTA (MMA M)
constexpr int kBC = 64;       // keys per block (MMA N of S, K of PV)
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if m grows by > 8
constexpr float kLn2 = 0.693147180559945309f;

template <int HD>
struct Cfg {
  static constexpr int kAtoms = HD / 64;                 // 64-column swizzle atoms
  static constexpr int kAtomBytes = kBR * 128;           // 128 rows x 128 B (Q, O)
  static constexpr int kTileBytes = kAtoms * kAtomBytes; // one 128-row bf16 tile
  static constexpr int kKVAtom = kBC * 128;              // 64 rows x 128 B (K, V)
  static constexpr int kKVTile = kAtoms * kKVAtom;
  static constexpr int kKSt = 2;
  static constexpr int kVSt = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kKSt * kKVTile;
  static constexpr int kOffBar = kOffV + kVSt * kKVTile;
  // barriers: q_full, k_full[], k_empty[], v_full[], v_empty[], s_full[2],
  // p_full[2], o_done, drain
  static constexpr int kNumBar = 1 + 2 * kKSt + 2 * kVSt + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 16;
  // d <= 128: at least 100 KB, so no more than two CTAs (two 256-column TMEM
  // allocations) are resident on an SM.
  static constexpr int kSmemBytes =
      HD == 256 ? kUsed + 1024 : (kUsed + 1024 > 102400 ? kUsed + 1024 : 102400);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM columns: S buffers at 0 and 64, O at 128
  static constexpr uint32_t kColO = 128;
  static constexpr uint32_t kTmemCols = HD == 256 ? 512 : 256;
  static constexpr int kMinBlocks = HD == 256 ? 1 : 2;
};

__device__ __forceinline__ uint32_t s_col(int b) { return b ? 64u : 0u; }

// Named barrier over 128 threads that also returns the AND of `pred` over them.
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

// DROP: dropout on P; MASKX: a sliding window or a block mask.  Separate
// instantiations, so the kernel without them carries none of their code
// (the window and block-mask terms cost the plain case a few per cent).
template <int HD, bool DROP, bool MASKX>
__global__ void __launch_bounds__(kThreads, Cfg<HD>::kMinBlocks)
    fa_fwd_1q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdArgs a) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t pad = ((raw_u32 + 1023u) & ~1023u) - raw_u32;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw_u32 + pad;

  const uint32_t sQ = sb + C::kOffQ;
  const uint32_t sK = sb + C::kOffK;
  const uint32_t sV = sb + C::kOffV;
  const uint32_t bar0 = sb + C::kOffBar;
  const uint32_t bar_q = bar0;
  auto bar_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (1 + C::kKSt + s); };
  auto bar_vfull = [&](int s) { return bar0 + 8u * (1 + 2 * C::kKSt + s); };
  auto bar_vempty = [&](int s) { return bar0 + 8u * (1 + 2 * C::kKSt + C::kVSt + s); };
  const uint32_t bar_sfull0 = bar0 + 8u * (1 + 2 * C::kKSt + 2 * C::kVSt);
  const uint32_t bar_pfull0 = bar_sfull0 + 16u;
  const uint32_t bar_odone = bar_pfull0 + 16u;
  const uint32_t bar_drain = bar_odone + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Longest query blocks (causal) first, in groups of ranks, head-major inside
  // a group: the CTAs in flight share a few K/V blocks per head in L2.
  int bh, qt;
  cta_tile(static_cast<int>(blockIdx.x), a.n_qtiles, a.BH, a.tile_group, &bh, &qt);
  qt = a.n_qtiles - 1 - qt;
  const int q0 = qt * kBR;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  // The 64-key blocks this query block visits: a range from the key padding,
  // causal and window terms, thinned by row qt of the block mask (whose
  // 128-key blocks are pairs of 64-key blocks).  Every role walks the same
  // list; warp 2 counts it.
  const int window = MASKX ? a.window : -1;
  int klo, khi;
  {
    int h = (kv_limit + kBC - 1) / kBC;
    if (a.causal || window >= 0) h = min(h, 2 * qt + 2);  // keys <= q0 + 127
    const int l = window >= 0 ? max(0, q0 - window) / kBC : 0;
    klo = l;
    khi = max(h, l);
  }
  const uint8_t* bmr =
      (MASKX && a.bmask) ? a.bmask + static_cast<long long>(qt) * a.nb : nullptr;
  auto next_kb = [&](int kb) -> int {  // next visited 64-key block at or after kb
    if constexpr (MASKX) {
      if (bmr == nullptr) return kb;
      while (kb < khi && !block_on(bmr, 1, kb >> 1)) ++kb;
    }
    return kb;
  };
  volatile int* n_steps = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  if (MASKX && warp == 2 && bmr != nullptr) {
    int n = 0;
    for (int b0 = klo; b0 < khi; b0 += 32) {
      const int kb = b0 + lane;
      n += __popc(__ballot_sync(0xffffffffu, kb < khi && block_on(bmr, 1, kb >> 1)));
    }
    if (lane == 0) *n_steps = n;
  }

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kKSt; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int s = 0; s < C::kVSt; ++s) {
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
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{a.err, abort_flag};
  // Without a block mask the list is the whole range (no count to read).
  const int T = bmr ? *n_steps : khi - klo;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar_q, C::kTileBytes);
      for (int c = 0; c < C::kAtoms; ++c)
        tma_load_3d(sQ + c * C::kAtomBytes, &tmQ, c * 64, q0, bh, bar_q, pol_q);
      int last_k[C::kKSt], last_v[C::kVSt];
      for (int s = 0; s < C::kKSt; ++s) last_k[s] = -1;
      for (int s = 0; s < C::kVSt; ++s) last_v[s] = -1;
      int kb = next_kb(klo);
      for (int j = 0; j < T; ++j, kb = next_kb(kb + 1)) {
        const int ks = j % C::kKSt, vs = j % C::kVSt;
        if (j >= C::kKSt && !mbar_wait(bar_kempty(ks), ((j / C::kKSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_kfull(ks), C::kKVTile);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(sK + ks * C::kKVTile + c * C::kKVAtom, &tmK, c * 64, kb * kBC, bh,
                      bar_kfull(ks), pol_kv);
        last_k[ks] = j;
        if (j >= C::kVSt && !mbar_wait(bar_vempty(vs), ((j / C::kVSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_vfull(vs), C::kKVTile);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(sV + vs * C::kKVTile + c * C::kKVAtom, &tmV, c * 64, kb * kBC, bh,
                      bar_vfull(vs), pol_kv);
        last_v[vs] = j;
      }
      if (*abort_flag) {
        // Unwinding: let the copies already issued land before the CTA exits.
        // Load j is the (j / stages)-th use of its stage, so its completion is
        // the phase of that parity.
        mbar_wait_drain(bar_q, 0);
        for (int s = 0; s < C::kKSt; ++s)
          if (last_k[s] >= 0) mbar_wait_drain(bar_kfull(s), (last_k[s] / C::kKSt) & 1);
        for (int s = 0; s < C::kVSt; ++s)
          if (last_v[s] >= 0) mbar_wait_drain(bar_vfull(s), (last_v[s] / C::kVSt) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t idS = idesc_bf16(kBR, kBC, false, false);
      constexpr uint32_t idO = idesc_bf16(kBR, HD, false, true);
      constexpr int kD = HD / 16, kC = kBC / 16;  // k-steps over d, over a key block
      // K-major operands: step k covers columns [16k, 16k+16) of d, i.e. atom
      // k/4, byte offset 32*(k%4) inside the 128-byte swizzled row.  The
      // resident Q tile's descriptors are built once.
      uint64_t aQ[kD];
      {
        const uint64_t d0 = sdesc_sw128(sQ, 16, 1024);
#pragma unroll
        for (int k = 0; k < kD; ++k) aQ[k] = sdesc_add(d0, (k >> 2) * C::kAtomBytes + (k & 3) * 32);
      }
      bool ok = mbar_wait(bar_q, 0, ab);
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1, vs = jj % C::kVSt;
        if (!mbar_wait(bar_pfull0 + 8u * bb, (jj >> 1) & 1, ab)) return false;
        if (!mbar_wait(bar_vfull(vs), (jj / C::kVSt) & 1, ab)) return false;
        tc_fence_after();
        // B = V_j, MN-major: 16 key rows per step (two 8-row groups, SBO
        // 1024 B); 64-column atoms of d are kKVAtom apart (LBO).  A = P_j
        // from TMEM, 8 columns (16 bf16 keys) per step.
        uint64_t b[kC];
        uint32_t a[kC];
        const uint64_t d0 = sdesc_sw128(sV + vs * C::kKVTile, C::kKVAtom, 1024);
        const uint32_t pcol = tmem + s_col(bb);
#pragma unroll
        for (int k = 0; k < kC; ++k) {
          b[k] = sdesc_add(d0, k * 2048);
          a[k] = pcol + 8u * k;
        }
        mma_ts_k(tmem + C::kColO, a, b, idO, jj > 0 ? 1u : 0u);
        mma_commit(bar_odone);
        mma_commit(bar_vempty(vs));
        return true;
      };
      for (int j = 0; ok && j < T; ++j) {
        const int bb = j & 1, ks = j % C::kKSt;
        if (j >= 2 && !mbar_wait(bar_odone, (j - 2) & 1, ab)) { ok = false; break; }
        if (!mbar_wait(bar_kfull(ks), (j / C::kKSt) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        {
          uint64_t b[kD];
          const uint64_t d0 = sdesc_sw128(sK + ks * C::kKVTile, 16, 1024);
#pragma unroll
          for (int k = 0; k < kD; ++k) b[k] = sdesc_add(d0, (k >> 2) * C::kKVAtom + (k & 3) * 32);
          mma_ss_k(tmem + s_col(bb), aQ, b, idS, 0u);
        }
        mma_commit(bar_sfull0 + 8u * bb);
        mma_commit(bar_kempty(ks));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(T - 1);
      // Drain: all MMAs issued above complete before TMEM is released.
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
    float lh_run = 0.f;                     // row sum of P rounded to bf16
    bool ok = true;
    const uint32_t hh = static_cast<uint32_t>(bh % a.H), bsq = static_cast<uint32_t>(b);
    const int q_last = min(q0 + kBR, a.N) - 1;  // last real query row of the block
    int kb = next_kb(klo);
    for (int j = 0; j < T; ++j, kb = next_kb(kb + 1)) {
      const int bb = j & 1;
      const int key0 = kb * kBC;
      // Dropout keep bits of this row's 64 keys, drawn before S arrives.
      uint64_t km = 0;
      if constexpr (DROP)
        km = keep32(static_cast<uint32_t>(key0), static_cast<uint32_t>(grow), hh, bsq, a.seed_lo,
                    a.seed_hi, a.drop_thr) |
             static_cast<uint64_t>(keep32(static_cast<uint32_t>(key0 + 32),
                                          static_cast<uint32_t>(grow), hh, bsq, a.seed_lo,
                                          a.seed_hi, a.drop_thr))
                 << 32;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull0 + 8u * bb, (j >> 1) & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tl + s_col(bb) + 32 * c, sr[c]);
      tmem_wait_ld();
      // Element masking only in blocks holding a key some row does not see
      // (the window terms kept apart: folded into one expression they change
      // how the compiler schedules the whole loop, which cost the plain case).
      bool need_mask = (key0 + kBC > kv_limit) || (a.causal && key0 + kBC - 1 > q0);
      if constexpr (MASKX)
        need_mask = need_mask || (window >= 0 && (key0 + kBC - 1 > q0 || key0 < q_last - window));
      if (need_mask) {
        if (!MASKX || window < 0) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int key = key0 + 32 * c + e;
              const bool keep = (key < kv_limit) & !((a.causal != 0) & (key > grow));
              sr[c][e] = keep ? sr[c][e] : __float_as_uint(-INFINITY);  // select, no branch
            }
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int key = key0 + 32 * c + e;
              const bool keep = visible(grow, key, kv_limit, a.causal, window);
              sr[c][e] = keep ? sr[c][e] : __float_as_uint(-INFINITY);
            }
        }
      }
      // Row max as a tree (independent partial maxima, no long dependency chain).
      float mxp[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mxp[t] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mxp[e & 7] = fmaxf(mxp[e & 7], __uint_as_float(sr[c][e]));
      const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                             fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      const float m_cand = fmaxf(m_run, mx * a.scale_log2);
      const bool grow_max = m_cand > m_run + kRescaleThreshold;
      const float m_new = grow_max ? m_cand : m_run;
      const float alpha = grow_max ? ex2(m_run - m_new) : 1.f;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // P = 2^(s * scale * log2e - m) with packed fp32 pairs (one FMA and one
      // add per two elements).  The row sum of P gives L.  O is divided by a
      // second sum, lh: in masked tiles it adds P rounded to bf16 -- the
      // weights the product actually applies to V -- and elsewhere P itself.
      // A row with fewer visible keys than a tile has no fully visible tile, so
      // for it lh is exactly the sum of the weights applied, which keeps its O
      // accurate; for longer rows the two sums differ by far less than the
      // bf16 rounding of O.
      const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2);
      const uint64_t nm2 = f2_pack(-m_use, -m_use);
      float sum_l, sum_h;
      // With dropout the product takes P * Z / q; L and the divisor of O stay
      // the sums of the undropped P.
      auto p_tile = [&](auto mode) {
        constexpr bool kRounded = decltype(mode)::value == 1;
        constexpr bool kDrop = decltype(mode)::value == 2;
        uint64_t se[2] = {0ull, 0ull}, sh[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])),
                             scl2, nm2),
                      t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            if constexpr (kDrop) {
              const int kk = 32 * c + 2 * e;
              pk[e] = pack_bf16((km >> kk) & 1u ? p0 * a.drop_scale : 0.f,
                                (km >> (kk + 1)) & 1u ? p1 * a.drop_scale : 0.f);
            } else {
              pk[e] = pack_bf16(p0, p1);
            }
            se[e & 1] = f2_add(se[e & 1], f2_pack(p0, p1));
            if constexpr (kRounded) sh[e & 1] = f2_add(sh[e & 1], bf16x2_to_f2(pk[e]));
          }
          // P occupies the first 64 columns of the S buffer (2 bf16 per column).
          tmem_st16(tl + s_col(bb) + 16 * c, pk);
        }
        float u0, u1;
        f2_unpack(f2_add(se[0], se[1]), u0, u1);
        sum_l = u0 + u1;
        sum_h = sum_l;
        if constexpr (kRounded) {
          f2_unpack(f2_add(sh[0], sh[1]), u0, u1);
          sum_h = u0 + u1;
        }
      };
      if constexpr (DROP)
        p_tile(std::integral_constant<int, 2>{});
      else if (need_mask)
        p_tile(std::integral_constant<int, 1>{});
      else
        p_tile(std::integral_constant<int, 0>{});
      l_run = l_run * alpha + sum_l;
      lh_run = lh_run * alpha + sum_h;
      m_run = m_new;
      if (j > 0 && __any_sync(0xffffffffu, grow_max)) {
        // O holds P_0..P_{j-1} V; rescale it once PV_{j-1} has landed.  (Only
        // PV_{j-1} can be pending: PV_{j-2} completed before S_j was issued, so
        // the parity of this wait is unambiguous even when earlier ones were
        // skipped.)
        if (!__all_sync(0xffffffffu, mbar_wait(bar_odone, (j - 1) & 1, ab))) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tl + C::kColO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tl + C::kColO + 32 * c, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull0 + 8u * bb);
    }
    if (ok && T > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_odone, (T - 1) & 1, ab));
      tc_fence_after();
    }
    // All four softmax warps take the same branch: AND of every thread's ok.
    ok = bar_and_128(1, ok && *abort_flag == 0);
    if (ok) {
      // ---------------------------------------------------------- epilogue
      const float inv_l = lh_run > 0.f ? 1.f / lh_run : 0.f;
      if (grow < a.N) {
        const float Lv = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        a.L[static_cast<long long>(bh) * a.N + grow] = Lv;
      }
      // O / l -> bf16 -> the (now idle) Q tile buffer, in the same swizzled
      // layout TMA uses, then one TMA store per 64-column atom.
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        if (T > 0) {
          tmem_ld32(tl + C::kColO + 32 * c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        const int atom = (32 * c) / 64;
        const int chunk0 = ((32 * c) % 64) / 8;  // 16-byte chunk within the 128-byte row
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * t + 0]) * inv_l, __uint_as_float(o[8 * t + 1]) * inv_l);
          v.y = pack_bf16(__uint_as_float(o[8 * t + 2]) * inv_l, __uint_as_float(o[8 * t + 3]) * inv_l);
          v.z = pack_bf16(__uint_as_float(o[8 * t + 4]) * inv_l, __uint_as_float(o[8 * t + 5]) * inv_l);
          v.w = pack_bf16(__uint_as_float(o[8 * t + 6]) * inv_l, __uint_as_float(o[8 * t + 7]) * inv_l);
          const int phys = (chunk0 + t) ^ (row & 7);
          *reinterpret_cast<uint4*>(smem + C::kOffQ + atom * C::kAtomBytes + row * 128 + phys * 16) = v;
        }
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (warp == 2 && lane == 0) {
        for (int c = 0; c < C::kAtoms; ++c) tma_store_3d(&tmO, sQ + c * C::kAtomBytes, c * 64, q0, bh);
        bulk_commit();
        bulk_wait0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int HD, bool DROP, bool MASKX>
cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         const CUtensorMap& tmO, const FwdArgs& a, cudaStream_t stream) {
  using C = Cfg<HD>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_fwd_1q_kernel<HD, DROP, MASKX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = static_cast<long long>(a.n_qtiles) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdArgs ag = a;
  ag.tile_group = tile_group(a.causal != 0 && a.window < 0, a.n_qtiles, a.BH, C::kMinBlocks,
                             4ll * a.N * HD);  // K and V of a head, bf16
  fa_fwd_1q_kernel<HD, DROP, MASKX><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV,
                                                                                    tmO, ag);
  return cudaGetLastError();
}

}  // namespace

template <int HD>
cudaError_t launch_fwd_d(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdArgs& a,
                            cudaStream_t stream) {
  const bool maskx = a.window >= 0 || a.bmask != nullptr;
  if (a.drop_thr)
    return maskx ? launch_fwd_t<HD, true, true>(tmQ, tmK, tmV, tmO, a, stream)
                 : launch_fwd_t<HD, true, false>(tmQ, tmK, tmV, tmO, a, stream);
  return maskx ? launch_fwd_t<HD, false, true>(tmQ, tmK, tmV, tmO, a, stream)
               : launch_fwd_t<HD, false, false>(tmQ, tmK, tmV, tmO, a, stream);
}

cudaError_t launch_fwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdArgs& a,
                          cudaStream_t stream) {
  switch (d) {
    case 64: return launch_fwd_d<64>(tmQ, tmK, tmV, tmO, a, stream);
    case 128: return launch_fwd_d<128>(tmQ, tmK, tmV, tmO, a, stream);
    case 256: return launch_fwd_d<256>(tmQ, tmK, tmV, tmO, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
