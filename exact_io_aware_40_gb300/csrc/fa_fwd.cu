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
// This kernel serves the calls with a sliding window, a block mask or dropout
// (fa_fwd_1q.cu serves the rest).  GB300 mapping: one CTA owns two 128-row
// query blocks A and B of one (batch, head) and streams K_j, V_j once for both.
//   warp 0      TMA producer: Q_A, Q_B once; K_j, V_j through smem rings
//               (128-byte swizzle, 64-column atoms).
//   warp 1      tcgen05 issuer (one thread), per key block j:
//                 O_A += P_A V_j;  S_A = Q_A K_{j+1}^T;  O_B += P_B V_j;  S_B = Q_B K_{j+1}^T
//               so while one softmax warpgroup works on its S the tensor pipe
//               runs the other block's products.  Owns TMEM (512 columns:
//               S_A, S_B at 0 and 128, O_A, O_B at 256 and 256 + d).
//   warps 4-7   softmax of block A, warps 8-11 softmax of block B: thread t
//               owns query row t (= TMEM lane t); reads its S row, masks,
//               updates (m, l), writes P (bf16) over the first 64 columns of
//               its S buffer, rescales its O row in TMEM when the row maximum
//               grew by more than 2^8, and finally writes O / l (TMA store) and L.
// The commit that announces S_X(j+1) also covers every earlier product of the
// issuing thread, PV_X(j) included, so O_X is stable whenever its softmax
// warpgroup holds a fresh S_X: the rescale needs no extra wait.
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

constexpr int kBR = 128;      // query rows per block (MMA M)
constexpr int kBC = 128;      // keys per block (MMA N of S, K of PV)
constexpr int kThreads = 384;
// Registers per thread after setmaxnreg: warps 0-3 (producer, MMA) and the
// softmax warpgroups.  The dropout variant moves 8 more to the softmax, which
// also runs the random-number generator.
template <bool DROP> constexpr int kRegsLow = DROP ? 56 : 64;
template <bool DROP> constexpr int kRegsHigh = DROP ? 224 : 216;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if m grows by > 8
constexpr float kLn2 = 0.693147180559945309f;

template <int HD>
struct Cfg {
  static constexpr int kAtoms = HD / 64;                 // 64-column swizzle atoms
  static constexpr int kAtomBytes = kBR * 128;           // 128 rows x 128 B
  static constexpr int kTileBytes = kAtoms * kAtomBytes; // one 128-row bf16 tile
  static constexpr int kKSt = HD == 64 ? 3 : 2;
  static constexpr int kVSt = HD == 64 ? 3 : 2;
  static constexpr int kOffQ = 0;                          // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKSt * kTileBytes;
  static constexpr int kOffBar = kOffV + kVSt * kTileBytes;
  // q_full[2], k_full[], k_empty[], v_full[], v_empty[], s_full[2], p_full[2],
  // o_final[2], drain
  static constexpr int kNumBar = 2 + 2 * kKSt + 2 * kVSt + 2 + 2 + 2 + 1;
  // misc: tmem slot, abort flag, then the key-block walk (TA, TB, lo[2], hi[2], ulo, uhi)
  static constexpr int kOffMisc = kOffBar + kNumBar * 8;
  static constexpr int kUsed = kOffMisc + 48;
  static constexpr int kSmemBytes = kUsed + 1024;  // + alignment of the base
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kTmemCols = 512;
};

// Named barrier over `n` threads that also returns the AND of `pred` over them.
__device__ __forceinline__ bool bar_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// DROP: dropout on P (a separate instantiation, so the kernel without it
// carries none of its code).
template <int HD, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
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
  auto bar_qfull = [&](int x) { return bar0 + 8u * x; };
  auto bar_kfull = [&](int s) { return bar0 + 8u * (2 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (2 + C::kKSt + s); };
  auto bar_vfull = [&](int s) { return bar0 + 8u * (2 + 2 * C::kKSt + s); };
  auto bar_vempty = [&](int s) { return bar0 + 8u * (2 + 2 * C::kKSt + C::kVSt + s); };
  const uint32_t bar_s0 = bar0 + 8u * (2 + 2 * C::kKSt + 2 * C::kVSt);
  auto bar_sfull = [&](int x) { return bar_s0 + 8u * x; };
  auto bar_pfull = [&](int x) { return bar_s0 + 16u + 8u * x; };
  auto bar_ofinal = [&](int x) { return bar_s0 + 32u + 8u * x; };
  const uint32_t bar_drain = bar_s0 + 48u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Head-major order with the longest query blocks (causal) of a head first.
  const int n_pairs = (a.n_qtiles + 1) / 2;
  const int bh = static_cast<int>(blockIdx.x / n_pairs);
  const int pr = n_pairs - 1 - static_cast<int>(blockIdx.x % n_pairs);
  const int qtA = 2 * pr;
  const int b = bh / a.H;
  int kv_limit = a.N;
  if (a.kv_len != nullptr) kv_limit = min(max(a.kv_len[b], 0), a.N);
  const bool hasB = qtA + 1 < a.n_qtiles;
  // Key blocks each query block can see: a range from the key padding, causal
  // and window terms, thinned by the block mask.  The CTA walks the union of
  // both blocks' lists in increasing order (each K_j, V_j is loaded once);
  // block X processes the first T_X entries of the walk, and an entry inside
  // that prefix that X does not see is computed fully masked.
  // The walk (T_A, T_B, lo[2], hi[2], ulo, uhi) is set up once by warp 3.
  int* walk = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  if (warp == 3) {
    int loA, hiA, loB = 0, hiB = 0;
    key_block_range(qtA, kv_limit, a.causal, a.window, &loA, &hiA);
    if (hasB) key_block_range(qtA + 1, kv_limit, a.causal, a.window, &loB, &hiB);
    const int ulo = loB < hiB ? min(loA, loB) : loA;
    const int uhi = max(hiA, hiB);
    const uint8_t* bmA = a.bmask ? a.bmask + static_cast<long long>(qtA) * a.nb : nullptr;
    const uint8_t* bmB = (a.bmask && hasB) ? a.bmask + static_cast<long long>(qtA + 1) * a.nb : nullptr;
    // T_A, T_B: entry index (+1) of the last block each query block sees.
    int n = 0, ta = 0, tb = 0;
    for (int b0 = ulo; b0 < uhi; b0 += 32) {
      const int kb = b0 + lane;
      const bool sa = kb < uhi && kb >= loA && kb < hiA && block_on(bmA, 1, kb);
      const bool sb2 = kb < uhi && kb >= loB && kb < hiB && block_on(bmB, 1, kb);
      const uint32_t on = __ballot_sync(0xffffffffu, sa || sb2);
      const int idx = n + __popc(on & ((1u << lane) - 1u));
      ta = max(ta, sa ? idx + 1 : 0);
      tb = max(tb, sb2 ? idx + 1 : 0);
      n += __popc(on);
    }
    ta = __reduce_max_sync(0xffffffffu, ta);
    tb = __reduce_max_sync(0xffffffffu, tb);
    if (lane == 0) {
      walk[0] = ta;
      walk[1] = tb;
      walk[2] = loA;
      walk[3] = loB;
      walk[4] = hiA;
      walk[5] = hiB;
      walk[6] = ulo;
      walk[7] = uhi;
    }
  }

  if (tid == 0) {
    mbar_init(bar_qfull(0), 1);
    mbar_init(bar_qfull(1), 1);
    for (int s = 0; s < C::kKSt; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int s = 0; s < C::kVSt; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_sfull(x), 1);
      mbar_init(bar_pfull(x), 4);
      mbar_init(bar_ofinal(x), 1);
    }
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
  const int TA = walk[0], TB = walk[1];
  const int T = max(TA, TB);
  // Bounds re-read from shared memory at each use: kept in registers they
  // push the producer and softmax warps past their register budgets.
  volatile int* vw = walk;
  const int ulo = walk[6];
  auto sees = [&](int x, int kb) -> bool {  // does query block X see key block kb?
    const uint8_t* row = a.bmask ? a.bmask + static_cast<long long>(qtA + x) * a.nb : nullptr;
    return kb >= vw[2 + x] && kb < vw[4 + x] && block_on(row, 1, kb);
  };
  auto next_kb = [&](int kb) -> int {  // next entry of the walk at or after kb
    const int uhi = vw[7];
    while (kb < uhi && !sees(0, kb) && !sees(1, kb)) ++kb;
    return kb;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow<DROP>));
    if (warp == 0 && lane == 0 && T > 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      for (int x = 0; x < (hasB ? 2 : 1); ++x) {
        mbar_arrive_expect_tx(bar_qfull(x), C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(sQ + x * C::kTileBytes + c * C::kAtomBytes, &tmQ, c * 64, (qtA + x) * kBR, bh,
                      bar_qfull(x), pol_q);
      }
      int last_k[C::kKSt], last_v[C::kVSt];
      for (int s = 0; s < C::kKSt; ++s) last_k[s] = -1;
      for (int s = 0; s < C::kVSt; ++s) last_v[s] = -1;
      int kb = next_kb(ulo);
      for (int j = 0; j < T; ++j, kb = next_kb(kb + 1)) {
        const int ks = j % C::kKSt, vs = j % C::kVSt;
        if (j >= C::kKSt && !mbar_wait(bar_kempty(ks), ((j / C::kKSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_kfull(ks), C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(sK + ks * C::kTileBytes + c * C::kAtomBytes, &tmK, c * 64, kb * kBC, bh,
                      bar_kfull(ks), pol_kv);
        last_k[ks] = j;
        if (j >= C::kVSt && !mbar_wait(bar_vempty(vs), ((j / C::kVSt) & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(bar_vfull(vs), C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(sV + vs * C::kTileBytes + c * C::kAtomBytes, &tmV, c * 64, kb * kBC, bh,
                      bar_vfull(vs), pol_kv);
        last_v[vs] = j;
      }
      if (*abort_flag) {
        // Unwinding: let the copies already issued land before the CTA exits.
        // Load j is the (j / stages)-th use of its stage, so its completion is
        // the phase of that parity.
        mbar_wait_drain(bar_qfull(0), 0);
        if (hasB) mbar_wait_drain(bar_qfull(1), 0);
        for (int s = 0; s < C::kKSt; ++s)
          if (last_k[s] >= 0) mbar_wait_drain(bar_kfull(s), (last_k[s] / C::kKSt) & 1);
        for (int s = 0; s < C::kVSt; ++s)
          if (last_v[s] >= 0) mbar_wait_drain(bar_vfull(s), (last_v[s] / C::kVSt) & 1);
      }
    } else if (warp == 1 && lane == 0 && T > 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = idesc_bf16(kBR, kBC, false, false);
      constexpr uint32_t idO = idesc_bf16(kBR, HD, false, true);
      bool ok = true;
      // S_X(j) = Q_X K_j^T into S buffer X (columns 128 X).
      auto issue_s = [&](int x, int j) -> bool {
        const int ks = j % C::kKSt;
        if (j == 0 && !mbar_wait(bar_qfull(x), 0, ab)) return false;
        if (!mbar_wait(bar_kfull(ks), (j / C::kKSt) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t qbase = sQ + x * C::kTileBytes, kbase = sK + ks * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          // K-major operands: step k covers columns [16k, 16k+16) of d, i.e.
          // atom k/4, byte offset 32*(k%4) inside the 128-byte swizzled row.
          const uint32_t off = (k >> 2) * C::kAtomBytes + (k & 3) * 32;
          mma_ss(tmem + 128u * x, sdesc_sw128(qbase + off, 16, 1024),
                 sdesc_sw128(kbase + off, 16, 1024), idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull(x));
        // the last reader of K_j releases its stage
        if (x == 1 || j >= TB) mma_commit(bar_kempty(ks));
        return true;
      };
      // O_X (+)= P_X(j) V_j with P_X read from TMEM.
      auto issue_pv = [&](int x, int j) -> bool {
        const int vs = j % C::kVSt;
        if (!mbar_wait(bar_pfull(x), j & 1, ab)) return false;
        // the first reader of V_j waits for it
        if ((x == 0 || j >= TA) && !mbar_wait(bar_vfull(vs), (j / C::kVSt) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + vs * C::kTileBytes;
        const uint32_t ocol = C::kColO + static_cast<uint32_t>(HD) * x;
#pragma unroll
        for (int k = 0; k < kBC / 16; ++k) {
          // B = V_j, MN-major: 16 key rows per step (two 8-row groups, SBO
          // 1024 B); 64-column atoms of d are kAtomBytes apart (LBO).
          const uint64_t bdesc = sdesc_sw128(vbase + k * 2048, C::kAtomBytes, 1024);
          mma_ts(tmem + ocol, tmem + 128u * x + k * 8, bdesc, idO, (j > 0 || k > 0) ? 1u : 0u);
        }
        if (j == (x == 0 ? TA : TB) - 1) mma_commit(bar_ofinal(x));
        if (x == 1 || j >= TB) mma_commit(bar_vempty(vs));
        return true;
      };
      if (TA > 0) ok = issue_s(0, 0);
      if (ok && TB > 0) ok = issue_s(1, 0);
      for (int j = 0; ok && j < T; ++j) {
        // S_X(j+1) overwrites P_X(j): the product just before it reads P_X(j)
        // first (MMAs of one thread execute in issue order).
        if (j < TA) {
          ok = issue_pv(0, j);
          if (ok && j + 1 < TA) ok = issue_s(0, j + 1);
        }
        if (ok && j < TB) {
          ok = issue_pv(1, j);
          if (ok && j + 1 < TB) ok = issue_s(1, j + 1);
        }
      }
      // Drain: all MMAs issued above complete before TMEM is released.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh<DROP>));
    // ------------------------------------------------------------ softmax
    const int x = (warp >> 2) - 1;          // 0: block A (warps 4-7), 1: block B (warps 8-11)
    const int Tn = x == 0 ? TA : TB;        // TB = 0 when there is no block B
    const int quarter = warp & 3;           // TMEM lanes [32*quarter, +32)
    const int row = quarter * 32 + lane;    // row of the tile = TMEM lane
    const int q0 = (qtA + x) * kBR;
    const int grow = q0 + row;              // query index
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t scol = 128u * x;
    const uint32_t ocol = C::kColO + static_cast<uint32_t>(HD) * x;
    float m_run = -INFINITY;                // running max, log2 units (scaled)
    float l_run = 0.f;                      // row sum of P
    float lh_run = 0.f;                     // row sum of P rounded to bf16
    bool ok = true;
    int kb = next_kb(ulo);
    const uint32_t hh = static_cast<uint32_t>(bh % a.H), bb = static_cast<uint32_t>(b);
    for (int j = 0; j < Tn; ++j) {
      // Dropout keep bits of this row's 128 keys, drawn while S is computed;
      // the empty asm keeps the generator from being scheduled among the S
      // registers below (it would not fit in the register budget there).
      uint32_t kmask4[4] = {0u, 0u, 0u, 0u};
      if constexpr (DROP) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          kmask4[c] = keep32(static_cast<uint32_t>(kb * kBC + 32 * c), static_cast<uint32_t>(grow),
                             hh, bb, a.seed_lo, a.seed_hi, a.drop_thr);
        asm volatile("" : "+r"(kmask4[0]), "+r"(kmask4[1]), "+r"(kmask4[2]), "+r"(kmask4[3]));
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(x), j & 1, ab))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + scol + 32 * c, sr[c]);
      tmem_wait_ld();
      const int key0 = kb * kBC;
      const bool tile_on = sees(x, kb);  // false: a block of the walk X does not see
      const bool crossing = !tile_on || tile_crosses(q0, key0, a.N, kv_limit, a.causal, a.window);
      if (crossing) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = key0 + 32 * c + e;
            const bool keep = tile_on & visible(grow, key, kv_limit, a.causal, a.window);
            sr[c][e] = keep ? sr[c][e] : __float_as_uint(-INFINITY);  // select, no branch
          }
      }
      // Row max as a tree (independent partial maxima, no long dependency chain).
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
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // P = 2^(s * scale * log2e - m) with packed fp32 pairs (one FMA and one
      // add per two elements).  The row sum of P gives L.  O is divided by a
      // second sum, lh: in masked tiles it adds P rounded to bf16 -- the
      // weights the product actually applies to V -- and elsewhere P itself.
      // A row with fewer than 128 visible keys has no fully visible tile, so
      // for it lh is exactly the sum of the weights applied, which keeps its O
      // accurate; for longer rows the two sums differ by far less than the
      // bf16 rounding of O.
      const uint64_t scl2 = f2_pack(a.scale_log2, a.scale_log2);
      const uint64_t nm2 = f2_pack(-m_use, -m_use);
      // With dropout the product takes P * Z / q; L and the divisor of O stay
      // the sums of the undropped P.
      float sum_l, sum_h;
      auto p_tile = [&](auto mode) {
        constexpr bool kRounded = decltype(mode)::value == 1;
        constexpr bool kDrop = decltype(mode)::value == 2;
        uint64_t se[2] = {0ull, 0ull}, sh[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
          const uint32_t kmask = kmask4[c];  // dropout keep bits of the chunk's 32 keys
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])),
                             scl2, nm2),
                      t0, t1);
            const float p0 = ex2(t0), p1 = ex2(t1);
            if constexpr (kDrop) {
              const float d0 = (kmask >> (2 * e)) & 1u ? p0 * a.drop_scale : 0.f;
              const float d1 = (kmask >> (2 * e + 1)) & 1u ? p1 * a.drop_scale : 0.f;
              pk[e] = pack_bf16(d0, d1);
            } else {
              pk[e] = pack_bf16(p0, p1);
            }
            se[e & 1] = f2_add(se[e & 1], f2_pack(p0, p1));
            if constexpr (kRounded) sh[e & 1] = f2_add(sh[e & 1], bf16x2_to_f2(pk[e]));
          }
          // P occupies the first 64 columns of the S buffer (2 bf16 per column).
          tmem_st16(tl + scol + 16 * c, pk);
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
      else if (crossing)
        p_tile(std::integral_constant<int, 1>{});
      else
        p_tile(std::integral_constant<int, 0>{});
      l_run = l_run * alpha + sum_l;
      lh_run = lh_run * alpha + sum_h;
      m_run = m_new;
      if (j > 0 && __any_sync(0xffffffffu, grow_max)) {
        // O_X holds P_X(0..j-1) V; every product writing it has completed (see
        // the header), so it can be rescaled in place.
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + ocol + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tl + ocol + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull(x));
      kb = next_kb(kb + 1);
    }
    if (ok && Tn > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_ofinal(x), 0, ab));
      tc_fence_after();
    }
    // All four warps of this warpgroup take the same branch.
    ok = bar_and(1 + x, 128, ok && *abort_flag == 0);
    if (ok && (x == 0 || hasB)) {
      // ---------------------------------------------------------- epilogue
      const float inv_l = lh_run > 0.f ? 1.f / lh_run : 0.f;
      if (grow < a.N) {
        const float Lv = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        a.L[static_cast<long long>(bh) * a.N + grow] = Lv;
      }
      // O / l -> bf16 -> the (now idle) Q_X tile buffer, in the same swizzled
      // layout TMA uses, then one TMA store per 64-column atom.  Every lane
      // takes part in the warp-collective TMEM loads; TMA clips rows >= N.
      const int qoff = C::kOffQ + x * C::kTileBytes;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        if (Tn > 0) {
          tmem_ld32(tl + ocol + 32 * c, o);
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
          *reinterpret_cast<uint4*>(smem + qoff + atom * C::kAtomBytes + row * 128 + phys * 16) = v;
        }
      }
      fence_proxy_async_smem();
      bar_sync(1 + x, 128);
      if (quarter == 0 && lane == 0) {
        for (int c = 0; c < C::kAtoms; ++c)
          tma_store_3d(&tmO, sQ + x * C::kTileBytes + c * C::kAtomBytes, c * 64, q0, bh);
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

template <int HD, bool DROP>
cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         const CUtensorMap& tmO, const FwdArgs& a, cudaStream_t stream) {
  using C = Cfg<HD>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    // The register split (setmaxnreg) must fit in what the launch provides,
    // or the increasing warpgroups would wait for registers forever.
    cudaFuncAttributes fattr;
    e = cudaFuncGetAttributes(&fattr, fa_fwd_kernel<HD, DROP>);
    if (e != cudaSuccess) return e;
    if (fattr.numRegs * kThreads < 128 * kRegsLow<DROP> + 256 * kRegsHigh<DROP>)
      return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(fa_fwd_kernel<HD, DROP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = static_cast<long long>((a.n_qtiles + 1) / 2) * a.BH;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_fwd_kernel<HD, DROP><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV,
                                                                                    tmO, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdArgs& a,
                       cudaStream_t stream) {
  if (fwd_one_block(d, a.window, a.bmask, a.drop_thr))
    return launch_fwd_1q(d, tmQ, tmK, tmV, tmO, a, stream);
  switch (d) {
    case 64:
      return a.drop_thr ? launch_fwd_t<64, true>(tmQ, tmK, tmV, tmO, a, stream)
                        : launch_fwd_t<64, false>(tmQ, tmK, tmV, tmO, a, stream);
    case 128:
      return a.drop_thr ? launch_fwd_t<128, true>(tmQ, tmK, tmV, tmO, a, stream)
                        : launch_fwd_t<128, false>(tmQ, tmK, tmV, tmO, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
