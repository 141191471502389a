// masks.cuh -- which 128 x 128 tiles of the attention matrix a CTA visits.
//
// The mask set of query i (the key positions it attends to) intersects up to
// four terms: key padding j < kv_len[b]; causal j <= i; a sliding window
// i - w <= j <= i (a local band, the bxzpzcl.cn article's "滑动窗口注意力"
// feature, section "高级功能配置"); and a block-sparse mask over pairs of
// 128-row query blocks and 128-key blocks (the paper's abstract; fmread.com
// summary, section 六 item 3).  The first three make the visible key blocks of
// a query block (and the visible query blocks of a key block) a contiguous
// range; the block mask then leaves some blocks of that range out.  Kernels
// visit only the blocks left, in increasing order, and mask elements only in
// tiles that cross a boundary.
#pragma once
#include <cstdint>

namespace fa {

constexpr int kMaskBlock = 128;  // block size of the block-sparse mask

// [lo, hi): key blocks that can hold a visible key for some row of query
// block qt, before the block mask.
__device__ __forceinline__ void key_block_range(int qt, int kv_limit, int causal, int window,
                                                int* lo, int* hi) {
  int h = (kv_limit + kMaskBlock - 1) / kMaskBlock;
  if (causal || window >= 0) h = min(h, qt + 1);
  int l = 0;
  if (window >= 0) l = max(0, qt * kMaskBlock - window) / kMaskBlock;
  *lo = l;
  *hi = max(h, l);
}

// [lo, hi): query blocks (of n_qblocks) that can see a key of key block kt,
// before the block mask.
__device__ __forceinline__ void query_block_range(int kt, int n_qblocks, int kv_limit, int causal,
                                                  int window, int* lo, int* hi) {
  const int k0 = kt * kMaskBlock;
  if (k0 >= kv_limit) {
    *lo = *hi = 0;
    return;
  }
  int l = (causal || window >= 0) ? kt : 0;
  int h = n_qblocks;
  if (window >= 0) {
    const long long last = static_cast<long long>(k0) + kMaskBlock - 1 + window;
    h = static_cast<int>(min(static_cast<long long>(h), last / kMaskBlock + 1));
  }
  *lo = l;
  *hi = max(h, l);
}

// Is block b on in a block-mask row or column (`m` points at its first entry,
// consecutive blocks `stride` bytes apart)?  A null mask keeps every block.
__device__ __forceinline__ bool block_on(const uint8_t* m, int stride, int b) {
  return m == nullptr || __ldg(m + static_cast<long long>(b) * stride) != 0;
}

// First block >= b in [b, hi) that the mask keeps (hi if none).
__device__ __forceinline__ int next_block(const uint8_t* m, int stride, int b, int hi) {
  if (m == nullptr) return b;
  while (b < hi && __ldg(m + static_cast<long long>(b) * stride) == 0) ++b;
  return b;
}

// Number of kept blocks in [lo, hi); called by a whole warp.
__device__ __forceinline__ int count_blocks(const uint8_t* m, int stride, int lo, int hi) {
  if (m == nullptr) return hi - lo;
  int n = 0;
  for (int b0 = lo; b0 < hi; b0 += 32) {
    const int b = b0 + static_cast<int>(threadIdx.x & 31);
    const bool on = b < hi && __ldg(m + static_cast<long long>(b) * stride) != 0;
    n += __popc(__ballot_sync(0xffffffffu, on));
  }
  return n;
}

// The (batch-head, tile rank) a CTA owns.  Ranks are taken in groups of
// `group` consecutive ranks, rank 0 first, and head-major inside a group;
// group >= n_tiles is plain head-major order.  Rank 0 is the tile with the
// most work under a causal mask: when one group of all heads about fills the
// GPU's resident CTAs, the longest tiles of every head start in the first
// waves instead of the last head's starting near the end of the grid, and
// the CTAs of one head in a group still walk K/V (or Q/dO) side by side.
__host__ __device__ __forceinline__ void cta_tile(int cta, int n_tiles, int BH, int group,
                                                  int* bh, int* rank) {
  int w_full = group < n_tiles ? group : n_tiles;
  if (w_full < 1) w_full = 1;
  const int g = cta / (w_full * BH);
  const int first = g * w_full;  // first rank of the group
  const int left = n_tiles - first;
  const int w = w_full < left ? w_full : left;  // ranks in this group
  const int r = cta - first * BH;
  *bh = r / w;
  *rank = first + r % w;
}

// Element mask inside a tile: is key `key` visible from query `row`?
__device__ __forceinline__ bool visible(int row, int key, int kv_limit, int causal, int window) {
  const bool band = (causal != 0) | (window >= 0);
  return (key < kv_limit) & !(band & (key > row)) & !((window >= 0) & (key < row - window));
}

// Does the tile (rows [q0, min(q0 + 128, N)), keys [k0, k0 + 128)) hold a
// key that some of its rows do not see?  Keys past kv_limit (N included)
// count as unseen.
__device__ __forceinline__ bool tile_crosses(int q0, int k0, int N, int kv_limit, int causal,
                                             int window) {
  const bool band = (causal != 0) | (window >= 0);
  const int q_last = min(q0 + kMaskBlock, N) - 1;
  return (k0 + kMaskBlock > kv_limit) | (band & (k0 + kMaskBlock - 1 > q0)) |
         ((window >= 0) & (k0 < q_last - window));
}

}  // namespace fa
