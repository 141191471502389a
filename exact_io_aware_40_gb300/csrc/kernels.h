// kernels.h -- internal interface between the C-ABI layer (fa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

struct FwdArgs {
  float* L;             // fp32 [B*H, N]
  const int* kv_len;    // device int32 [B] or nullptr
  int* err;             // device error word
  int H, N, BH;
  int n_qtiles;         // ceil(N / 128)
  float scale_log2;     // scale * log2(e)
  int causal;
  int window;           // < 0: none; w >= 0: keys i - w <= j <= i only
  const uint8_t* bmask; // block mask [nb, nb] (query block, key block) or nullptr
  int nb;               // ceil(N / 128)
  uint32_t drop_thr;    // dropout: 0 = none, else floor(p * 65536)
  uint32_t seed_lo, seed_hi;
  float drop_scale;     // 65536 / (65536 - drop_thr)
  float out_scale;      // factor applied to O (e4m3 forward: V's dequantisation factor)
  int tile_group;       // CTA order (cta_tile in masks.cuh); set by the launcher
};

// Multiprocessors of the current device (cached per device; 0 on error).
int sm_count();

// Unique id of the calling thread's current CUDA context (the driver never
// reuses one within a process, so a device reset shows up as a new id).
// Device addresses of this library's __device__ variables are cached under
// it.  Returns false on a driver error.
bool current_context_id(unsigned long long* id);

// Group width for cta_tile.  Only a causal mask without a window gives the
// CTAs of a launch very different amounts of work (the longest tile has
// n_tiles times the shortest's; a window makes them about equal); then one
// group of all BH heads should about fill the resident CTAs (ctas_per_sm x
// SMs).  Otherwise plain head-major order.  With a width of 1 the CTAs of a
// head in flight share no reads, so that order pays only while the operands
// every CTA of a head streams (head_bytes per head) stay in L2 for all
// heads: a 2048-token, 128-head d = 128 backward (128 MB of Q and dO) ran
// 8 % slower tile-major; 96 heads of 1024 x 64 (25 MB) gained.
inline int tile_group(bool causal, int n_tiles, int BH, int ctas_per_sm, long long head_bytes) {
  if (!causal || BH <= 0) return n_tiles;
  const int g = ctas_per_sm * sm_count() / BH;
  if (g >= 2) return g > n_tiles ? n_tiles : g;
  return static_cast<long long>(BH) * head_bytes <= (32ll << 20) ? 1 : n_tiles;
}

// Forward (fa_fwd.cu): one 128-row query block per CTA and 64-key blocks
// (the K and V maps use kFwdKvRows-row boxes), two CTAs per SM at d = 64 and
// 128, one at d = 256; causal, key padding, window, block mask and dropout.
// grid = ceil(N/128) * BH.
constexpr int kFwdKvRows = 64;
cudaError_t launch_fwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdArgs& a,
                       cudaStream_t stream);

// e4m3 forward, d = 128 (fa_fwd_fp8.cu): V [BH, N, 128] -> V^T [BH, 128,
// Npad] (Npad = N rounded up to 16, zero-filled), then the forward with Q, K
// maps over uint8 [BH, N, 128] (128 x 128 boxes), the V^T map over uint8
// [BH, 128, Npad] (128 x 128 boxes) and the bf16 O map of fa_fwd.
cudaError_t launch_transpose_v8(const void* V, void* Vt, int BH, int N, int Npad,
                                cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVt,
                           const CUtensorMap& tmO, const FwdArgs& a, cudaStream_t stream);

struct BwdPreArgs {
  const uint16_t* O;    // bf16 [BH, N, d]
  const uint16_t* dO;   // bf16 [BH, N, d]
  float* D;             // fp32 [BH, N]: rowsum(dO * O)
  long long rows;       // BH * N
  int d;
};
cudaError_t launch_bwd_pre(const BwdPreArgs& a, cudaStream_t stream);

struct BwdArgs {
  const float* L;       // fp32 [BH, N] (natural-log logsumexp)
  const float* D;       // fp32 [BH, N]
  uint16_t* dK;         // bf16 [BH, N, d]
  uint16_t* dV;         // bf16 [BH, N, d]
  const int* kv_len;
  int* err;
  int H, N, BH;
  int n_ktiles;         // ceil(N / 128): key blocks of the dK/dV kernel
  int n_qtiles;         // query steps: ceil(N / bwd_dkdv_qrows(d)) for dK/dV, ceil(N / 128) for dQ
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  int causal;
  int window;           // < 0: none; w >= 0: keys i - w <= j <= i only
  const uint8_t* bmask; // block mask [nb, nb] (query block, key block) or nullptr
  int nb;               // ceil(N / 128)
  uint32_t drop_thr;    // dropout: 0 = none, else floor(p * 65536)
  uint32_t seed_lo, seed_hi;
  float drop_scale;     // 65536 / (65536 - drop_thr)
  int tile_group;       // CTA order (cta_tile in masks.cuh); set by the launcher
};

// Query rows per step of the dK/dV kernel (the box height of its Q and dO
// maps) and keys per step of the dQ kernel (the box height of its K and V maps).
inline int bwd_dkdv_qrows(int d) { return d == 256 ? 32 : 128; }
inline int bwd_dq_krows(int d) { return d == 256 ? 32 : 128; }

// dK, dV: grid = ceil(N/128) * BH * (d == 256 ? 2 : 1) (d = 256: one CTA per
// 128-column half of dK, dV).  Q and dO maps use bwd_dkdv_qrows(d)-row boxes,
// K and V 128-row boxes.
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const BwdArgs& a,
                            cudaStream_t stream);
// d = 64, 128: the 128-wide variants (fa_bwd_wide.cu), same arguments.
cudaError_t launch_bwd_dkdv_wide(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                 const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq_wide(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                               const CUtensorMap& tmV, const CUtensorMap& tmdO,
                               const CUtensorMap& tmdQ, const BwdArgs& a, cudaStream_t stream);
// dQ: grid = ceil(N/128) * BH.  Q, dO and dQ maps
// use 128-row boxes, K and V bwd_dq_krows(d)-row boxes.
cudaError_t launch_bwd_dq(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                          const BwdArgs& a, cudaStream_t stream);

}  // namespace fa
