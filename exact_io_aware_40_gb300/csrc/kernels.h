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
};

// Forward: grid = n_qtiles * BH CTAs.
cudaError_t launch_fwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdArgs& a,
                       cudaStream_t stream);

struct BwdPreArgs {
  const uint16_t* O;    // bf16 [BH, N, d]
  const uint16_t* dO;   // bf16 [BH, N, d]
  float* D;             // fp32 [BH, N]: rowsum(dO * O)
  float* dq_acc;        // fp32 [BH, N, d], zeroed here
  long long rows;       // BH * N
  int d;
};
cudaError_t launch_bwd_pre(const BwdPreArgs& a, cudaStream_t stream);

struct BwdArgs {
  const float* L;       // fp32 [BH, N] (natural-log logsumexp)
  const float* D;       // fp32 [BH, N]
  float* dq_acc;        // fp32 [BH, N, d]
  uint16_t* dK;         // bf16 [BH, N, d]
  uint16_t* dV;         // bf16 [BH, N, d]
  const int* kv_len;
  int* err;
  int H, N, BH;
  int n_ktiles, n_qtiles;
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  int causal;
};
// Rows per query tile of the backward kernel's TMA boxes for Q and dO.
inline int bwd_query_rows(int d) { return d == 128 ? 64 : 128; }

// tmdQ: fp32 view of the dQ accumulator (box: d columns x 64 rows), used by
// the d = 128 kernel's bulk reductions.
cudaError_t launch_bwd(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                       const BwdArgs& a, cudaStream_t stream);

struct BwdPostArgs {
  const float* dq_acc;  // fp32 [BH, N, d]
  uint16_t* dQ;         // bf16
  long long n;          // elements
  float scale;
};
cudaError_t launch_bwd_post(const BwdPostArgs& a, cudaStream_t stream);

}  // namespace fa
