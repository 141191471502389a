// fa_bwd_prep.cu -- the HBM-bound pass before the backward kernels:
// D_i = sum_c dO_ic * O_ic (fp32) for every row.  D_i equals sum_j P_ij dP_ij,
// the row term of the softmax gradient dS = P o (dP - D), because
// O_i = sum_j P_ij V_j.
#include "kernels.h"

namespace fa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Each thread owns 8 consecutive elements (16 bytes) of one row; the d/8
// threads of a row reduce with shuffles (d/8 divides 32).
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdPreArgs a) {
  const int tpr = a.d / 8;  // threads per row: 8 (d=64) or 16 (d=128)
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gtid / tpr;
  const int part = static_cast<int>(gtid % tpr);
  float acc = 0.f;
  if (row < a.rows) {
    const long long off = row * a.d + part * 8;
    const uint4 o = *reinterpret_cast<const uint4*>(a.O + off);
    const uint4 g = *reinterpret_cast<const uint4*>(a.dO + off);
    acc = bf16_lo(o.x) * bf16_lo(g.x) + bf16_hi(o.x) * bf16_hi(g.x) + bf16_lo(o.y) * bf16_lo(g.y) +
          bf16_hi(o.y) * bf16_hi(g.y) + bf16_lo(o.z) * bf16_lo(g.z) + bf16_hi(o.z) * bf16_hi(g.z) +
          bf16_lo(o.w) * bf16_lo(g.w) + bf16_hi(o.w) * bf16_hi(g.w);
  }
  for (int w = tpr / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (row < a.rows && part == 0) a.D[row] = acc;
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreArgs& a, cudaStream_t stream) {
  if (a.d % 8 != 0 || 32 % (a.d / 8) != 0) return cudaErrorInvalidValue;
  const long long threads = a.rows * (a.d / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  bwd_pre_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
