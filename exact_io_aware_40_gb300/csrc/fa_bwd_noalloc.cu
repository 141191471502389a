// fa_bwd_noalloc.cu -- the backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd needs a caller-provided workspace (the fp32 row terms D of the
// softmax gradient).  Some callers cannot produce one: code that runs under a
// host framework that owns every device byte through its own pool and forbids
// allocating behind its back, and latency-critical paths where allocating or
// freeing device memory may synchronise the whole device.  fa_bwd_noalloc
// serves them from a fixed scratch array compiled into this library instead.
// It runs exactly the kernels of fa_bwd (prepare, dK/dV, dQ) for every head
// dimension fa_bwd takes, with the scratch array as the workspace; it calls no
// allocator.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "kernels.h"

namespace {

// The scratch array.  Every GPU on which this library is loaded holds these
// FA_BWD_NOALLOC_SCRATCH_BYTES bytes until the process exits.  In host code the
// name is only a host-side stand-in: kernels must receive the device address
// returned by cudaGetSymbolAddress, never &g_noalloc_scratch.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device.  It is looked up
// once per device (the first call on a device may load this library's device
// code there) and again only if the device's context has changed since, as
// after a device reset, when the cached address would be stale.
fa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  if (!fa::current_context_id(&ctx)) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* L, void* dQ, void* dK, void* dV,
                                    int B, int H, int N, int d, float scale, int causal,
                                    const int32_t* kv_len, fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;  // a head dimension fa_bwd does not take
  // Larger problems than the fixed scratch holds are refused, not truncated.
  if (need > static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES)) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  fa_status st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  // fa_bwd validates the remaining arguments (the head dimension among them);
  // its prepare stage overwrites the scratch before the other stages read it,
  // so no state of an earlier call leaks in.
  return fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, scratch, need,
                stream);
}
