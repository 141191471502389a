// fa_api.cu -- the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, the per-device error word, and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {

bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static std::atomic<void*> fn_cur{nullptr}, fn_id{nullptr};
  void* fc = fn_cur.load(std::memory_order_acquire);
  void* fi = fn_id.load(std::memory_order_acquire);
  if (fc == nullptr || fi == nullptr) {
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fc, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || fc == nullptr)
      return false;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fi, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || fi == nullptr)
      return false;
    fn_cur.store(fc, std::memory_order_release);
    fn_id.store(fi, std::memory_order_release);
  }
  CUcontext ctx = nullptr;
  if (reinterpret_cast<GetCurrentFn>(fc)(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {
    // No context yet on this thread: cudaSetDevice makes the device's primary
    // context current (initialising it if needed).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
    if (reinterpret_cast<GetCurrentFn>(fc)(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  }
  return reinterpret_cast<GetIdFn>(fi)(ctx, id) == CUDA_SUCCESS;
}

int sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace fa

namespace {

// One error word per device, written by kernels that give up on a stalled
// pipeline; read and cleared by fa_check_error.
__device__ int g_fa_error_word;

constexpr int kMaxDevices = 64;

// Signature of the driver's cuTensorMapEncodeTiled (CUDA 12.0 ABI version).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};
EncodeTiledFn g_encode = nullptr;

fa_status current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Device address of this device's error word, cached per device and looked
// up again when the device's context has changed (after a device reset).
fa_status error_word(int dev, int** out) {
  unsigned long long ctx = 0;
  if (!fa::current_context_id(&ctx)) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr || g_err_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_error_word) != cudaSuccess) return FA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
    g_err_ctx[dev] = ctx;
  }
  *out = g_err_ptr[dev];
  return FA_OK;
}

fa_status encoder(EncodeTiledFn* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FA_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return FA_OK;
}

// Tensor map over a bf16 [BH, N, d] tensor, seen as 3-D (d, N, BH) with a
// (64, rows, 1) box and 128-byte swizzle: one box is one 64-column atom of a
// `rows`-row tile.  Rows past N of a head read as zero (and are not written),
// so tiles never spill into the next head.
fa_status map_bf16(EncodeTiledFn enc, CUtensorMap* m, const void* base, int d,
                   int N, int BH, int rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(N)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Tensor map over a one-byte [BH, rows, inner] tensor, seen as 3-D (inner,
// rows, BH) with a (128, box_rows, 1) box and 128-byte swizzle (one box row is
// one 128-byte atom).  Out-of-range elements read as zero.
fa_status map_u8(EncodeTiledFn enc, CUtensorMap* m, const void* base, int inner, int rows,
                 int BH, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(inner) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  if (tiles * BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A pipeline stage whose producer never arrives: every thread of one CTA waits
// on an mbarrier that nothing signals, through the same bounded wait the
// attention kernels use, and must give up after `limit_ns`.
__global__ void stalled_wait_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(fa::smem_u32(&bar), 1);
    flag = 0;
    fa::fence_mbar_init();
  }
  __syncthreads();
  const fa::Abort ab{err, &flag};
  fa::mbar_wait(fa::smem_u32(&bar), 0, ab, limit_ns);
  __syncthreads();
}

}  // namespace

extern "C" {

fa_status fa_selftest_stalled_wait(uint64_t limit_ns, fa_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  int dev;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  int* err;
  if ((st = error_word(dev, &err)) != FA_OK) return st;
  stalled_wait_kernel<<<1, 64, 0, stream>>>(err, limit_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

// window < -1 is invalid; the window and block-mask terms run at every head
// dimension.
fa_status check_mask(int window) {
  if (window < -1) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Dropout parameters of the kernels: the integer keep threshold
// floor(p * 65536) (0: no dropout) and the unbiased scale 65536 / (65536 - thr).
struct Drop {
  uint32_t thr = 0, seed_lo = 0, seed_hi = 0;
  float scale = 1.f;
};
fa_status make_drop(float p, uint64_t seed, Drop* out) {
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_INVALID_ARG;
  Drop z;
  const double t = std::floor(static_cast<double>(p) * 65536.0);
  z.thr = static_cast<uint32_t>(t > 65535.0 ? 65535.0 : t);
  z.seed_lo = static_cast<uint32_t>(seed & 0xffffffffu);
  z.seed_hi = static_cast<uint32_t>(seed >> 32);
  z.scale = static_cast<float>(65536.0 / (65536.0 - static_cast<double>(z.thr)));
  *out = z;
  return FA_OK;
}

fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                   int N, int d, float scale, int causal, const int32_t* kv_len, int window,
                   const uint8_t* block_mask, float dropout_p, uint64_t seed,
                   fa_stream_t stream) {
  if (!Q || !K || !V || !O || !L) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if ((st = check_mask(window)) != FA_OK) return st;
  Drop drop;
  if ((st = make_drop(dropout_p, seed, &drop)) != FA_OK) return st;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(L, 4) ||
      (kv_len && !aligned(kv_len, 4)))
    return FA_ERR_INVALID_ARG;
  int dev;
  if ((st = current_device(&dev)) != FA_OK) return st;
  int* err;
  if ((st = error_word(dev, &err)) != FA_OK) return st;
  EncodeTiledFn enc;
  if ((st = encoder(&enc)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, to;
  if ((st = map_bf16(enc, &tq, Q, d, N, BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tk, K, d, N, BH, fa::kFwdKvRows)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tv, V, d, N, BH, fa::kFwdKvRows)) != FA_OK) return st;
  if ((st = map_bf16(enc, &to, O, d, N, BH, 128)) != FA_OK) return st;
  fa::FwdArgs a;
  a.L = L;
  a.kv_len = kv_len;
  a.err = err;
  a.H = H;
  a.N = N;
  a.BH = BH;
  a.n_qtiles = (N + 127) / 128;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.window = window;
  a.bmask = block_mask;
  a.nb = (N + 127) / 128;
  a.drop_thr = drop.thr;
  a.seed_lo = drop.seed_lo;
  a.seed_hi = drop.seed_hi;
  a.drop_scale = drop.scale;
  a.out_scale = 1.f;
  a.tile_group = a.n_qtiles;  // the launcher picks the CTA order
  if (fa::launch_fwd(d, tq, tk, tv, to, a, stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd_kvlen(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                       int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                       fa_stream_t stream) {
  return fwd_impl(Q, K, V, O, L, B, H, N, d, scale, causal, kv_len, -1, nullptr, 0.f, 0, stream);
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                 int N, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_impl(Q, K, V, O, L, B, H, N, d, scale, causal, nullptr, -1, nullptr, 0.f, 0,
                  stream);
}

fa_status fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                        int window, const uint8_t* block_mask, fa_stream_t stream) {
  return fwd_impl(Q, K, V, O, L, B, H, N, d, scale, causal, kv_len, window, block_mask, 0.f, 0,
                  stream);
}

fa_status fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                         int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                         int window, const uint8_t* block_mask, float dropout_p,
                         uint64_t dropout_seed, fa_stream_t stream) {
  return fwd_impl(Q, K, V, O, L, B, H, N, d, scale, causal, kv_len, window, block_mask, dropout_p,
                  dropout_seed, stream);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d != 128) return 0;
  const size_t npad = (static_cast<size_t>(N) + 15) / 16 * 16;
  return round256(static_cast<size_t>(B) * H * d * npad);
}

fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                     int H, int N, int d, float scale, float descale_q, float descale_k,
                     float descale_v, int causal, const int32_t* kv_len, void* workspace,
                     size_t workspace_bytes, fa_stream_t stream) {
  if (!Q || !K || !V || !O || !L || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  for (float f : {descale_q, descale_k, descale_v})
    if (!std::isfinite(f) || !(f > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
      !aligned(L, 4) || (kv_len && !aligned(kv_len, 4)) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_fwd_fp8_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  const float prod = scale * descale_q * descale_k;
  if (!std::isfinite(prod) || !(prod > 0.f)) return FA_ERR_INVALID_ARG;
  int dev;
  if ((st = current_device(&dev)) != FA_OK) return st;
  int* err;
  if ((st = error_word(dev, &err)) != FA_OK) return st;
  EncodeTiledFn enc;
  if ((st = encoder(&enc)) != FA_OK) return st;
  const int BH = B * H;
  const int npad = (N + 15) / 16 * 16;
  CUtensorMap tq, tk, tvt, to;
  if ((st = map_u8(enc, &tq, Q, d, N, BH, 128)) != FA_OK) return st;
  if ((st = map_u8(enc, &tk, K, d, N, BH, 128)) != FA_OK) return st;
  if ((st = map_u8(enc, &tvt, workspace, npad, d, BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &to, O, d, N, BH, 128)) != FA_OK) return st;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.L = L;
  a.kv_len = kv_len;
  a.err = err;
  a.H = H;
  a.N = N;
  a.BH = BH;
  a.n_qtiles = (N + 127) / 128;
  a.scale_log2 = prod * kLog2e;
  a.causal = causal ? 1 : 0;
  a.window = -1;
  a.nb = a.n_qtiles;
  a.drop_scale = 1.f;
  a.out_scale = descale_v;
  a.tile_group = a.n_qtiles;  // the launcher picks the CTA order
  if (fa::launch_transpose_v8(V, workspace, BH, N, npad, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  if (fa::launch_fwd_fp8(tq, tk, tvt, to, a, stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  return round256(static_cast<size_t>(B) * H * N * sizeof(float));
}

static fa_status check_workspace(const void* ws, size_t bytes, int B, int H, int N, int d) {
  if (!ws || !aligned(ws, 256)) return FA_ERR_INVALID_ARG;
  if (bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status fa_bwd_prepare(const void* O, const void* dO, int B, int H, int N, int d,
                         void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!O || !dO) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d, 1.f);
  if (st != FA_OK) return st;
  if (!aligned(O, 16) || !aligned(dO, 16)) return FA_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FA_OK) return st;
  fa::BwdPreArgs pre;
  pre.O = static_cast<const uint16_t*>(O);
  pre.dO = static_cast<const uint16_t*>(dO);
  pre.D = static_cast<float*>(workspace);
  pre.rows = static_cast<long long>(B) * H * N;
  pre.d = d;
  return fa::launch_bwd_pre(pre, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Shared validation and argument block of the two recompute kernels.
static fa_status bwd_args(const void* Q, const void* K, const void* V, const void* dO,
                          const float* L, int B, int H, int N, int d, float scale, int causal,
                          const int32_t* kv_len, int window, const uint8_t* block_mask,
                          float dropout_p, uint64_t seed, const void* workspace,
                          size_t workspace_bytes, fa::BwdArgs* a, EncodeTiledFn* enc) {
  if (!Q || !K || !V || !dO || !L) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if ((st = check_mask(window)) != FA_OK) return st;
  Drop drop;
  if ((st = make_drop(dropout_p, seed, &drop)) != FA_OK) return st;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(dO, 16) ||
      !aligned(L, 4) || (kv_len && !aligned(kv_len, 4)))
    return FA_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FA_OK) return st;
  int dev;
  if ((st = current_device(&dev)) != FA_OK) return st;
  int* err;
  if ((st = error_word(dev, &err)) != FA_OK) return st;
  if ((st = encoder(enc)) != FA_OK) return st;
  a->L = L;
  a->D = static_cast<const float*>(workspace);
  a->dK = nullptr;
  a->dV = nullptr;
  a->kv_len = kv_len;
  a->err = err;
  a->H = H;
  a->N = N;
  a->BH = B * H;
  a->n_ktiles = (N + 127) / 128;
  a->n_qtiles = 0;
  a->scale = scale;
  a->scale_log2 = scale * kLog2e;
  a->causal = causal ? 1 : 0;
  a->window = window;
  a->bmask = block_mask;
  a->nb = (N + 127) / 128;
  a->drop_thr = drop.thr;
  a->seed_lo = drop.seed_lo;
  a->seed_hi = drop.seed_hi;
  a->drop_scale = drop.scale;
  a->tile_group = a->n_ktiles;  // the launchers pick the CTA order
  return FA_OK;
}

static fa_status dkdv_impl(const void* Q, const void* K, const void* V, const void* dO,
                           const float* L, void* dK, void* dV, int B, int H, int N, int d,
                           float scale, int causal, const int32_t* kv_len, int window,
                           const uint8_t* block_mask, float dropout_p, uint64_t seed,
                           const void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!dK || !dV || !aligned(dK, 16) || !aligned(dV, 16)) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a;
  EncodeTiledFn enc;
  fa_status st = bwd_args(Q, K, V, dO, L, B, H, N, d, scale, causal, kv_len, window, block_mask,
                          dropout_p, seed, workspace, workspace_bytes, &a, &enc);
  if (st != FA_OK) return st;
  a.dK = static_cast<uint16_t*>(dK);
  a.dV = static_cast<uint16_t*>(dV);
  const int qrows = fa::bwd_dkdv_qrows(d);
  a.n_qtiles = (N + qrows - 1) / qrows;
  CUtensorMap tq, tk, tv, tdo;
  if ((st = map_bf16(enc, &tq, Q, d, N, a.BH, qrows)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tk, K, d, N, a.BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tv, V, d, N, a.BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tdo, dO, d, N, a.BH, qrows)) != FA_OK) return st;
  return fa::launch_bwd_dkdv(d, tq, tk, tv, tdo, a, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static fa_status dq_impl(const void* Q, const void* K, const void* V, const void* dO,
                         const float* L, void* dQ, int B, int H, int N, int d, float scale,
                         int causal, const int32_t* kv_len, int window,
                         const uint8_t* block_mask, float dropout_p, uint64_t seed,
                         const void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!dQ || !aligned(dQ, 16)) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a;
  EncodeTiledFn enc;
  fa_status st = bwd_args(Q, K, V, dO, L, B, H, N, d, scale, causal, kv_len, window, block_mask,
                          dropout_p, seed, workspace, workspace_bytes, &a, &enc);
  if (st != FA_OK) return st;
  a.n_qtiles = (N + 127) / 128;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if ((st = map_bf16(enc, &tq, Q, d, N, a.BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tk, K, d, N, a.BH, fa::bwd_dq_krows(d))) != FA_OK) return st;
  if ((st = map_bf16(enc, &tv, V, d, N, a.BH, fa::bwd_dq_krows(d))) != FA_OK) return st;
  if ((st = map_bf16(enc, &tdo, dO, d, N, a.BH, 128)) != FA_OK) return st;
  if ((st = map_bf16(enc, &tdq, dQ, d, N, a.BH, 128)) != FA_OK) return st;
  return fa::launch_bwd_dq(d, tq, tk, tv, tdo, tdq, a, stream) == cudaSuccess ? FA_OK
                                                                              : FA_ERR_CUDA;
}

static fa_status bwd_impl(const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                          int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                          int window, const uint8_t* block_mask, float dropout_p, uint64_t seed,
                          void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!Q || !K || !V || !O || !dO || !L || !dQ || !dK || !dV || !workspace)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if ((st = check_mask(window)) != FA_OK) return st;
  Drop drop;
  if ((st = make_drop(dropout_p, seed, &drop)) != FA_OK) return st;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
      !aligned(dO, 16) || !aligned(dQ, 16) || !aligned(dK, 16) || !aligned(dV, 16) ||
      !aligned(L, 4) || (kv_len && !aligned(kv_len, 4)))
    return FA_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FA_OK) return st;
  if ((st = fa_bwd_prepare(O, dO, B, H, N, d, workspace, workspace_bytes, stream)) != FA_OK)
    return st;
  if ((st = dkdv_impl(Q, K, V, dO, L, dK, dV, B, H, N, d, scale, causal, kv_len, window,
                      block_mask, dropout_p, seed, workspace, workspace_bytes, stream)) != FA_OK)
    return st;
  return dq_impl(Q, K, V, dO, L, dQ, B, H, N, d, scale, causal, kv_len, window, block_mask,
                 dropout_p, seed, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO,
                      const float* L, void* dK, void* dV, int B, int H, int N, int d, float scale,
                      int causal, const int32_t* kv_len, const void* workspace,
                      size_t workspace_bytes, fa_stream_t stream) {
  return dkdv_impl(Q, K, V, dO, L, dK, dV, B, H, N, d, scale, causal, kv_len, -1, nullptr, 0.f, 0,
                   workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, const float* L,
                    void* dQ, int B, int H, int N, int d, float scale, int causal,
                    const int32_t* kv_len, const void* workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
  return dq_impl(Q, K, V, dO, L, dQ, B, H, N, d, scale, causal, kv_len, -1, nullptr, 0.f, 0,
                 workspace, workspace_bytes, stream);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                 float scale, int causal, const int32_t* kv_len, void* workspace,
                 size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, -1, nullptr,
                  0.f, 0, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                        int window, const uint8_t* block_mask, void* workspace,
                        size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, window,
                  block_mask, 0.f, 0, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                         int window, const uint8_t* block_mask, float dropout_p,
                         uint64_t dropout_seed, void* workspace, size_t workspace_bytes,
                         fa_stream_t stream) {
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, scale, causal, kv_len, window,
                  block_mask, dropout_p, dropout_seed, workspace, workspace_bytes, stream);
}

fa_status fa_check_error(fa_stream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int dev;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  int* err;
  if ((st = error_word(dev, &err)) != FA_OK) return st;
  int host = 0;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
    return host == FA_ERR_TIMEOUT ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // extern "C"
