/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa_sm103.so).
 *
 * The operation is exact scaled-dot-product attention computed by the tiled,
 * IO-aware method ("FlashAttention: Fast and Memory-Efficient Exact Attention
 * with IO-Awareness", abstract): Q is cut into blocks of B_r rows and K, V into
 * blocks of B_c rows (study notes "FlashAttention学习笔记", section
 * "分块计算整体流程(Tiling)"); each block product S_ij = Q_i K_j^T is masked and
 * folded into a running softmax (apxml.com chapter "高效注意力算法实现
 * (FlashAttention)", section "在线Softmax"), so that the N x N matrices S and P
 * never reach device memory.  The result equals standard attention (same
 * chapter, "FlashAttention不改变注意力的数学定义"):
 *
 *     O = softmax(scale * Q K^T + mask) V,     L = rowwise logsumexp (natural log)
 *
 * The backward pass recomputes P from L instead of reading a stored N x N
 * matrix (fmread.com summary, section 三.2, "反向传播优化").
 *
 * Conventions shared by every entry point:
 *   - Q, K, V, O, dO, dQ, dK, dV: bf16, contiguous [B, H, N, d] (d fastest),
 *     DEVICE pointers, 16-byte aligned.  L and the workspace's statistics are
 *     fp32; L is [B, H, N].
 *   - d must be 64, 128 or 256; B, H, N >= 1; B*H*ceil(N/128) < 2^31 (element
 *     offsets are 64-bit, so tensors may exceed 2^31 elements).
 *   - scale multiplies Q K^T before the mask and the softmax (usually 1/sqrt(d));
 *     it must be finite and > 0.
 *   - causal != 0 masks key j for query i when j > i (square attention,
 *     diagonal kept).
 *   - kv_len (optional, DEVICE int32 [B]): keys j >= kv_len[b] are masked for
 *     every query of batch b; values are clamped to [0, N].  A query with no
 *     visible key gets O = 0, L = -inf and zero gradients.
 *   - Ownership: the caller owns every buffer.  The library allocates no device
 *     memory in these calls; its only device state is one 4-byte error word per
 *     device (a static device variable).
 *   - Asynchrony: every call only enqueues work on `stream` (NULL = the legacy
 *     default stream) and returns; nothing synchronises except
 *     fa_check_error().
 *   - Errors: invalid arguments return FA_ERR_INVALID_ARG (or
 *     FA_ERR_UNSUPPORTED for a head dim or size the kernels do not handle) and
 *     enqueue nothing.  A failed launch returns FA_ERR_CUDA.  A kernel that
 *     detects a stalled pipeline gives up after a time limit, records
 *     FA_ERR_TIMEOUT in the device error word and returns; fa_check_error()
 *     reports it.  No C++ exception crosses this interface.
 *   - Aliasing: outputs must not overlap inputs or each other.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4
} fa_status;

/*
 * Forward pass (study notes "FlashAttention学习笔记", "Forward运作流程":
 * S_ij = Q_i K_j^T, masked safe softmax, O_ij = P_ij V_j, with the running
 * statistics of the online softmax).
 *   Q, K, V  in : bf16 [B, H, N, d]
 *   O       out : bf16 [B, H, N, d], rounded to nearest even
 *   L       out : fp32 [B, H, N], L_i = ln sum_{j visible} exp(scale * q_i.k_j)
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                 int N, int d, float scale, int causal, fa_stream_t stream);

/* Same as fa_fwd with per-batch key padding; kv_len may be NULL (= all N). */
fa_status fa_fwd_kvlen(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                       int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                       fa_stream_t stream);

/*
 * Forward with two more mask terms, the pages' extensions of the method:
 *   window      : -1 = none.  w >= 0 keeps key j for query i only when
 *                 i - w <= j <= i (local causal band; the bxzpzcl.cn article
 *                 names sliding-window attention among the supported features,
 *                 section "高级功能配置").
 *   block_mask  : NULL = none, or a DEVICE uint8 array [nb, nb], nb =
 *                 ceil(N / FA_MASK_BLOCK), row-major over (query block, key
 *                 block) pairs of FA_MASK_BLOCK x FA_MASK_BLOCK positions,
 *                 shared by every batch and head; 0 leaves the pair out
 *                 (block-sparse attention: the paper's abstract; fmread.com
 *                 summary, section 六 item 3).  The caller owns it; it is read
 *                 while the enqueued work runs.
 * All mask terms intersect (causal, kv_len, window, block mask).  Pairs the
 * block mask leaves out are never computed: the kernels visit only the
 * blocks a query block (or key block) keeps.  A query that keeps no key gets
 * O = 0, L = -inf.
 * Errors: window < -1 gives FA_ERR_INVALID_ARG.  Otherwise as fa_fwd_kvlen.
 */
#define FA_MASK_BLOCK 128
fa_status fa_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                        int window, const uint8_t* block_mask, fa_stream_t stream);

/*
 * Forward with dropout on the attention weights (the study notes list dropout
 * among the steps fused into the kernel, section "Kernel融合"), plus every
 * mask term of fa_fwd_masked:
 *   dropout_p     : drop probability, 0 <= p < 1 (0 = no dropout).  Weight
 *                   P_ij is kept and scaled by 1/q, or replaced by 0; O uses
 *                   the dropped weights, L stays the logsumexp of the scores.
 *   dropout_seed  : 64-bit key of the generator.
 * Decisions: Philox4x32-10 (Salmon et al., SC'11) at counter (j / 8, i, h, b)
 * with key (seed low word, seed high word); its 128 bits are eight 16-bit
 * values, value j % 8 (low half of word (j % 8) / 2 first) deciding key j:
 * kept iff value >= thr = floor(p * 65536), so q = (65536 - thr) / 65536 and
 * the scale is exactly 1/q.  The same (seed, p) gives the same decisions in
 * fa_bwd_dropout, which must be called with them.
 * Errors: p outside [0, 1) gives FA_ERR_INVALID_ARG; otherwise as
 * fa_fwd_masked.
 */
fa_status fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                         int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                         int window, const uint8_t* block_mask, float dropout_p,
                         uint64_t dropout_seed, fa_stream_t stream);

/*
 * Forward with 8-bit floating-point inputs, the FP8 direction the pages name
 * for the method (bxzpzcl.cn article, section "量化技术深度融合").
 *   Q, K, V   in : e4m3 codes (1 byte: sign, 4 exponent bits with bias 7, 3
 *                  mantissa bits; no infinities, 0x7F/0xFF are NaN, largest
 *                  finite 448), contiguous [B, H, N, d], DEVICE, 16-byte aligned
 *   descale_q, descale_k, descale_v : per-tensor factors, finite and > 0; the
 *                  values are factor * code
 *   O        out : bf16 [B, H, N, d] = softmax(scale * (dq Q)(dk K)^T + mask) (dv V)
 *   L        out : fp32 [B, H, N], as fa_fwd
 *   workspace    : DEVICE, >= fa_fwd_fp8_workspace_bytes(B, H, N, d) bytes,
 *                  256-byte aligned; receives a transposed copy of V
 * The products run in e4m3 with fp32 accumulation; P enters the PV product
 * rounded to e4m3 and O is divided by the sum of those rounded weights.
 * d must be 128 (FA_ERR_UNSUPPORTED otherwise).  Masks: causal and kv_len.
 */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);
fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                     int H, int N, int d, float scale, float descale_q, float descale_k,
                     float descale_v, int causal, const int32_t* kv_len, void* workspace,
                     size_t workspace_bytes, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: the fp32 [B, H, N] row terms
 * D_i = sum_c dO_ic O_ic, rounded up to 256 bytes.  Returns 0 for invalid
 * sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass: recomputes P = exp(scale * Q K^T - L) tile by tile (never
 * storing it) and returns the gradients of sum(O * dO):
 *   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,
 *   dK = scale dS^T Q,  with D_i = sum_c dO_ic O_ic.
 *   Q, K, V, O, dO  in : bf16 [B, H, N, d]   (O and L from fa_fwd/fa_fwd_kvlen
 *   L               in : fp32 [B, H, N]       with the same scale/mask)
 *   dQ, dK, dV     out : bf16 [B, H, N, d]; all three are deterministic
 *                        (no atomics: the same inputs give the same bits)
 *   workspace          : device, >= fa_bwd_workspace_bytes(B,H,N,d) bytes,
 *                        256-byte aligned; contents on entry are ignored.
 * Gradients with respect to L are not part of this interface.
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* L, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                 float scale, int causal, const int32_t* kv_len, void* workspace,
                 size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd with the window and block-mask terms of fa_fwd_masked (same meaning,
 * same errors); O and L must come from fa_fwd_masked with the same masks.
 * Key blocks (and query blocks) the masks leave out are skipped.
 */
fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                        int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                        int window, const uint8_t* block_mask, void* workspace,
                        size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd_masked with dropout: gradients of sum(O * dO) for the O of
 * fa_fwd_dropout with the same masks, dropout_p and dropout_seed (the
 * decisions are regenerated, never stored).  dV = (P Z / q)^T dO and
 * dS = P o ((dO V^T) Z / q - D), D_i = sum_c dO_ic O_ic.
 */
fa_status fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                         int window, const uint8_t* block_mask, float dropout_p,
                         uint64_t dropout_seed, void* workspace, size_t workspace_bytes,
                         fa_stream_t stream);

/*
 * The three stages fa_bwd enqueues, for callers that want to schedule or time
 * them separately.  Arguments mean the same as in fa_bwd; each validates its
 * own arguments.  fa_bwd == fa_bwd_prepare; fa_bwd_dkdv; fa_bwd_dq.
 *   fa_bwd_prepare: D_i = sum_c dO_ic O_ic into the workspace (HBM-bound).
 *   fa_bwd_dkdv:    one pass per 128-key block over all query rows: dK, dV.
 *                   Needs a prepared workspace.
 *   fa_bwd_dq:      one pass per 128-row query block over all keys: dQ.
 *                   Needs a prepared workspace; independent of fa_bwd_dkdv.
 */
fa_status fa_bwd_prepare(const void* O, const void* dO, int B, int H, int N, int d,
                         void* workspace, size_t workspace_bytes, fa_stream_t stream);
fa_status fa_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO,
                      const float* L, void* dK, void* dV, int B, int H, int N, int d, float scale,
                      int causal, const int32_t* kv_len, const void* workspace,
                      size_t workspace_bytes, fa_stream_t stream);
fa_status fa_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, const float* L,
                    void* dQ, int B, int H, int N, int d, float scale, int causal,
                    const int32_t* kv_len, const void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/*
 * Capacity of the fixed scratch array behind fa_bwd_noalloc: 16 MiB.  Every
 * GPU on which the library is loaded holds this much device memory until the
 * process exits.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * fa_bwd without a workspace argument.  The paper and the pages have no
 * counterpart to this entry point: it exists for callers that cannot allocate
 * device memory -- code running under a host framework that owns every device
 * byte through its own pool, and latency-critical paths on which cudaMalloc or
 * cudaFree could synchronise the device.  It computes exactly what fa_bwd
 * computes (same kernels, same arguments minus the workspace, every head
 * dimension fa_bwd takes: 64, 128, 256) and allocates nothing: its workspace
 * is a file-scope device array of FA_BWD_NOALLOC_SCRATCH_BYTES bytes inside
 * this library.
 *   - Size limit: returns FA_ERR_UNSUPPORTED, and enqueues nothing, when
 *     fa_bwd_workspace_bytes(B, H, N, d) exceeds FA_BWD_NOALLOC_SCRATCH_BYTES,
 *     i.e. when B * H * N exceeds 4,194,304 rows (B=1, H=16, N=16384 fits;
 *     B=8, H=64, N=8200 does not), and for a head dimension other than 64,
 *     128 or 256.
 *   - First call on a device: looks up the array's device address there
 *     (cudaGetSymbolAddress, which may load the library's device code on that
 *     device).  Make that first call before any stream capture.  The address
 *     is cached per device and looked up again when the device's context has
 *     changed (after cudaDeviceReset, for example).
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents; each call overwrites what it reads before reading
 *     it.  Calls whose work overlaps on the GPU (different streams without
 *     ordering between them) race on the array and give wrong results --
 *     order them.
 */
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, float scale, int causal, const int32_t* kv_len,
                         fa_stream_t stream);

/*
 * Failure-detection self test: launches one CTA whose threads wait on a
 * pipeline barrier that is never signalled, through the same time-bounded
 * wait every kernel of this library uses.  The wait gives up after limit_ns
 * nanoseconds (0 < limit_ns <= 1e10) and records FA_ERR_TIMEOUT in the device
 * error word, so a following fa_check_error(stream) returns FA_ERR_TIMEOUT and
 * the context stays usable.  Enqueues only; returns FA_OK once launched.
 */
fa_status fa_selftest_stalled_wait(uint64_t limit_ns, fa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's error
 * word (FA_ERR_TIMEOUT if a kernel gave up), or FA_ERR_CUDA if the stream
 * itself reports an error.
 */
fa_status fa_check_error(fa_stream_t stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
