/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library, libfa_gb300.so.
 *
 * What is computed (exact scaled-dot-product self-attention):
 *   For batch b and query head h, with key/value head g = h / (Hq / Hkv),
 *     S = scale * Q[b,h] K[b,g]^T,  P = softmax(S) per row,  O[b,h] = P V[b,g],
 *     LSE[b,h,i] = ln sum_j exp(S[i,j])   (natural log, scale included).
 *   Causal: query i sees key j iff j <= i.
 *   Pages: [QBank-36] "十九、分布式与系统方向的标准答案速查区", question #36
 *   ("FlashAttention 为什么常被说成是 IO-aware 优化"), parts 2-3 (S = QK^T,
 *   P = softmax(S), O = PV over B x H x L x d tensors; tiling with an online
 *   softmax, S and P never written to HBM); [Lecture] Stanford lecture
 *   summary, "推导 FlashAttention 的在线 softmax" (running max and
 *   numerator/denominator rescaled by exp(old - new); the backward pass
 *   recomputes from small saved statistics), "GPU 显存和注意力瓶颈" (causal
 *   self-attention) and "减少缓存表示并验证草稿" (Hq query heads sharing
 *   Hkv key/value groups: Hkv == Hq is multi-head, Hkv == 1 multi-query).
 *   The result is exact up to floating-point rounding: bf16 inputs, fp32
 *   accumulation, bf16 outputs (round to nearest even), fp32 LSE.
 *
 * Conventions shared by every entry point:
 *   - Tensors are DEVICE pointers to contiguous row-major arrays:
 *       q, o, dO, dq : bf16 [B, Hq,  N, d]     (d innermost)
 *       k, v, dk, dv : bf16 [B, Hkv, N, d]
 *       lse          : fp32 [B, Hq,  N]
 *   - Every pointer must be 16-byte aligned (FA_ERR_MISALIGNED otherwise).
 *   - d must be 64 or 128 (FA_ERR_UNSUPPORTED_HEADDIM otherwise);
 *     B, Hq, Hkv, N >= 1, Hq % Hkv == 0, B <= 65535, N <= 8388480
 *     (65535 tiles of 128 rows) and ceil(N/128)*Hq*B < 2^31
 *     (FA_ERR_BAD_SHAPE otherwise).
 *   - scale must be finite and > 0 (FA_ERR_BAD_ARGUMENT otherwise).
 *   - Outputs must not overlap any input or each other (FA_ERR_ALIASING).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued on it and the call returns without synchronising.  The library
 *     never allocates or frees memory; the caller owns every buffer.
 *   - Errors are returned as fa_status; nothing aborts or prints.  Argument
 *     checks happen before any CUDA call, so an invalid call enqueues nothing.
 *   - Requires a compute capability 10.3 (GB300) device current on the
 *     calling thread (FA_ERR_UNSUPPORTED_DEVICE otherwise).
 *   - Every device-side wait is bounded: if a kernel's internal wait runs out
 *     (it should not), the kernel stops, leaves its outputs incomplete and
 *     records FA_ERR_DEVICE_TIMEOUT, which fa_last_device_status() reports
 *     (see there for FA_ERR_DEVICE_DRAIN).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_NULL_PTR = 1,             /* a required pointer is NULL */
  FA_ERR_BAD_SHAPE = 2,            /* B, Hq, Hkv, N < 1, Hq % Hkv != 0, or too large */
  FA_ERR_UNSUPPORTED_HEADDIM = 3,  /* d not in {64, 128} */
  FA_ERR_MISALIGNED = 4,           /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE_TOO_SMALL = 5,  /* workspace_bytes < fa_bwd_workspace_bytes(...) */
  FA_ERR_UNSUPPORTED_DEVICE = 6,   /* current device is not sm_103 */
  FA_ERR_LAUNCH = 7,               /* a kernel launch or tensor-map encode failed */
  FA_ERR_DEVICE_TIMEOUT = 8,       /* a device-side bounded wait ran out */
  FA_ERR_CUDA = 9,                 /* another CUDA runtime error */
  FA_ERR_BAD_ARGUMENT = 10,        /* scale not finite / not > 0, causal not 0/1 */
  FA_ERR_ALIASING = 11,            /* an output overlaps an input or another output */
  FA_ERR_SCRATCH_LIMIT = 12,       /* fa_bwd_noalloc: problem needs more than FA_NOALLOC_SCRATCH_BYTES */
  FA_ERR_DEVICE_DRAIN = 13         /* after a device timeout a kernel exited with its own copies or MMAs
                                      possibly still in flight: the library refuses further launches on
                                      that device for the rest of the process */
} fa_status;

/*
 * Forward pass.  Writes o [B,Hq,N,d] bf16 and lse [B,Hq,N] fp32.
 * q, k, v are read only.  One kernel launch.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                 int d, int causal, float scale, void* stream);

/*
 * Generalised forward: fa_fwd with these extensions.
 *   - Nq query rows against Nk keys (q, o: [B,Hq,Nq,d]; k, v: [B,Hkv,Nk,d];
 *     lse: [B,Hq,Nq]).  The queries are the last Nq positions: query row i
 *     stands at key position p_i = i + Nk - Nq (the decode shape: a few new
 *     queries attending to a long key/value history).  Nq == Nk == N is fa_fwd.
 *   - causal = 1: key j is visible to query row i iff j <= p_i (needs Nq <= Nk).
 *   - window = w >= 1 (needs causal = 1): also j > p_i - w, a sliding local
 *     window, the visibility pattern the pages ("ZeRO 与 FlashAttention 各优化
 *     什么?", 注意力瓶颈与优化路线; "38.解释FlashAttention的显存优化原理", part 2)
 *     name as an alternative to full attention.  window = 0: no window.
 *   - num_splits = S >= 1: the key tiles are cut into S contiguous chunks that
 *     are computed independently (more parallel work for few query rows); each
 *     chunk's (O_s, LSE_s) goes to the workspace and a second kernel merges
 *     them: O = sum_s e^(LSE_s - m) O_s / sum_s e^(LSE_s - m), LSE = m + ln
 *     sum_s e^(LSE_s - m), m = max_s LSE_s -- the streaming-softmax rescale of
 *     "推导 FlashAttention 的在线 softmax" applied to whole chunks.  S = 1 needs
 *     no workspace (workspace may be NULL) and is one kernel launch.
 * When Hq > Hkv and Nq is small (Hq/Hkv * Nq <= 128, Nq < 128) the query
 * rows of all heads of a kv group share one 128-row tile, so each K/V tile is
 * read once per group.
 * Errors: FA_ERR_BAD_ARGUMENT for window < 0, window > 0 without causal,
 * causal with Nq > Nk, or num_splits outside [1, 4096];
 * FA_ERR_WORKSPACE_TOO_SMALL if S > 1 and workspace_bytes <
 * fa_fwd_ex_workspace_bytes(...); otherwise as fa_fwd.  Outputs must not
 * overlap inputs, each other or the workspace.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int causal, int window, int num_splits, float scale, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Workspace bytes fa_fwd_ex needs for num_splits splits: per-split O, fp32
 * [S, B*Hq*Nq, d], then per-split LSE, fp32 [S, B*Hq*Nq], each rounded up to
 * 256 bytes.  0 for num_splits == 1 or invalid shapes.
 */
size_t fa_fwd_ex_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits);

/*
 * A split count for fa_fwd_ex on the current device: the count (1..64) that
 * minimises the key tiles processed by the busiest SM, each work item
 * costing about two key tiles extra.  Returns 1 for problems that already
 * fill the GPU (or invalid shapes).
 */
int fa_fwd_ex_default_splits(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window);

/*
 * Bytes of device workspace fa_bwd needs: the fp32 dQ accumulator
 * [B,Hq,N,d], then LSE*log2(e) and the row term D = rowsum(dO * O), each
 * fp32 [B*Hq, ceil(N/128)*128]; every part rounded up to 256 bytes.
 * Returns 0 for invalid shapes.  O(N * d) per head: no N x N buffer.
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);

/*
 * Backward pass: given q, k, v, the forward's o and lse, and dO, writes
 * dq [B,Hq,N,d], dk and dv [B,Hkv,N,d] (bf16), the gradients of
 * sum(dO * O).  P is recomputed tile by tile from lse; no N x N buffer.
 * `workspace` (device, >= fa_bwd_workspace_bytes) is scratch owned by the
 * caller; its contents on entry do not matter.  Equivalent to
 * fa_bwd_preprocess + fa_bwd_dkdv + fa_bwd_dq_convert in that order.
 * dq is not bitwise reproducible run to run: the fp32 dQ accumulation order
 * across key tiles is not fixed.  dk and dv are (one owner per key tile).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd with two options.
 *   window = w >= 1 with causal = 1: P is recomputed with key j visible to
 *     query i iff i - w < j <= i (the sliding window of fa_fwd_ex), and only
 *     the (query tile, key tile) pairs inside that band are visited;
 *     window = 0 is plain causal / full attention.  o and lse must come from
 *     the forward with the same window.  Self-attention only (Nq == Nk == N).
 *   deterministic = 1: dQ is accumulated per 128-row query tile by a separate
 *     kernel that walks the key tiles in a fixed order, so dQ (like dK, dV,
 *     always) is bitwise reproducible from run to run; it costs the S and dP
 *     recomputation a second time (3 more MMAs per tile pair, against 1 dQ
 *     MMA and the fp32 reduction saved).  deterministic = 0 adds the key
 *     tiles' dQ partials into an fp32 accumulator in arrival order (faster,
 *     reproducible only up to rounding).  Same workspace either way.
 * FA_ERR_BAD_ARGUMENT for window < 0, window > 0 without causal, or
 * deterministic not 0/1; otherwise as fa_bwd.  fa_bwd is
 * fa_bwd_ex(..., window = 0, deterministic = 0, ...).
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                    int deterministic, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward step 1: D = rowsum(dO * O) and LSE * log2(e) into the workspace
 * (padded per head to a multiple of 128 rows); zero the dQ accumulator.
 */
fa_status fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int Hq, int Hkv, int N, int d,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward step 2: dk, dv (written) and the dQ accumulator (added into),
 * recomputing P from the LSE step 1 staged in the workspace.  Needs step 1.
 */
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B, int Hq,
                      int Hkv, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Backward step 3: dq = bf16(scale * dQ accumulator). Needs step 2. */
fa_status fa_bwd_dq_convert(void* dq, int B, int Hq, int Hkv, int N, int d, float scale, const void* workspace,
                            size_t workspace_bytes, void* stream);

/* Static text for a status code (never NULL). */
const char* fa_strerror(fa_status status);

/*
 * Synchronises `stream`, then returns and clears the first device-side error
 * any kernel of this library recorded on the current device (FA_OK if none),
 * or FA_ERR_CUDA if the synchronisation itself failed.  If `detail` is not
 * NULL it receives 3 ints: flattened block index, wait-site id, thread index.
 *
 * A kernel whose bounded wait ran out stops its other roles and, on its way
 * out, waits (bounded again) for the TMA copies and MMAs it had already
 * issued before it frees its tensor memory.  If one of those drain waits also
 * gives up, work of that block may still have been in flight when it exited;
 * the call then returns FA_ERR_DEVICE_DRAIN (detail: block, drain site, -1)
 * and from then on every entry point that would launch on this device
 * returns FA_ERR_DEVICE_DRAIN without enqueuing anything.
 */
fa_status fa_last_device_status(void* stream, int* detail);

/*
 * Self-test of the bounded-wait mechanism: launches one CTA that waits on a
 * barrier nothing will complete, with a limit of `timeout_ns` nanoseconds
 * (1e3 .. 1e10).  Afterwards fa_last_device_status() must report
 * FA_ERR_DEVICE_TIMEOUT and the device stays usable.  No fault is involved.
 */
fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/*
 * Self-test of the drain path: one CTA waits, the way a kernel does on its
 * way out for the copies and MMAs it issued, on a barrier nothing completes,
 * limited to `timeout_ns` (1e3 .. 1e10).  No copy or MMA is actually in
 * flight and no fault is involved.  Afterwards fa_last_device_status()
 * reports FA_ERR_DEVICE_DRAIN (site 98) and this process can launch nothing
 * more on the device through this library: run it in a process of its own.
 */
fa_status fa_selftest_drain_timeout(unsigned long long timeout_ns, void* stream);

/*
 * Backward pass for callers that must not allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot hand fa_bwd a workspace: code that runs under a memory manager
 * owning every byte of the device (a framework's caching pool, an inference
 * runtime with a fixed arena), hosts whose plugins are not allowed to call
 * cudaMalloc/cudaFree at run time, and hot paths where cudaMalloc is too
 * costly or would synchronise the device.
 *
 * Same arguments, layout and result as fa_bwd, without the workspace: the
 * scratch (fp32 dQ accumulator and row term, fa_bwd_workspace_bytes() bytes)
 * lives in a fixed FA_NOALLOC_SCRATCH_BYTES buffer compiled into this
 * library.  Every GPU that loads the library keeps that buffer until the
 * process exits.  The call allocates and frees nothing.
 *   - Problems whose fa_bwd_workspace_bytes() exceeds the buffer are rejected
 *     with FA_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   - The first call on a device looks the buffer's device address up once
 *     (with that device current); make that first call before any stream
 *     capture begins.
 *   - All calls on a device share the one buffer and each starts by clearing
 *     what must start at zero.  Calls whose kernels overlap on the GPU (other
 *     streams, or other threads) race on it: serialise them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                         int causal, float scale, void* stream);

/*
 * Text of the most recent CUDA runtime error behind an FA_ERR_LAUNCH or
 * FA_ERR_CUDA status returned on the calling thread ("no error" if none).
 * Static string, never NULL.
 */
const char* fa_last_cuda_error(void);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
