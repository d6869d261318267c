// Internal launcher interface between the C-ABI layer (fa_api.cu) and the
// kernels.  Nothing here is exported from the shared library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sm103a.cuh"

namespace fa {

struct FwdArgs {
  void* o;            // [B, Hq, Nq, d] bf16 (one split)
  float* lse;         // [B, Hq, Nq] fp32, natural log (one split)
  float* o_part;      // [splits, B*Hq*Nq, d] fp32 per-split O (several splits, workspace)
  float* lse_part;    // [splits, B*Hq*Nq] fp32 per-split LSE (several splits, workspace)
  int B, Hq, Hkv, Nq, Nk;
  int causal;         // key j visible to query row i iff j <= i + Nk - Nq
  int window;         // > 0: also j > i + Nk - Nq - window
  int packed;         // a query tile holds all Hq/Hkv heads of a kv group (Hq/Hkv * Nq <= 128)
  int nqt;            // query tiles per unit (1 when packed)
  int units;          // B*Hq, or B*Hkv when packed
  int splits;         // key range split into chunks of split_tiles 128-key tiles
  int split_tiles;
  float scale_log2;   // scale * log2(e)
};

struct BwdArgs {
  const float* lse2;  // [B*Hq, ntp] fp32, LSE * log2(e), padded per head to ntp = ceil(N/128)*128 (workspace)
  const float* drow;  // [B*Hq, ntp] fp32, rowsum(dO * O), same padding (workspace)
  float* dq_accum;    // [B, Hq, N, d] fp32 (workspace)
  void* dk;           // [B, Hkv, N, d] bf16
  void* dv;           // [B, Hkv, N, d] bf16
  int B, Hq, Hkv, N;
  int causal;
  int window;         // > 0: key j visible to query i only if j > i - window (with causal)
  int with_dq;        // 1: also add the dQ partials into dq_accum; 0: dK, dV only
  int v8;             // dK and dV 32-byte aligned: their rows are written 32 bytes at a time
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e)
};

struct DqArgs {
  const float* lse2;  // [B*Hq, ntp] fp32, LSE * log2(e), padded (workspace)
  const float* drow;  // [B*Hq, ntp] fp32, rowsum(dO * O), padded (workspace)
  void* dq;           // [B, Hq, N, d] bf16
  int B, Hq, Hkv, N;
  int causal, window;
  float scale;
  float scale_log2;
};

// Deterministic dQ: persistent CTAs walking query-tile items, fixed accumulation order.
cudaError_t launch_bwd_dq(int d, const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                          const TmaMap4& tdo, const DqArgs& a, const DevStatus& st, int num_sms,
                          cudaStream_t stream);

// `tq` views Q as {d, Hq*Nq, B}; `to` (O as a {d, N, Hq, B} bf16 map) is
// used by the plain self-attention instance only.
cudaError_t launch_fwd(int d, const TmaMap3& tq, const TmaMap4& tk, const TmaMap4& tv,
                       const TmaMap4& to, const FwdArgs& a, const DevStatus& st, int num_sms,
                       cudaStream_t stream);

// (O, LSE) of several key splits -> O (bf16), LSE.
cudaError_t launch_fwd_merge(int d, const FwdArgs& a, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dO, const float* lse, float* lse2, float* drow,
                                  float* dq_accum, long long heads, int N, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_dkdv(int d, const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                            const TmaMap4& tdo, const TmaMap3& tdq, const BwdArgs& a, const DevStatus& st,
                            int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_dq_convert(const float* dq_accum, void* dq, float scale, long long n, int num_sms,
                                  cudaStream_t stream);

// One-time set-up of the current device for each translation unit's kernels
// (shared-memory sizes; the forward also checks that every instance was
// compiled with the register count its warpgroup split assumes).
cudaError_t configure_fwd_kernels();
cudaError_t configure_bwd_kernels();
cudaError_t configure_dq_kernels();

inline cudaError_t configure_kernels() {
  cudaError_t e = configure_fwd_kernels();
  if (e == cudaSuccess) e = configure_bwd_kernels();
  if (e == cudaSuccess) e = configure_dq_kernels();
  return e;
}

}  // namespace fa
