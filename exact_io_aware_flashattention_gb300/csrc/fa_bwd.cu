// Exact attention backward on sm_103a, recomputing P tile by tile from the
// saved log-sum-exp instead of storing it ([FA-memory] "38.解释FlashAttention的
// 显存优化原理", part 2(2); [QBank-36] part 7; [Lecture] "推导 FlashAttention 的
// 在线 softmax", closing paragraphs).
//
// Three kernels on the caller's stream:
//   1. preprocess: D_i = sum_c dO[i,c] * O[i,c] (warp-shuffle reduction) and
//      zero the fp32 dQ accumulator.
//   2. dkdv: one CTA owns one 128-key tile of one kv head and loops over every
//      query head of its group and every 128-query tile that can see it.  dK
//      and dV accumulate in tensor memory and are written once: no atomics.
//      Per (query tile, key tile) it recomputes S^T = K Q^T, P^T = exp(S^T -
//      LSE), dP^T = V dO^T, dS^T = P^T * (dP^T - D), and issues
//      dV += P^T dO, dK += dS^T Q, dQ_partial = dS K; the dQ partial is added
//      into the fp32 accumulator (the separate dQ reduction).
//   3. dq_convert: dQ = bf16(scale * accumulator).
//
// dkdv CTA layout (192 threads):
//   warp 0     TMA producer (K, V once; Q_i, dO_i per item)
//   warp 1     TMEM allocator and MMA issuer
//   warps 2-5  compute warpgroup: thread t owns key row t of the tile for
//              S^T / dP^T / dK / dV, and query row t for the dQ partial.
// Tensor memory: S^T (then the dQ partial) at column 0, dP^T at 128,
// dV at 256, dK at 256 + d.
#include "fa_internal.h"
#include "sm103a.cuh"

namespace fa {

namespace {

constexpr int kT = 128;             // rows per query tile and per key tile
constexpr int kThreads = 192;
constexpr uint32_t kBlockBytes = 128u * 128u;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdSmem {
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;
  static constexpr uint32_t kDO = kQ + kTile;
  static constexpr uint32_t kP = kDO + kTile;
  static constexpr uint32_t kDS = kP + 128u * 128u * 2u;
  static constexpr uint32_t kLse = kDS + 128u * 128u * 2u;   // 2 x 128 fp32
  static constexpr uint32_t kDr = kLse + 1024u;               // 2 x 128 fp32
  static constexpr uint32_t kBar = kDr + 1024u;
  static constexpr uint32_t kBytes = kBar + 256u;
  static constexpr uint32_t kAlloc = kBytes + 1024u;
};

enum : int {
  kSiteKV = 11, kSiteQEmpty, kSiteQFull, kSiteDqEmpty, kSiteDoFull, kSitePFull, kSiteDsFull,
  kSiteSFull, kSiteDpFull, kSiteDqFull, kSiteDkvDone, kSiteWgSync
};

struct Bars {
  uint64_t kv_full, q_full, do_full, qdo_empty;
  uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_empty, dkv_done, drain, wg_sync;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdArgs args, const DevStatus st) {
  using L = BwdSmem<D>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kvh = blockIdx.x;
  const int b = blockIdx.y;
  const int j = blockIdx.z;                       // key tile (small j = most work, launched first)
  const int N = args.N;
  const int nt = (N + kT - 1) / kT;
  const int G = args.Hq / args.Hkv;
  const int i0 = args.causal ? j : 0;            // first query tile that sees key tile j
  const int nqi = nt - i0;
  const int n_items = G * nqi;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->qdo_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->ds_full, 128);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 128);
    mbar_init(&bars->dkv_done, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->wg_sync, 128);
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + D;

  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sDO = smem_u32(smem + L::kDO);
  const uint32_t sP = smem_u32(smem + L::kP);
  const uint32_t sDS = smem_u32(smem + L::kDS);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->kv_full, 2 * L::kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_4d(smem + L::kK + a * kBlockBytes, &tmK, &bars->kv_full, a * 64, j * kT, kvh, b);
        tma_load_4d(smem + L::kV + a * kBlockBytes, &tmV, &bars->kv_full, a * 64, j * kT, kvh, b);
      }
      int issued = 0;
      for (int t = 0; t < n_items; ++t) {
        const int h = kvh * G + t / nqi;
        const int i = i0 + t % nqi;
        if (t > 0 && !mbar_wait(&bars->qdo_empty, (t - 1) & 1, st, abort_flag, kSiteQEmpty)) break;
        mbar_arrive_expect_tx(&bars->q_full, L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_4d(smem + L::kQ + a * kBlockBytes, &tmQ, &bars->q_full, a * 64, i * kT, h, b);
        mbar_arrive_expect_tx(&bars->do_full, L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_4d(smem + L::kDO + a * kBlockBytes, &tmDO, &bars->do_full, a * 64, i * kT, h, b);
        ++issued;
      }
      mbar_wait_drain(&bars->kv_full, 0, st.timeout_ns);
      if (issued) {
        mbar_wait_drain(&bars->q_full, (issued - 1) & 1, st.timeout_ns);
        mbar_wait_drain(&bars->do_full, (issued - 1) & 1, st.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);   // S^T, dP^T
      constexpr uint32_t idKM = idesc_bf16(128, D, false, true);      // dV, dK
      constexpr uint32_t idMM = idesc_bf16(128, D, true, true);       // dQ
      bool ok = mbar_wait(&bars->kv_full, 0, st, abort_flag, kSiteKV);
      for (int t = 0; ok && t < n_items; ++t) {
        const uint32_t ph = t & 1;
        if (!mbar_wait(&bars->q_full, ph, st, abort_flag, kSiteQFull)) break;
        if (t > 0 && !mbar_wait(&bars->dq_empty, (t - 1) & 1, st, abort_flag, kSiteDqEmpty)) break;
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          mma_bf16_ss(tS, desc_kmajor(sK, k16, kBlockBytes), desc_kmajor(sQ, k16, kBlockBytes), idSS, k16 > 0);
        mma_commit(&bars->s_full);
        if (!mbar_wait(&bars->do_full, ph, st, abort_flag, kSiteDoFull)) break;
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          mma_bf16_ss(tDP, desc_kmajor(sV, k16, kBlockBytes), desc_kmajor(sDO, k16, kBlockBytes), idSS, k16 > 0);
        mma_commit(&bars->dp_full);
        if (!mbar_wait(&bars->p_full, ph, st, abort_flag, kSitePFull)) break;
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          mma_bf16_ss(tDV, desc_kmajor(sP, k16, kBlockBytes), desc_mnmajor(sDO, k16, kBlockBytes), idKM,
                      (t > 0 || k16 > 0) ? 1u : 0u);
        if (!mbar_wait(&bars->ds_full, ph, st, abort_flag, kSiteDsFull)) break;
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          mma_bf16_ss(tDK, desc_kmajor(sDS, k16, kBlockBytes), desc_mnmajor(sQ, k16, kBlockBytes), idKM,
                      (t > 0 || k16 > 0) ? 1u : 0u);
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          mma_bf16_ss(tS, desc_mnmajor(sDS, k16, kBlockBytes), desc_mnmajor(sK, k16, kBlockBytes), idMM,
                      k16 > 0 ? 1u : 0u);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->qdo_empty);
      }
      mma_commit(&bars->dkv_done);
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, st.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int key = j * kT + r;
    const float sl2 = args.scale_log2;
    float* sLse = reinterpret_cast<float*>(smem + L::kLse);
    float* sDr = reinterpret_cast<float*>(smem + L::kDr);
    const float* lse_g = reinterpret_cast<const float*>(args.lse);
    bool ok = true;
    for (int t = 0; t < n_items; ++t) {
      const uint32_t ph = t & 1;
      const int h = kvh * G + t / nqi;
      const int i = i0 + t % nqi;
      const size_t head = (size_t)b * args.Hq + h;
      const int qrow = i * kT + r;
      float* lse_t = sLse + (t & 1) * 128;
      float* dr_t = sDr + (t & 1) * 128;
      lse_t[r] = (qrow < N) ? lse_g[head * N + qrow] * kLog2e : INFINITY;
      dr_t[r] = (qrow < N) ? args.drow[head * N + qrow] : 0.f;
      // All 128 threads have staged this item's LSE / D (and are done with
      // the buffer's previous use two items ago).
      mbar_arrive(&bars->wg_sync);
      if (!mbar_wait_warp(&bars->wg_sync, ph, st, abort_flag, kSiteWgSync)) { ok = false; break; }

      if (!mbar_wait_warp(&bars->s_full, ph, st, abort_flag, kSiteSFull)) { ok = false; break; }
      tc_fence_after();
      uint32_t pr[4][32];
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, pr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(pr[c]);
      const bool key_valid = key < N;
      const bool diag = args.causal && (i == j);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = c * 32 + e;
          float p = ex2(fmaf(__uint_as_float(pr[c][e]), sl2, -lse_t[col]));
          if (!key_valid || (diag && key > i * kT + col)) p = 0.f;
          pr[c][e] = __float_as_uint(p);
        }
      }
      // P^T row -> shared memory (bf16, swizzled)
#pragma unroll
      for (int a = 0; a < 2; ++a) {
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const int col = a * 64 + c16 * 8;
          const uint32_t* x = &pr[col >> 5][col & 31];
          st_shared_v4(sP + a * kBlockBytes + swz128(r, c16),
                       pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                       pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                       pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                       pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);

      if (!mbar_wait_warp(&bars->dp_full, ph, st, abort_flag, kSiteDpFull)) { ok = false; break; }
      tc_fence_after();
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t dp[32];
        tmem_ld32(tDP + lane_off + c * 32, dp);
        tmem_wait_ld();
        reg_fence(dp);
        uint32_t ds[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c * 32 + e;
          const float d0 = __uint_as_float(pr[c][e]) * (__uint_as_float(dp[e]) - dr_t[col]);
          const float d1 = __uint_as_float(pr[c][e + 1]) * (__uint_as_float(dp[e + 1]) - dr_t[col + 1]);
          ds[e >> 1] = pack_bf16(d0, d1);
        }
        // 32 columns = 4 chunks of 16 bytes in column block c/2.
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c16 = (c & 1) * 4 + q4;
          st_shared_v4(sDS + (c >> 1) * kBlockBytes + swz128(r, c16), ds[q4 * 4], ds[q4 * 4 + 1],
                       ds[q4 * 4 + 2], ds[q4 * 4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);

      if (!mbar_wait_warp(&bars->dq_full, ph, st, abort_flag, kSiteDqFull)) { ok = false; break; }
      tc_fence_after();
      __syncwarp();
      float* dq_row = args.dq_accum + (head * N + (size_t)qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tS + lane_off + c * 32, v);
        tmem_wait_ld();
        reg_fence(v);
        if (qrow < N) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            atomicAdd(reinterpret_cast<float4*>(dq_row + c * 32 + e),
                      make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                  __uint_as_float(v[e + 3])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->dq_empty);
    }

    if (ok && mbar_wait_warp(&bars->dkv_done, 0, st, abort_flag, kSiteDkvDone)) {
      tc_fence_after();
      const size_t kvrow = ((size_t)b * args.Hkv + kvh) * N + (size_t)key;
      __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(args.dv) + kvrow * D;
      __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(args.dk) + kvrow * D;
      __syncwarp();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const uint32_t src = (pass == 0 ? tDV : tDK) + lane_off;
        __nv_bfloat16* dst = pass == 0 ? dv_row : dk_row;
        const float mul = pass == 0 ? 1.f : args.scale;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(src + c * 32, v);
          tmem_wait_ld();
          reg_fence(v);
          if (key < N) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(v[q * 8 + 0]) * mul, __uint_as_float(v[q * 8 + 1]) * mul);
              w.y = pack_bf16(__uint_as_float(v[q * 8 + 2]) * mul, __uint_as_float(v[q * 8 + 3]) * mul);
              w.z = pack_bf16(__uint_as_float(v[q * 8 + 4]) * mul, __uint_as_float(v[q * 8 + 5]) * mul);
              w.w = pack_bf16(__uint_as_float(v[q * 8 + 6]) * mul, __uint_as_float(v[q * 8 + 7]) * mul);
              *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = w;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D_i = rowsum(dO_i * O_i) with a shuffle reduction over the D/8 lanes that
// share a row; also zeroes the dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                                const uint4* __restrict__ dO,
                                                                float* __restrict__ drow, float4* __restrict__ dq_accum,
                                                                long long rows) {
  constexpr int kTpr = D / 8;  // threads per row, 16 bytes each
  const long long total = rows * kTpr;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x; i0 < total; i0 += stride) {
    const long long idx = i0 + threadIdx.x;
    float s = 0.f;
    if (idx < total) {
      const uint4 a = o[idx];
      const uint4 g = dO[idx];
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]);
        const float2 fg = __bfloat1622float2(g2[e]);
        s = fmaf(fa.x, fg.x, s);
        s = fmaf(fa.y, fg.y, s);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (idx < total && (idx % kTpr) == 0) drow[idx / kTpr] = s;
  }
  const long long n4 = rows * (D / 4);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    dq_accum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                                uint4* __restrict__ dq, float scale, long long n8) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = acc[2 * i];
    const float4 c = acc[2 * i + 1];
    uint4 w;
    w.x = pack_bf16(a.x * scale, a.y * scale);
    w.y = pack_bf16(a.z * scale, a.w * scale);
    w.z = pack_bf16(c.x * scale, c.y * scale);
    w.w = pack_bf16(c.z * scale, c.w * scale);
    dq[i] = w;
  }
}

}  // namespace

template <int D>
static cudaError_t launch_dkdv_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const BwdArgs& a, const DevStatus& st, cudaStream_t stream) {
  using L = BwdSmem<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e =
      cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int nt = (a.N + kT - 1) / kT;
  dim3 grid(a.Hkv, a.B, nt);
  fa_bwd_dkdv_kernel<D><<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, tdo, a, st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, const DevStatus& st, cudaStream_t stream) {
  if (d == 64) return launch_dkdv_d<64>(tq, tk, tv, tdo, a, st, stream);
  return launch_dkdv_d<128>(tq, tk, tv, tdo, a, st, stream);
}

static int grid_for(long long work_items, int num_sms) {
  long long blocks = (work_items + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dO, float* drow, float* dq_accum, long long rows,
                                  int num_sms, cudaStream_t stream) {
  const int grid = grid_for(rows * (d / 8), num_sms);
  if (d == 64)
    fa_bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                           static_cast<const uint4*>(dO), drow,
                                                           reinterpret_cast<float4*>(dq_accum), rows);
  else
    fa_bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                            static_cast<const uint4*>(dO), drow,
                                                            reinterpret_cast<float4*>(dq_accum), rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const float* dq_accum, void* dq, float scale, long long n, int num_sms,
                                  cudaStream_t stream) {
  const long long n8 = n / 8;
  fa_bwd_dq_convert_kernel<<<grid_for(n8, num_sms), 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_accum),
                                                                       static_cast<uint4*>(dq), scale, n8);
  return cudaGetLastError();
}

}  // namespace fa
