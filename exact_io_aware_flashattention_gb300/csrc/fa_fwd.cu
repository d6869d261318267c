// Exact attention forward on sm_103a: O = softmax(scale * Q K^T) V and the
// per-row log-sum-exp, computed tile by tile without any N x N buffer.
//
// Method ([QBank-36] "FlashAttention 为什么常被说成是 IO-aware 优化", part 3;
// [Lecture] "推导 FlashAttention 的在线 softmax"): for one 128-row tile of
// queries, stream 128-key tiles of K and V; for each, form the score tile in
// tensor memory, update a running row max m and running denominator l,
// rescale the running output by exp(m_old - m_new) when the max grows, and
// accumulate P V.  O / l and LSE = m + ln l are written once at the end.
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0     TMA producer: Q tile once, then K_j / V_j into a 2-stage ring
//   warp 1     TMEM allocator and tcgen05.mma issuer (one elected thread)
//   warps 2-5  softmax warpgroup: thread t of the group owns query row t of
//              the tile (TMEM lane t), so row max / row sum are in-thread
// Tensor memory (512 columns): S double buffer at columns 0 and 128
// (fp32 128 x 128 each), O accumulator at column 256 (fp32 128 x d).
// P (bf16, 128 x 128) goes through a shared-memory tile as the A operand of
// the P V MMA.
#include "fa_internal.h"
#include "sm103a.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;       // query rows per tile
constexpr int kBN = 128;       // keys per tile
constexpr int kStages = 2;     // K/V ring depth
constexpr int kThreads = 192;
constexpr uint32_t kBlockBytes = 128u * 128u;   // one 64-column block of a 128-row bf16 tile

template <int D>
struct FwdSmem {
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTile;
  static constexpr uint32_t kV = kK + kStages * kTile;
  static constexpr uint32_t kP = kV + kStages * kTile;
  static constexpr uint32_t kBar = kP + 128u * 128u * 2u;
  static constexpr uint32_t kBytes = kBar + 256u;
  static constexpr uint32_t kAlloc = kBytes + 1024u;   // slack for 1024-byte alignment
};

// Wait-site ids reported in the status words.
enum : int { kSiteQ = 1, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSitePFull, kSiteVFull, kSiteSFull, kSiteODone };

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t k_empty[kStages];
  uint64_t v_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args, const DevStatus st) {
  using L = FwdSmem<D>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int N = args.N;
  const int nt = (N + kBM - 1) / kBM;
  const int qt = args.causal ? (nt - 1 - (int)blockIdx.z) : (int)blockIdx.z;
  const int kvh = h / (args.Hq / args.Hkv);
  const int n_kv = args.causal ? min(qt + 1, nt) : nt;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tS0 = tmem, tS1 = tmem + 128, tO = tmem + 256;

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sP = smem_u32(smem + L::kP);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int k_issued[kStages] = {0, 0}, v_issued[kStages] = {0, 0};
      mbar_arrive_expect_tx(&bars->q_full, L::kTile);
      for (int a = 0; a < kAtoms; ++a)
        tma_load_4d(smem + L::kQ + a * kBlockBytes, &tmQ, &bars->q_full, a * 64, qt * kBM, h, b);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages, r = j / kStages;
        if (r > 0 && !mbar_wait(&bars->k_empty[s], (r - 1) & 1, st, abort_flag, kSiteKEmpty)) break;
        mbar_arrive_expect_tx(&bars->k_full[s], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_4d(smem + L::kK + s * L::kTile + a * kBlockBytes, &tmK, &bars->k_full[s], a * 64, j * kBN,
                      kvh, b);
        ++k_issued[s];
        if (r > 0 && !mbar_wait(&bars->v_empty[s], (r - 1) & 1, st, abort_flag, kSiteVEmpty)) break;
        mbar_arrive_expect_tx(&bars->v_full[s], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_4d(smem + L::kV + s * L::kTile + a * kBlockBytes, &tmV, &bars->v_full[s], a * 64, j * kBN,
                      kvh, b);
        ++v_issued[s];
      }
      // Every copy issued must have landed before the CTA may exit.
      mbar_wait_drain(&bars->q_full, 0, st.timeout_ns);
      for (int s = 0; s < kStages; ++s) {
        if (k_issued[s]) mbar_wait_drain(&bars->k_full[s], (k_issued[s] - 1) & 1, st.timeout_ns);
        if (v_issued[s]) mbar_wait_drain(&bars->v_full[s], (v_issued[s] - 1) & 1, st.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
      bool ok = mbar_wait(&bars->q_full, 0, st, abort_flag, kSiteQ);
      auto issue_s = [&](int j) -> bool {
        const int s = j % kStages;
        if (!mbar_wait(&bars->k_full[s], (j / kStages) & 1, st, abort_flag, kSiteKFull)) return false;
        tc_fence_after();
        const uint32_t kt = sK + s * L::kTile;
        const uint32_t dS = (j & 1) ? tS1 : tS0;
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          mma_bf16_ss(dS, desc_kmajor(sQ, k16, kBlockBytes), desc_kmajor(kt, k16, kBlockBytes), idS, k16 > 0);
        mma_commit(&bars->s_full[j & 1]);
        mma_commit(&bars->k_empty[s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) break;
        if (!mbar_wait(&bars->p_full, j & 1, st, abort_flag, kSitePFull)) break;
        tc_fence_after();
        const int s = j % kStages;
        if (!mbar_wait(&bars->v_full[s], (j / kStages) & 1, st, abort_flag, kSiteVFull)) break;
        tc_fence_after();
        const uint32_t vt = sV + s * L::kTile;
#pragma unroll
        for (int k16 = 0; k16 < kBN / 16; ++k16)
          mma_bf16_ss(tO, desc_kmajor(sP, k16, kBlockBytes), desc_mnmajor(vt, k16, kBlockBytes), idO,
                      (j > 0 || k16 > 0) ? 1u : 0u);
        mma_commit(&bars->o_done);
        mma_commit(&bars->v_empty[s]);
      }
      // No MMA may still be writing tensor memory when it is freed.
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, st.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // row within the tile == TMEM lane
    const int row = qt * kBM + r;                // query index
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float sl2 = args.scale_log2;
    float m_run = -INFINITY;                     // running max of scale*log2(e)*s
    float l_run = 0.f;                           // running denominator
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait_warp(&bars->s_full[j & 1], (j >> 1) & 1, st, abort_flag, kSiteSFull)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = ((j & 1) ? tS1 : tS0) + lane_off;
      uint32_t sr[4][32];
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(sr[c]);

      const int key0 = j * kBN;
      const bool need_mask = (key0 + kBN > N) || (args.causal && j == qt);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = __uint_as_float(sr[c][e]);
          if (need_mask) {
            const int key = key0 + c * 32 + e;
            if (key >= N || (args.causal && key > row)) x = -INFINITY;
          }
          sr[c][e] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_run - m_use);
      uint32_t pk[64];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c][e]), sl2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c][e + 1]), sl2, -m_use));
          rs += p0 + p1;
          pk[(c * 32 + e) >> 1] = pack_bf16(p0, p1);
        }
      }
      l_run = l_run * alpha + rs;
      m_run = m_new;

      if (j > 0) {
        // P V of the previous tile must be done: it frees the P tile and the
        // O accumulator can be rescaled.
        if (!mbar_wait_warp(&bars->o_done, (j - 1) & 1, st, abort_flag, kSiteODone)) { ok = false; break; }
        tc_fence_after();
        __syncwarp();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row r -> shared memory, two 64-key column blocks, swizzled.
#pragma unroll
      for (int a = 0; a < 2; ++a) {
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const int base = a * 32 + c16 * 4;
          st_shared_v4(sP + a * kBlockBytes + swz128(r, c16), pk[base], pk[base + 1], pk[base + 2], pk[base + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    if (ok && mbar_wait_warp(&bars->o_done, (n_kv - 1) & 1, st, abort_flag, kSiteODone)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const size_t head = (size_t)b * args.Hq + h;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(args.o) + (head * N + (size_t)row) * D;
      __syncwarp();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_wait_ld();
        reg_fence(o);
        if (row < N) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[v * 8 + 0]) * inv_l, __uint_as_float(o[v * 8 + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(o[v * 8 + 2]) * inv_l, __uint_as_float(o[v * 8 + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(o[v * 8 + 4]) * inv_l, __uint_as_float(o[v * 8 + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(o[v * 8 + 6]) * inv_l, __uint_as_float(o[v * 8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + v * 8) = w;
          }
        }
      }
      if (row < N) args.lse[head * N + row] = (m_run + __log2f(l_run)) * 0.69314718055994530942f;
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

}  // namespace

template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdArgs& a, const DevStatus& st, cudaStream_t stream) {
  using L = FwdSmem<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int nt = (a.N + kBM - 1) / kBM;
  dim3 grid(a.Hq, a.B, nt);
  fa_fwd_kernel<D><<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, a, st);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& a,
                       const DevStatus& st, cudaStream_t stream) {
  if (d == 64) return launch_fwd_d<64>(tq, tk, tv, a, st, stream);
  return launch_fwd_d<128>(tq, tk, tv, a, st, stream);
}

}  // namespace fa
