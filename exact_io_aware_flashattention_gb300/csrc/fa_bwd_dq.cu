// Deterministic dQ for the attention backward: persistent, one CTA per SM.
// An item is one 128-row query tile of one (head, batch); the CTA walks the
// key tiles the item can see and accumulates dQ = scale * sum_j dS_j K_j in
// tensor memory, in a fixed order, so dQ is bitwise reproducible (the dK/dV
// kernel then runs without its dQ partials).
// It recomputes what the dK/dV kernel recomputes, from the saved LSE
// ([FA-memory] "38.解释FlashAttention的显存优化原理", part 2(2); [QBank-36]
// part 7), with queries instead of keys on the tensor-memory lanes:
//   S = Q K_j^T, P = 2^(S * scale * log2 e - LSE * log2 e),
//   dP = dO V_j^T, dS = P (dP - D), dQ += dS K_j.
//
// Items go heaviest first (the last query tile first under causal masking)
// and are dealt to the CTAs in snake order.  The K / V rings, the two S
// buffers and their barriers run on across items (a tile counter); the next
// item's Q / dO are loaded as soon as the item's last dP MMA has completed,
// while its last dS, dQ MMA and epilogue finish, and the next item's first dQ
// MMA waits until the epilogue has read dQ out of tensor memory.
//
// CTA layout (320 threads):
//   warp 0      TMA producer: per item Q, dO and the item's 128 LSE / D
//               values, K and V per key tile (rings of kStages)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-9   two compute warpgroups: thread t of a group owns query row t
//               (TMEM lane t); group g handles key columns [64g, 64g+64) of S
//               and dP and head-dim columns [g d/2, (g+1) d/2) of the output.
// Tensor memory: two S buffers (0, 128), dP at 256, dQ at 384.  dS (bf16) is
// written over each group's own first 32 columns of its S buffer and read
// there by the dQ MMA.  Tensor pipe order: S_0 dP_0 | S_1 dP_1 dQ_0 | S_2 dP_2
// dQ_1 ...  S_{j+2} reuses S buffer j % 2 once dQ_j has read dS_j from it;
// dP_{j+1} waits until the compute threads have read dP_j.  An item's last
// tile issues its own dQ right after its dP (S_0 dP_0 dQ_0 for one tile).
#include "fa_internal.h"
#include "sm103a.cuh"

namespace fa {

namespace {

constexpr int kT = 128;
constexpr int kThreads = 320;
constexpr uint32_t kBlockBytes = 128u * 128u;

template <int D>
struct DqSmem {
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kDO = kQ + kTile;
  static constexpr uint32_t kK = kDO + kTile;                 // kStages
  static constexpr uint32_t kV = kK + kStages * kTile;        // kStages
  static constexpr uint32_t kLse = kV + kStages * kTile;      // 128 fp32
  static constexpr uint32_t kDr = kLse + 512u;                // 128 fp32
  static constexpr uint32_t kBar = kDr + 512u;
  static constexpr uint32_t kBytes = kBar + 256u;
};

enum : int {
  kSiteQ = 41, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteSFull, kSiteDpFull, kSiteDpFree,
  kSiteDsFull, kSiteDqDone, kSiteDqFinal, kSiteQEmpty, kSiteLdFree, kSiteDqFree,
  // drains on the way out
  kDrainQ = 61, kDrainK, kDrainV, kDrainMma
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], ds_full[2], dq_done[2];
  uint64_t dp_full, dp_free, dq_final, drain;
  uint64_t q_empty;   // the item's last dP MMA done: Q / dO may be replaced
  uint64_t ld_free;   // every compute thread has read the item's LSE / D
  uint64_t dq_free;   // the item's dQ read out of tensor memory
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Item u: query tile nt - 1 - u / (Hq B) (heaviest first under causal
// masking), then head fastest and batch, so the query heads of one kv group
// run side by side on neighbouring CTAs and share K / V through L2.
struct Item {
  int h, b, i, jlo, n;
};

__device__ __forceinline__ Item decode_item(int u, const DqArgs& a, int nt) {
  const int per = a.Hq * a.B;
  const int t = u / per;
  const int rem = u - t * per;
  Item it;
  it.h = rem % a.Hq;
  it.b = rem / a.Hq;
  it.i = nt - 1 - t;
  // Key tiles [jlo, jlo + n) hold keys some row of the tile may see.
  const int jhi = a.causal ? it.i + 1 : nt;
  it.jlo = a.window > 0 ? max(0, it.i * kT - a.window + 1) / kT : 0;
  it.n = jhi - it.jlo;
  return it;
}

// The CTA's k-th item: rounds of gridDim.x items, alternating direction.
__device__ __forceinline__ int item_of_round(int k) {
  const int g = gridDim.x;
  return k * g + ((k & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ TmaMap4 tmQ, const __grid_constant__ TmaMap4 tmK,
                     const __grid_constant__ TmaMap4 tmV, const __grid_constant__ TmaMap4 tmDO,
                     const DqArgs args, const DevStatus st) {
  using L = DqSmem<D>;
  constexpr int kAtoms = D / 64;
  constexpr int SK = L::kStages;
  constexpr int kHalfD = D / 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(st, kErrDeviceTimeout, 40);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int nt = (N + kT - 1) / kT;
  const int G = args.Hq / args.Hkv;
  const int n_items = args.Hq * args.B * nt;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->ds_full[x], 256);
      mbar_init(&bars->dq_done[x], 1);
    }
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 256);
    mbar_init(&bars->dq_final, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->ld_free, 256);
    mbar_init(&bars->dq_free, 256);
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
  const uint32_t tDP = tmem + 256, tDQ = tmem + 384;
  const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
  const int ntp = nt * kT;                       // padded rows per head of the LSE / D arrays

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int nq = 0, nk = 0, nv = 0;                // Q / dO, K and V copies issued
      bool pok = true;
      for (int k = 0; pok; ++k) {
        const int u = item_of_round(k);
        if (u >= n_items) break;
        const Item it = decode_item(u, args, nt);
        // Q / dO and LSE / D of the previous item: its last dP MMA has
        // completed and every compute thread has read its LSE / D.
        if (nq > 0 && !mbar_wait(&bars->q_empty, (nq - 1) & 1, st, abort_flag, kSiteQEmpty)) break;
        if (nq > 0 && !mbar_wait(&bars->ld_free, (nq - 1) & 1, st, abort_flag, kSiteLdFree)) break;
        const size_t roff = ((size_t)it.b * args.Hq + it.h) * ntp + (size_t)it.i * kT;
        mbar_arrive_expect_tx(&bars->q_full, 2 * L::kTile + 1024u);
        for (int a = 0; a < kAtoms; ++a) {
          tma_load_4d(smem + L::kQ + a * kBlockBytes, &tmQ, &bars->q_full, a * 64, it.i * kT, it.h, it.b);
          tma_load_4d(smem + L::kDO + a * kBlockBytes, &tmDO, &bars->q_full, a * 64, it.i * kT, it.h, it.b);
        }
        bulk_load(smem + L::kLse, args.lse2 + roff, 512u, &bars->q_full);
        bulk_load(smem + L::kDr, args.drow + roff, 512u, &bars->q_full);
        ++nq;
        const int kvh = it.h / G;
        for (int jj = 0; jj < it.n; ++jj) {
          const int s = nk % SK, r = nk / SK;
          if (r > 0 && !mbar_wait(&bars->k_empty[s], (r - 1) & 1, st, abort_flag, kSiteKEmpty)) { pok = false; break; }
          mbar_arrive_expect_tx(&bars->k_full[s], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_4d(smem + L::kK + s * L::kTile + a * kBlockBytes, &tmK, &bars->k_full[s], a * 64,
                        (it.jlo + jj) * kT, kvh, it.b);
          ++nk;
          if (r > 0 && !mbar_wait(&bars->v_empty[s], (r - 1) & 1, st, abort_flag, kSiteVEmpty)) { pok = false; break; }
          mbar_arrive_expect_tx(&bars->v_full[s], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_4d(smem + L::kV + s * L::kTile + a * kBlockBytes, &tmV, &bars->v_full[s], a * 64,
                        (it.jlo + jj) * kT, kvh, it.b);
          ++nv;
        }
      }
      // Every copy issued must have landed before the CTA may exit: only the
      // last copy into each buffer can still be in flight.
      if (nq > 0) mbar_wait_drain(&bars->q_full, (nq - 1) & 1, st, kDrainQ);
      for (int s = 0; s < SK; ++s) {
        if (s < nk) mbar_wait_drain(&bars->k_full[s], ((nk - 1 - (nk - 1 - s) % SK) / SK) & 1, st, kDrainK);
        if (s < nv) mbar_wait_drain(&bars->v_full[s], ((nv - 1 - (nv - 1 - s) % SK) / SK) & 1, st, kDrainV);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (see issuer_wait in sm103a.cuh):
    // every lane polls the barriers and elect.sync picks the issuing lane.
    constexpr bool kWarpIssue = true;
    {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);   // S, dP
      constexpr uint32_t idQ = idesc_bf16(128, D, false, true);       // dQ += dS K (K as the MN-major operand)
      // Operand descriptors, built once: a K / V stage or a k16 step adds a constant.
      const uint64_t dQk = desc_kmajor(sQ, 0, kBlockBytes), dOk = desc_kmajor(sDO, 0, kBlockBytes);
      const uint64_t dKk = desc_kmajor(sK, 0, kBlockBytes), dKm = desc_mnmajor(sK, 0, kBlockBytes);
      const uint64_t dVk = desc_kmajor(sV, 0, kBlockBytes);
      // dQ of tile tg (the item's jj-th, item ci): A = dS in S buffer tg % 2
      // (group g's keys at columns 64g..), B = K; releases the K stage
      // afterwards.  The item's first dQ overwrites the accumulator, so it
      // waits until the previous item's dQ has been read out.
      auto issue_dq = [&](int tg, int jj, int ci) -> bool {
        const int x = tg & 1, s = tg % SK;
        if (jj == 0 && ci > 0 && !issuer_wait<kWarpIssue>(&bars->dq_free, (ci - 1) & 1, st, abort_flag, kSiteDqFree)) return false;
        if (!issuer_wait<kWarpIssue>(&bars->ds_full[x], (tg >> 1) & 1, st, abort_flag, kSiteDsFull)) return false;
        tc_fence_after();
        const uint64_t dk = dKm + (uint64_t)s * (L::kTile >> 4);
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          issue_ts<kWarpIssue>(tDQ, tmem + x * 128 + (k16 >> 2) * 64 + (k16 & 3) * 8, dk + desc_step_mnmajor(k16), idQ,
                      (jj > 0 || k16 > 0) ? 1u : 0u);
        issue_commit<kWarpIssue>(&bars->dq_done[x]);
        issue_commit<kWarpIssue>(&bars->k_empty[s]);
        return true;
      };
      bool ok = true;
      int tiles = 0;                             // tiles of the CTA's earlier items
      for (int k = 0, ci = 0; ok; ++k, ++ci) {
        const int u = item_of_round(k);
        if (u >= n_items) break;
        const int n = decode_item(u, args, nt).n;
        if (!issuer_wait<kWarpIssue>(&bars->q_full, ci & 1, st, abort_flag, kSiteQ)) break;
        for (int jj = 0; jj < n; ++jj) {
          const int tg = tiles + jj;
          const int x = tg & 1, s = tg % SK;
          // S_tg overwrites dS_{tg-2} (read by dQ_{tg-2}).
          if (tg >= 2 && !issuer_wait<kWarpIssue>(&bars->dq_done[x], ((tg - 2) >> 1) & 1, st, abort_flag, kSiteDqDone)) { ok = false; break; }
          if (!issuer_wait<kWarpIssue>(&bars->k_full[s], (tg / SK) & 1, st, abort_flag, kSiteKFull)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dk = dKk + (uint64_t)s * (L::kTile >> 4);
#pragma unroll
          for (int k16 = 0; k16 < D / 16; ++k16)
            issue_ss<kWarpIssue>(tmem + x * 128, dQk + desc_step_kmajor(k16, kBlockBytes),
                        dk + desc_step_kmajor(k16, kBlockBytes), idSS, k16 > 0);
          issue_commit<kWarpIssue>(&bars->s_full[x]);
          // dP_tg overwrites dP_{tg-1}: the compute threads must have read it.
          if (tg >= 1 && !issuer_wait<kWarpIssue>(&bars->dp_free, (tg - 1) & 1, st, abort_flag, kSiteDpFree)) { ok = false; break; }
          if (!issuer_wait<kWarpIssue>(&bars->v_full[s], (tg / SK) & 1, st, abort_flag, kSiteVFull)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dv = dVk + (uint64_t)s * (L::kTile >> 4);
#pragma unroll
          for (int k16 = 0; k16 < D / 16; ++k16)
            issue_ss<kWarpIssue>(tDP, dOk + desc_step_kmajor(k16, kBlockBytes), dv + desc_step_kmajor(k16, kBlockBytes),
                        idSS, k16 > 0);
          issue_commit<kWarpIssue>(&bars->dp_full);
          issue_commit<kWarpIssue>(&bars->v_empty[s]);
          if (jj == n - 1) issue_commit<kWarpIssue>(&bars->q_empty);   // the item's Q / dO are no longer read
          if (jj >= 1 && !issue_dq(tg - 1, jj - 1, ci)) { ok = false; break; }
          if (jj == n - 1 && !issue_dq(tg, jj, ci)) { ok = false; break; }
        }
        if (!ok) break;
        issue_commit<kWarpIssue>(&bars->dq_final);
        tiles += n;
      }
      issue_commit<kWarpIssue>(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, st, kDrainMma);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int g = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    bool ok = true;
    int tiles = 0;                                 // tiles of the CTA's earlier items
    for (int k = 0, ci = 0; ok; ++k, ++ci) {
      const int u = item_of_round(k);
      if (u >= n_items) break;
      const Item it = decode_item(u, args, nt);
      const int q = it.i * kT + r;                 // this thread's query
      if (!mbar_wait_warp(&bars->q_full, ci & 1, st, abort_flag, kSiteQ)) break;
      // Rows past N have LSE*log2(e) = +inf in the padded array: P = 0.
      const float lse2 = reinterpret_cast<const float*>(smem + L::kLse)[r];
      const float drow = reinterpret_cast<const float*>(smem + L::kDr)[r];
      mbar_arrive(&bars->ld_free);                 // the next item's LSE / D may replace them
      const uint64_t nl2 = f2pack(-lse2, -lse2);
      const uint64_t nd2 = f2pack(-drow, -drow);
      for (int jj = 0; jj < it.n; ++jj) {
        const int tg = tiles + jj;
        const int x = tg & 1;
        const int j = it.jlo + jj;
        if (!mbar_wait_warp(&bars->s_full[x], (tg >> 1) & 1, st, abort_flag, kSiteSFull)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem + x * 128 + lane_off + g * 64;
        uint32_t pr[2][32];
        tmem_ld32(tS, pr[0]);
        tmem_ld32(tS + 32, pr[1]);
        tmem_wait_ld();
        reg_fence(pr[0]);
        reg_fence(pr[1]);
        // Visible key columns of this group: [clo, chi) (causal: key <= q;
        // window: key > q - w; keys past N never).
        const int kc0 = j * kT + g * 64;           // key of the group's column 0
        int chi = min(64, N - kc0);
        if (args.causal) chi = min(chi, q + 1 - kc0);
        const int clo = args.window > 0 ? max(0, q - args.window + 1 - kc0) : 0;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = hq * 32 + e;
            float lo, hi;
            f2unpack(ffma2(f2pack(__uint_as_float(pr[hq][e]), __uint_as_float(pr[hq][e + 1])), sl2x2, nl2), lo, hi);
            lo = (col >= clo && col < chi) ? ex2(lo) : 0.f;
            hi = (col + 1 >= clo && col + 1 < chi) ? ex2(hi) : 0.f;
            pr[hq][e] = __float_as_uint(lo);
            pr[hq][e + 1] = __float_as_uint(hi);
          }
        }
        if (!mbar_wait_warp(&bars->dp_full, tg & 1, st, abort_flag, kSiteDpFull)) { ok = false; break; }
        tc_fence_after();
        uint32_t dp[2][32];
        tmem_ld32(tDP + lane_off + g * 64, dp[0]);
        tmem_ld32(tDP + lane_off + g * 64 + 32, dp[1]);
        tmem_wait_ld();
        reg_fence(dp[0]);
        reg_fence(dp[1]);
        tc_fence_before();
        mbar_arrive(&bars->dp_free);
        uint32_t ds[32];
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a0, a1;
            f2unpack(fmul2(f2pack(__uint_as_float(pr[hq][e]), __uint_as_float(pr[hq][e + 1])),
                           fadd2(f2pack(__uint_as_float(dp[hq][e]), __uint_as_float(dp[hq][e + 1])), nd2)),
                     a0, a1);
            ds[hq * 16 + e / 2] = cvt_bf16x2(a0, a1);
          }
        }
        // dS (bf16) over this group's own first 32 columns of the S buffer,
        // already read into registers: the A operand of dQ_jj.
        tmem_st32(tS, ds);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->ds_full[x]);
      }

      if (!ok) break;
      tiles += it.n;
      if (!mbar_wait_warp(&bars->dq_final, ci & 1, st, abort_flag, kSiteDqFinal)) break;
      tc_fence_after();
      uint32_t v[kHalfD / 32][32];
#pragma unroll
      for (int c = 0; c < kHalfD / 32; ++c) tmem_ld32(tDQ + lane_off + g * kHalfD + c * 32, v[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < kHalfD / 32; ++c) reg_fence(v[c]);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);                 // the next item's first dQ MMA may overwrite it
      if (q < N) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.dq) +
                             (((size_t)it.b * args.Hq + it.h) * N + (size_t)q) * D + g * kHalfD;
        // dQ rows start on 32-byte boundaries whenever dQ itself does.
        const bool v8 = (reinterpret_cast<uintptr_t>(args.dq) & 31u) == 0;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = cvt_bf16x2(__uint_as_float(v[c][2 * e]) * args.scale, __uint_as_float(v[c][2 * e + 1]) * args.scale);
          if (v8) {
            // 32-byte stores: a warp instruction writes whole 32-byte sectors of 32 rows.
            st_global_v8(dst + c * 32, w);
            st_global_v8(dst + c * 32 + 16, w + 8);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4*>(dst + c * 32 + e * 8) = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
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

}  // namespace

template <int D>
static cudaError_t configure_dq_d() {
  using L = DqSmem<D>;
  static_assert(L::kBytes <= 232448, "shared memory budget");
  static_assert(sizeof(Bars) <= 256, "barrier block");
  return cudaFuncSetAttribute(fa_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
}

cudaError_t configure_dq_kernels() {
  cudaError_t e = configure_dq_d<64>();
  if (e == cudaSuccess) e = configure_dq_d<128>();
  return e;
}

template <int D>
static cudaError_t launch_dq_d(const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                               const TmaMap4& tdo, const DqArgs& a, const DevStatus& st, int num_sms,
                               cudaStream_t stream) {
  using L = DqSmem<D>;
  // Persistent: one CTA per SM (the shared memory allows no second one),
  // never more CTAs than items.
  const long long items = (long long)a.Hq * a.B * ((a.N + kT - 1) / kT);
  const int grid = (int)(items < num_sms ? items : num_sms);
  fa_bwd_dq_kernel<D><<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, tdo, a, st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int d, const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                          const TmaMap4& tdo, const DqArgs& a, const DevStatus& st, int num_sms,
                          cudaStream_t stream) {
  if (d == 64) return launch_dq_d<64>(tq, tk, tv, tdo, a, st, num_sms, stream);
  return launch_dq_d<128>(tq, tk, tv, tdo, a, st, num_sms, stream);
}

}  // namespace fa
