// Exact attention backward on sm_103a, recomputing P tile by tile from the
// saved log-sum-exp instead of storing it ([FA-memory] "38.解释FlashAttention的
// 显存优化原理", part 2(2); [QBank-36] part 7; [Lecture] "推导 FlashAttention 的
// 在线 softmax", closing paragraphs).
//
// Three kernels on the caller's stream:
//   1. preprocess: D_i = sum_c dO[i,c] * O[i,c] (warp-shuffle reduction),
//      LSE_i * log2(e), both padded per head to a multiple of 128 rows (+inf
//      and 0 past N), and zero the fp32 dQ accumulator.
//   2. dkdv: persistent, one CTA per SM; a unit is one 128-key tile of one kv
//      head, and the CTA loops over every query head of its group and every
//      128-query tile that can see it.  dK and dV accumulate in tensor memory
//      and are written once per unit: no atomics.  The next unit's K / V load
//      as soon as the unit's last MMAs are done.
//      Per (query tile, key tile) it recomputes S^T = K Q^T, P^T = 2^(S^T *
//      scale * log2 e - LSE * log2 e), dP^T = V dO^T, dS^T = P^T (dP^T - D),
//      and issues dV += P^T dO, dK += dS^T Q, dQ_partial = dS K; the dQ
//      partial is added into the fp32 accumulator (the separate dQ reduction).
//   3. dq_convert: dQ = bf16(scale * accumulator).
//
// dkdv CTA layout (352 threads):
//   warp 0      TMA producer: K, V once; per item Q_i, dO_i (2 slots each) and
//               the item's 128 LSE / D values (bulk copies, 2 slots)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-5   compute warpgroup 0, warps 6-9 compute warpgroup 1: thread t
//               of a group owns key row t (TMEM lane t) for S^T, dP^T, dK, dV
//               and query row t for the dQ partial; group g handles query
//               columns [64g, 64g+64) and head-dim columns [g d/2, (g+1) d/2).
//   warp 10     dQ store: adds the staged dQ partials into the fp32
//               accumulator with TMA reduce-adds and returns the staging slots
// Tensor memory: S^T at columns 0-127; P^T (bf16) is written back over the
// group's own columns 0-31 / 64-95 and read there by the dV MMA, dS^T (bf16)
// over 32-63 / 96-127 and read there by the dK MMA;
// dP^T at 128-255, reused for the dQ partial; dV at 256, dK at 256 + d.
// dS^T (bf16) also goes to a shared-memory tile, read by the dQ MMA as dS
// (MN-major).
//
// Tensor pipe order per item t:  S_t, dP_t, dV_t, dK_t, dQ_t, S_{t+1}, ...
// S_{t+1} waits for dK_t (it overwrites P^T_t and dS^T_t); dP_{t+1} waits until
// the dQ partial of item t has been read out of the same columns.
#include "fa_internal.h"
#include "sm103a.cuh"

namespace fa {

namespace {

constexpr int kT = 128;             // rows per query tile and per key tile
constexpr int kThreads = 352;
constexpr uint32_t kBlockBytes = 128u * 128u;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdSmem {
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;          // 2 slots
  static constexpr uint32_t kDO = kQ + 2 * kTile;     // 2 slots
  static constexpr uint32_t kDS = kDO + 2 * kTile;
  static constexpr uint32_t kLse = kDS + 128u * 128u * 2u;   // 2 slots x 128 fp32
  static constexpr uint32_t kDr = kLse + 1024u;               // 2 slots x 128 fp32
  static constexpr uint32_t kBar = kDr + 1024u;
  static constexpr uint32_t kBytes = kBar + 256u;
};

enum : int {
  kSiteKV = 11, kSiteQEmpty, kSiteDoEmpty, kSiteLdEmpty, kSiteQFull, kSiteDvDone, kSiteDoFull, kSiteDqEmpty,
  kSitePFull, kSiteDsFull, kSiteLdFull, kSiteSFull, kSiteDpFull, kSiteDqFull, kSiteDkvDone, kSiteStFull, kSiteDkDone,
  // drains on the way out
  kDrainKV = 31, kDrainLd, kDrainQ, kDrainDo, kDrainMma
};

struct Bars {
  uint64_t kv_full, kv_empty, dkv_free;
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2], ld_full[2], ld_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, dk_done, dq_full, dq_empty, dkv_done, drain;
  uint64_t st_full[2][2];   // [slot][group]: the group's dQ partial of the slot's item is staged
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// A unit is one 128-key tile of one kv head of one batch; its CTA loops over
// every query head of the group and every query tile that sees the key tile
// (causal: i >= j; window w: i <= (128j + 126 + w) / 128).  Causal units go
// heaviest first (smallest key tile first), dealt to the persistent CTAs in
// snake order: rounds alternate direction over the CTAs.  Without causal
// masking every unit costs the same, and kHeadMajor puts the key tiles of one
// kv head next to each other: the units running at the same time then share
// the query tiles and dQ accumulator rows of a few heads, which stay in L2,
// instead of touching every head's.  (A run-time switch between the two
// orders slowed the causal kernel by 3-5 %, so the order is a compile-time
// parameter.)
struct Unit {
  int kvh, b, j, i0, nqi, n_items;
};

template <bool kHeadMajor>
__device__ __forceinline__ Unit decode_unit(int idx, const BwdArgs& a, int nt) {
  const int per = a.Hkv * a.B;
  Unit u;
  int kb;
  if constexpr (kHeadMajor) {
    kb = idx / nt;
    u.j = idx - kb * nt;
  } else {
    u.j = idx / per;
    kb = idx - u.j * per;
  }
  u.kvh = kb % a.Hkv;
  u.b = kb / a.Hkv;
  u.i0 = a.causal ? u.j : 0;
  const int i1 = a.window > 0 ? min(nt, (u.j * kT + kT - 2 + a.window) / kT + 1) : nt;
  u.nqi = i1 - u.i0;
  u.n_items = (a.Hq / a.Hkv) * u.nqi;
  return u;
}

__device__ __forceinline__ int unit_of_round(int k) {
  const int g = gridDim.x;
  return k * g + ((k & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// kDq = false: dK and dV only (the deterministic backward computes dQ in its
// own kernel): no dQ MMA, no dS tile in shared memory, no dQ staging or
// reduce-adds; the store warp idles.
template <int D, bool kDq, bool kHeadMajor>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ TmaMap4 tmQ, const __grid_constant__ TmaMap4 tmK,
                       const __grid_constant__ TmaMap4 tmV, const __grid_constant__ TmaMap4 tmDO,
                       const __grid_constant__ TmaMap3 tmDQ, const BwdArgs args, const DevStatus st) {
  using L = BwdSmem<D>;
  constexpr int kAtoms = D / 64;
  constexpr int kHalfD = D / 2;
  constexpr int kPasses = kHalfD / 32;   // 32-column dQ staging passes per group
  constexpr bool kWarpIssue = true;        // see the MMA issuer
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort;

  // The swizzled operand tiles need a 1024-byte aligned base.  The dynamic
  // shared memory of a kernel without static shared memory starts there; if
  // it ever did not, stop cleanly with an error instead of computing garbage.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(st, kErrDeviceTimeout, 10);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int nt = (N + kT - 1) / kT;
  const int G = args.Hq / args.Hkv;
  const int n_units = args.Hkv * args.B * nt;
  // Items are counted across the CTA's units (T = items of earlier units), so
  // the per-item barriers and the Q / dO / LSE slots run on without a break.

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);   // a unit's last MMAs done: K / V may be replaced
    mbar_init(&bars->dkv_free, 256); // the unit's dK / dV read out of tensor memory
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], kDq ? 2 : 1);   // dK/dQ MMAs done (+ dQ staging read by TMA)
      mbar_init(&bars->do_full[s], 1);
      mbar_init(&bars->do_empty[s], kDq ? 2 : 1);  // dP/dV MMAs done (+ dQ staging read by TMA)
      mbar_init(&bars->ld_full[s], 1);
      mbar_init(&bars->ld_empty[s], 256);
      for (int g = 0; g < 2; ++g) mbar_init(&bars->st_full[s][g], 128);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 256);
    mbar_init(&bars->dkv_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQ);
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
  const uint32_t sDS = smem_u32(smem + L::kDS);
  const int ntp = nt * kT;                       // padded rows per head of the LSE / D arrays
  // Staging block of the dQ partial of (slot, group g, 32-column pass q): for
  // d = 128 pass 0 uses block g of the slot's Q tile and pass 1 block g of
  // its dO tile; for d = 64 (one 16 KB block per tile) group 0 uses the Q
  // tile and group 1 the dO tile.  The Q-tile blocks are added first, so the
  // Q slot, needed first by the next item that uses it, is returned first.
  auto stage_in_q = [&](int g, int q) -> bool { return kPasses == 2 ? q == 0 : g == 0; };
  auto stage_addr = [&](int slot, int g, int q) -> uint32_t {
    return (stage_in_q(g, q) ? sQ : sDO) + slot * L::kTile + (kPasses == 2 ? g * kBlockBytes : 0u);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int n_ld[2] = {0, 0}, n_q[2] = {0, 0}, n_do[2] = {0, 0};   // copies issued per slot
      int n_kv = 0, T = 0;
      bool pok = true;
      for (int round = 0; pok; ++round) {
        const int uidx = unit_of_round(round);
        if (uidx >= n_units) break;
        const Unit un = decode_unit<kHeadMajor>(uidx, args, nt);
        // LSE*log2(e) and D of local item u (512 bytes each) go to slot
        // (T + u) % 2; they are issued one item ahead of that item's Q / dO.
        auto issue_ld = [&](int u) -> bool {
          if (u >= un.n_items) return true;
          const int tg = T + u;
          const int slot = tg & 1;
          if (tg >= 2 && !mbar_wait(&bars->ld_empty[slot], ((tg >> 1) - 1) & 1, st, abort_flag, kSiteLdEmpty))
            return false;
          const int h = un.kvh * G + u / un.nqi;
          const int i = un.i0 + u % un.nqi;
          const size_t roff = ((size_t)un.b * args.Hq + h) * ntp + (size_t)i * kT;
          mbar_arrive_expect_tx(&bars->ld_full[slot], 1024u);
          bulk_load(smem + L::kLse + slot * 512, args.lse2 + roff, 512u, &bars->ld_full[slot]);
          bulk_load(smem + L::kDr + slot * 512, args.drow + roff, 512u, &bars->ld_full[slot]);
          ++n_ld[slot];
          return true;
        };
        pok = issue_ld(0);
        for (int t = 0; pok && t < un.n_items; ++t) {
          const int tg = T + t;
          const int h = un.kvh * G + t / un.nqi;
          const int i = un.i0 + t % un.nqi;
          const int slot = tg & 1;
          const uint32_t ph = ((tg >> 1) - 1) & 1;   // phase of this slot's previous use
          if (tg >= 2 && !mbar_wait(&bars->q_empty[slot], ph, st, abort_flag, kSiteQEmpty)) { pok = false; break; }
          mbar_arrive_expect_tx(&bars->q_full[slot], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_4d(smem + L::kQ + slot * L::kTile + a * kBlockBytes, &tmQ, &bars->q_full[slot], a * 64,
                        i * kT, h, un.b);
          ++n_q[slot];
          if (tg >= 2 && !mbar_wait(&bars->do_empty[slot], ph, st, abort_flag, kSiteDoEmpty)) { pok = false; break; }
          mbar_arrive_expect_tx(&bars->do_full[slot], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_4d(smem + L::kDO + slot * L::kTile + a * kBlockBytes, &tmDO, &bars->do_full[slot], a * 64,
                        i * kT, h, un.b);
          ++n_do[slot];
          if (t == 0) {
            // K and V of the unit replace the previous unit's once its last
            // MMAs have completed (the unit's first Q / dO are already on
            // their way).
            if (n_kv > 0 && !mbar_wait(&bars->kv_empty, (n_kv - 1) & 1, st, abort_flag, kSiteKV)) {
              pok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->kv_full, 2 * L::kTile);
            for (int a = 0; a < kAtoms; ++a) {
              tma_load_4d(smem + L::kK + a * kBlockBytes, &tmK, &bars->kv_full, a * 64, un.j * kT, un.kvh, un.b);
              tma_load_4d(smem + L::kV + a * kBlockBytes, &tmV, &bars->kv_full, a * 64, un.j * kT, un.kvh, un.b);
            }
            ++n_kv;
          }
          pok = issue_ld(t + 1);
        }
        T += un.n_items;
      }
      // Every copy issued must have landed before the CTA may exit.
      if (n_kv) mbar_wait_drain(&bars->kv_full, (n_kv - 1) & 1, st, kDrainKV);
      for (int s = 0; s < 2; ++s) {
        if (n_ld[s]) mbar_wait_drain(&bars->ld_full[s], (n_ld[s] - 1) & 1, st, kDrainLd);
        if (n_q[s]) mbar_wait_drain(&bars->q_full[s], (n_q[s] - 1) & 1, st, kDrainQ);
        if (n_do[s]) mbar_wait_drain(&bars->do_full[s], (n_do[s] - 1) & 1, st, kDrainDo);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // kWarpIssue: the whole warp runs the issuer loop, every lane polls the
    // barriers and elect.sync picks the lane that issues each MMA and commit
    // (a converged warp issues tcgen05.mma faster than a lone lane); else
    // lane 0 alone.
    auto wait = [&](uint64_t* bar, uint32_t parity, int site) {
      return issuer_wait<kWarpIssue>(bar, parity, st, abort_flag, site);
    };
    auto ss = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) { issue_ss<kWarpIssue>(d, a, b, id, acc); };
    auto ts = [](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) { issue_ts<kWarpIssue>(d, a, b, id, acc); };
    auto commit = [](uint64_t* bar) { issue_commit<kWarpIssue>(bar); };
    if (kWarpIssue || lane == 0) {
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);   // S^T, dP^T
      constexpr uint32_t idKM = idesc_bf16(128, D, false, true);      // dV, dK
      constexpr uint32_t idMM = idesc_bf16(128, D, true, true);       // dQ
      // Operand descriptors, built once: a k16 step adds a constant.
      const uint64_t dKk = desc_kmajor(sK, 0, kBlockBytes), dVk = desc_kmajor(sV, 0, kBlockBytes);
      const uint64_t dKm = desc_mnmajor(sK, 0, kBlockBytes), dDSm = desc_mnmajor(sDS, 0, kBlockBytes);
      const uint64_t dQk0 = desc_kmajor(sQ, 0, kBlockBytes), dQk1 = desc_kmajor(sQ + L::kTile, 0, kBlockBytes);
      const uint64_t dOk0 = desc_kmajor(sDO, 0, kBlockBytes), dOk1 = desc_kmajor(sDO + L::kTile, 0, kBlockBytes);
      const uint64_t dQm0 = desc_mnmajor(sQ, 0, kBlockBytes), dQm1 = desc_mnmajor(sQ + L::kTile, 0, kBlockBytes);
      const uint64_t dOm0 = desc_mnmajor(sDO, 0, kBlockBytes), dOm1 = desc_mnmajor(sDO + L::kTile, 0, kBlockBytes);
      bool ok = true;
      int T = 0, nu = 0;
      for (int round = 0; ok; ++round, ++nu) {
        const int uidx = unit_of_round(round);
        if (uidx >= n_units) break;
        const Unit un = decode_unit<kHeadMajor>(uidx, args, nt);
        if (!wait(&bars->kv_full, nu & 1, kSiteKV)) break;
      for (int t = 0; ok && t < un.n_items; ++t) {
        const int tg = T + t;
        const int slot = tg & 1;
        const uint32_t sph = (tg >> 1) & 1;  // slot phase
        const uint32_t ph = tg & 1;          // per-item barrier phase
        const uint32_t pph = (tg - 1) & 1;   // previous item's phase
        const uint64_t dQk = slot ? dQk1 : dQk0, dOk = slot ? dOk1 : dOk0;
        const uint64_t dQm = slot ? dQm1 : dQm0, dOm = slot ? dOm1 : dOm0;
        if (!wait(&bars->q_full[slot], sph, kSiteQFull)) { ok = false; break; }
        // S_{t+1} overwrites the score region, which holds P^T_t (read by dV_t)
        // and dS^T_t (read by dK_t); dK_t is the later of the two.
        if (tg > 0 && !wait(&bars->dk_done, pph, kSiteDkDone)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          ss(tS, dKk + desc_step_kmajor(k16, kBlockBytes), dQk + desc_step_kmajor(k16, kBlockBytes), idSS,
                      k16 > 0);
        commit(&bars->s_full);
        if (!wait(&bars->do_full[slot], sph, kSiteDoFull)) { ok = false; break; }
        // dP_t overwrites the dQ partial of item t-1 (read out by then) or,
        // without dQ, dP^T of item t-1 (read before ds_full of t-1).
        if (kDq && tg > 0 && !wait(&bars->dq_empty, pph, kSiteDqEmpty)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          ss(tDP, dVk + desc_step_kmajor(k16, kBlockBytes), dOk + desc_step_kmajor(k16, kBlockBytes), idSS,
                      k16 > 0);
        commit(&bars->dp_full);
        if (!wait(&bars->p_full, ph, kSitePFull)) { ok = false; break; }
        // The unit's first dV / dK overwrite the previous unit's accumulators:
        // its epilogue must have read them out.
        if (t == 0 && nu > 0 && !wait(&bars->dkv_free, (nu - 1) & 1, kSiteDkvDone)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P^T for query columns 16*k16.. lives at column (k16/4)*64 + (k16%4)*8.
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          ts(tDV, tS + (k16 >> 2) * 64 + (k16 & 3) * 8, dOm + desc_step_mnmajor(k16), idKM,
                      (t > 0 || k16 > 0) ? 1u : 0u);
        commit(&bars->do_empty[slot]);
        if (!wait(&bars->ds_full, ph, kSiteDsFull)) { ok = false; break; }
        tc_fence_after();
        // dS^T for query columns 16*k16.. lives at column (k16/4)*64 + 32 + (k16%4)*8.
#pragma unroll
        for (int k16 = 0; k16 < kT / 16; ++k16)
          ts(tDK, tS + (k16 >> 2) * 64 + 32 + (k16 & 3) * 8, dQm + desc_step_mnmajor(k16), idKM,
                      (t > 0 || k16 > 0) ? 1u : 0u);
        commit(&bars->dk_done);
        if (kDq) {
#pragma unroll
          for (int k16 = 0; k16 < kT / 16; ++k16)
            ss(tDP, dDSm + desc_step_mnmajor(k16), dKm + desc_step_mnmajor(k16), idMM,
                        k16 > 0 ? 1u : 0u);
          commit(&bars->dq_full);
        }
        commit(&bars->q_empty[slot]);
      }
      if (!ok) break;
      commit(&bars->dkv_done);
      commit(&bars->kv_empty);
      T += un.n_items;
      }
      commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, st, kDrainMma);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ compute
    const int g = (warp - 2) >> 2;                 // warpgroup 0 or 1
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int c0 = g * 64;                         // this group's query columns
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    bool ok = true;
    int T = 0, nu = 0;
    for (int round = 0; ok; ++round, ++nu) {
    const int uidx = unit_of_round(round);
    if (uidx >= n_units) break;
    const Unit un = decode_unit<kHeadMajor>(uidx, args, nt);
    const int key = un.j * kT + r;
    for (int t = 0; t < un.n_items; ++t) {
      const int tg = T + t;
      const int slot = tg & 1;
      const uint32_t ph = tg & 1;
      const int i = un.i0 + t % un.nqi;
      auto dq_stage = [&](int q) { return stage_addr(slot, g, q); };
      const float* lse_t = reinterpret_cast<const float*>(smem + L::kLse + slot * 512) + c0;
      const float* dr_t = reinterpret_cast<const float*>(smem + L::kDr + slot * 512) + c0;
      if (!mbar_wait_warp(&bars->ld_full[slot], (tg >> 1) & 1, st, abort_flag, kSiteLdFull)) { ok = false; break; }
      if (!mbar_wait_warp(&bars->s_full, ph, st, abort_flag, kSiteSFull)) { ok = false; break; }
      tc_fence_after();
      uint32_t pr[2][32];
      tmem_ld32(tS + lane_off + c0, pr[0]);
      tmem_ld32(tS + lane_off + c0 + 32, pr[1]);
      tmem_wait_ld();
      reg_fence(pr[0]);
      reg_fence(pr[1]);
      // P^T[key, q] = 2^(s * sl2 - lse2[q]); zero where the key is past N or
      // (diagonal tile, causal) after the query.  Query rows past N have
      // lse2 = +inf in the padded array, which gives 0.
      // This key is visible to the group's query columns [clo, chi): causal
      // needs query >= key, a window w also query < key + w.
      const int qcol0 = i * kT + c0;               // query index of the group's column 0
      int clo = args.causal ? min(64, max(0, key - qcol0)) : 0;
      const int chi = args.window > 0 ? min(64, max(0, key + args.window - qcol0)) : 64;
      if (key >= N) clo = 64;
      uint32_t pk[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = q * 32 + e;
          const float4 l4 = *reinterpret_cast<const float4*>(lse_t + (col & ~3));
          const float la = (col & 2) ? l4.z : l4.x;
          const float lb = (col & 2) ? l4.w : l4.y;
          float lo, hi;
          f2unpack(ffma2(f2pack(__uint_as_float(pr[q][e]), __uint_as_float(pr[q][e + 1])), sl2x2,
                         f2pack(-la, -lb)),
                   lo, hi);
          lo = (col >= clo && col < chi) ? ex2(lo) : 0.f;
          hi = (col + 1 >= clo && col + 1 < chi) ? ex2(hi) : 0.f;
          pr[q][e] = __float_as_uint(lo);
          pr[q][e + 1] = __float_as_uint(hi);
          pk[col >> 1] = cvt_bf16x2(lo, hi);
        }
      }
      tmem_st32(tS + lane_off + c0, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);

      if (!mbar_wait_warp(&bars->dp_full, ph, st, abort_flag, kSiteDpFull)) { ok = false; break; }
      tc_fence_after();
      uint32_t dp[2][32];
      tmem_ld32(tDP + lane_off + c0, dp[0]);
      tmem_ld32(tDP + lane_off + c0 + 32, dp[1]);
      tmem_wait_ld();
      reg_fence(dp[0]);
      reg_fence(dp[1]);
      uint32_t ds[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int col = q * 32 + e;
          const float4 d4 = *reinterpret_cast<const float4*>(dr_t + col);
          float a0, a1, a2, a3;
          f2unpack(fmul2(f2pack(__uint_as_float(pr[q][e]), __uint_as_float(pr[q][e + 1])),
                         fadd2(f2pack(__uint_as_float(dp[q][e]), __uint_as_float(dp[q][e + 1])),
                               f2pack(-d4.x, -d4.y))),
                   a0, a1);
          f2unpack(fmul2(f2pack(__uint_as_float(pr[q][e + 2]), __uint_as_float(pr[q][e + 3])),
                         fadd2(f2pack(__uint_as_float(dp[q][e + 2]), __uint_as_float(dp[q][e + 3])),
                               f2pack(-d4.z, -d4.w))),
                   a2, a3);
          ds[col >> 1] = cvt_bf16x2(a0, a1);
          ds[(col >> 1) + 1] = cvt_bf16x2(a2, a3);
        }
      }
      // dS^T row -> tensor memory (this group's spare score columns, the A
      // operand of dK) and this group's 64-column block of the shared tile
      // (the A operand of dQ).
      tmem_st32(tS + lane_off + c0 + 32, ds);
      if (kDq) {
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16)
          st_shared_v4(sDS + g * kBlockBytes + swz128(r, c16), ds[c16 * 4], ds[c16 * 4 + 1], ds[c16 * 4 + 2],
                       ds[c16 * 4 + 3]);
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
      mbar_arrive(&bars->ld_empty[slot]);

      if (!kDq) continue;
      if (!mbar_wait_warp(&bars->dq_full, ph, st, abort_flag, kSiteDqFull)) { ok = false; break; }
      tc_fence_after();
      // dQ partial row r (a query) x this group's head-dim columns: read it out
      // of tensor memory (freeing those columns for dP^T of the next item) and
      // stage it 32 columns at a time, 128-byte swizzled, in this item's dO
      // and Q tiles -- free now: their last readers, the dV and dK MMAs, have
      // completed.  The store warp adds the staged blocks into the fp32
      // accumulator.
      {
        uint32_t v[kPasses][32];
#pragma unroll
        for (int q = 0; q < kPasses; ++q) tmem_ld32(tDP + lane_off + g * kHalfD + q * 32, v[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kPasses; ++q) reg_fence(v[q]);
        tc_fence_before();
        mbar_arrive(&bars->dq_empty);
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
          const uint32_t stage = dq_stage(q);
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16)
            st_shared_v4(stage + swz128(r, c16), v[q][c16 * 4], v[q][c16 * 4 + 1], v[q][c16 * 4 + 2],
                         v[q][c16 * 4 + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->st_full[slot][g]);
      }
    }

    if (!ok || !mbar_wait_warp(&bars->dkv_done, nu & 1, st, abort_flag, kSiteDkvDone)) {
      ok = false;
      break;
    }
    {
      tc_fence_after();
      const size_t kvrow = ((size_t)un.b * args.Hkv + un.kvh) * N + (size_t)key;
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const uint32_t src = (pass == 0 ? tDV : tDK) + lane_off + g * kHalfD;
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(pass == 0 ? args.dv : args.dk) + kvrow * D + g * kHalfD;
        const float mul = pass == 0 ? 1.f : args.scale;
#pragma unroll
        for (int q = 0; q < kHalfD / 32; ++q) {
          uint32_t v[32];
          tmem_ld32(src + q * 32, v);
          tmem_wait_ld();
          reg_fence(v);
          if (pass == 1 && q == kHalfD / 32 - 1) {
            // Last read of the unit's accumulators: the next unit may start
            // its first dV / dK MMA.
            tc_fence_before();
            mbar_arrive(&bars->dkv_free);
          }
          if (key < N) {
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              w[c] = cvt_bf16x2(__uint_as_float(v[2 * c]) * mul, __uint_as_float(v[2 * c + 1]) * mul);
            if (args.v8) {
              // One row's 64 bytes in two 32-byte stores: a warp instruction
              // writes whole 32-byte sectors of 32 rows.
              st_global_v8(dst + q * 32, w);
              st_global_v8(dst + q * 32 + 16, w + 8);
            } else {
#pragma unroll
              for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(dst + q * 32 + c * 8) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            }
          }
        }
      }
    }
    T += un.n_items;
    }
  } else {
    // ------------------------------------------------------------ dQ store
    // Per item: wait until both groups have staged their dQ partial, add each
    // 128 x 32 fp32 block into the accumulator with one tiled TMA reduce-add
    // (rows past N are clipped by the tensor map), and hand the item's dO and
    // Q slots back to the producer once TMA has read the staging.  Waiting
    // for those reads here keeps them off the compute warps.
    if (kDq && lane == 0) {
      bool sok = true;
      int T = 0;
      for (int round = 0; sok; ++round) {
      const int uidx = unit_of_round(round);
      if (uidx >= n_units) break;
      const Unit un = decode_unit<kHeadMajor>(uidx, args, nt);
      for (int t = 0; t < un.n_items; ++t) {
        const int tg = T + t;
        const int slot = tg & 1;
        const int head = un.b * args.Hq + un.kvh * G + t / un.nqi;
        const int i = un.i0 + t % un.nqi;
        if (!mbar_wait(&bars->st_full[slot][0], (tg >> 1) & 1, st, abort_flag, kSiteStFull) ||
            !mbar_wait(&bars->st_full[slot][1], (tg >> 1) & 1, st, abort_flag, kSiteStFull)) {
          sok = false;
          break;
        }
#pragma unroll
        for (int in_q = 1; in_q >= 0; --in_q) {
#pragma unroll
          for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int q = 0; q < kPasses; ++q)
              if (stage_in_q(g, q) == (in_q != 0))
                tma_reduce_add_3d(&tmDQ, stage_addr(slot, g, q), g * kHalfD + q * 32, i * kT, head);
          bulk_commit_group();
        }
        bulk_wait_read<1>();
        mbar_arrive(&bars->q_empty[slot]);
        bulk_wait_read<0>();
        mbar_arrive(&bars->do_empty[slot]);
      }
      T += un.n_items;
      }
      // The additions must have landed before the kernel is complete.
      bulk_wait_all();
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
// share a row, LSE_i * log2(e), both written padded to ntp rows per head
// (rows past N get D = 0 and +inf), and the dQ accumulator zeroed.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                                const uint4* __restrict__ dO,
                                                                const float* __restrict__ lse,
                                                                float* __restrict__ lse2, float* __restrict__ drow,
                                                                float4* __restrict__ dq_accum, long long heads, int N,
                                                                int ntp) {
  constexpr int kTpr = D / 8;  // threads per row, 16 bytes each
  const long long total = heads * ntp * kTpr;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x; i0 < total; i0 += stride) {
    const long long idx = i0 + threadIdx.x;
    const long long prow = idx / kTpr;             // padded row
    const long long head = prow / ntp;
    const int n = (int)(prow - head * ntp);
    const bool valid = idx < total && n < N;
    const long long row = head * N + n;
    float s = 0.f;
    if (valid) {
      const uint4 a = o[row * kTpr + idx % kTpr];
      const uint4 g = dO[row * kTpr + idx % kTpr];
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
    if (idx < total && (idx % kTpr) == 0) {
      drow[prow] = valid ? s : 0.f;
      lse2[prow] = valid ? lse[row] * kLog2e : INFINITY;
    }
  }
  if (dq_accum == nullptr) return;   // no accumulator (deterministic dQ)
  const long long n4 = heads * N * (D / 4);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += 4 * stride) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * stride < n4) dq_accum[i + u * stride] = z;
  }
}

__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                                uint4* __restrict__ dq, float scale, long long n8) {
  // Four independent 8-element groups per thread and iteration keep more
  // loads in flight (the accumulator is mostly still in L2).
  constexpr int kU = 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8; i0 += kU * stride) {
    float4 a[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        a[u] = acc[2 * i];
        c[u] = acc[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        uint4 w;
        w.x = cvt_bf16x2(a[u].x * scale, a[u].y * scale);
        w.y = cvt_bf16x2(a[u].z * scale, a[u].w * scale);
        w.z = cvt_bf16x2(c[u].x * scale, c[u].y * scale);
        w.w = cvt_bf16x2(c[u].z * scale, c[u].w * scale);
        dq[i] = w;
      }
    }
  }
}

}  // namespace

template <int D, bool kDq>
static cudaError_t configure_dkdv_d() {
  using L = BwdSmem<D>;
  static_assert(L::kBytes <= 232448, "shared memory budget");
  static_assert(sizeof(Bars) <= 256, "barrier block");
  cudaError_t e =
      cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, kDq, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, kDq, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
}

cudaError_t configure_bwd_kernels() {
  cudaError_t e = configure_dkdv_d<64, true>();
  if (e == cudaSuccess) e = configure_dkdv_d<64, false>();
  if (e == cudaSuccess) e = configure_dkdv_d<128, true>();
  if (e == cudaSuccess) e = configure_dkdv_d<128, false>();
  return e;
}

template <int D, bool kDq>
static cudaError_t launch_dkdv_d(const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                                 const TmaMap4& tdo, const TmaMap3& tdq, const BwdArgs& a, const DevStatus& st,
                                 int num_sms, cudaStream_t stream) {
  using L = BwdSmem<D>;
  const long long units = (long long)a.Hkv * a.B * ((a.N + kT - 1) / kT);
  const int grid = (int)(units < num_sms ? units : num_sms);
  if (a.causal)
    fa_bwd_dkdv_kernel<D, kDq, false><<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, tdo, tdq, a, st);
  else
    fa_bwd_dkdv_kernel<D, kDq, true><<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, tdo, tdq, a, st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const TmaMap4& tq, const TmaMap4& tk, const TmaMap4& tv,
                            const TmaMap4& tdo, const TmaMap3& tdq, const BwdArgs& a, const DevStatus& st,
                            int num_sms, cudaStream_t stream) {
  if (a.with_dq) {
    if (d == 64) return launch_dkdv_d<64, true>(tq, tk, tv, tdo, tdq, a, st, num_sms, stream);
    return launch_dkdv_d<128, true>(tq, tk, tv, tdo, tdq, a, st, num_sms, stream);
  }
  if (d == 64) return launch_dkdv_d<64, false>(tq, tk, tv, tdo, tdq, a, st, num_sms, stream);
  return launch_dkdv_d<128, false>(tq, tk, tv, tdo, tdq, a, st, num_sms, stream);
}

static int grid_for(long long work_items, int num_sms) {
  long long blocks = (work_items + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dO, const float* lse, float* lse2, float* drow,
                                  float* dq_accum, long long heads, int N, int num_sms, cudaStream_t stream) {
  const int ntp = (N + kT - 1) / kT * kT;
  const int grid = grid_for(heads * ntp * (d / 8), num_sms);
  if (d == 64)
    fa_bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                           static_cast<const uint4*>(dO), lse, lse2, drow,
                                                           reinterpret_cast<float4*>(dq_accum), heads, N, ntp);
  else
    fa_bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(o),
                                                            static_cast<const uint4*>(dO), lse, lse2, drow,
                                                            reinterpret_cast<float4*>(dq_accum), heads, N, ntp);
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
