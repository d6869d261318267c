// Exact attention forward on sm_103a: O = softmax(scale * Q K^T) V and the
// per-row log-sum-exp, computed tile by tile without any N x N buffer.
//
// Method ([QBank-36] "FlashAttention 为什么常被说成是 IO-aware 优化", part 3;
// [Lecture] "推导 FlashAttention 的在线 softmax"): for one 128-row tile of
// queries, stream 128-key tiles of K and V; for each, form the score tile in
// tensor memory, update a running row max m and running denominator l,
// rescale the running output by exp(m_old - m_new) when the max grows, and
// accumulate P V.  O / l and LSE = m + ln l are written once at the end.
// Multiplying numerator and denominator by one factor leaves their ratio
// unchanged ([Lecture], same section), so the reference max may lag the true
// max: it is only raised when the true max exceeds it by more than 24 (log2
// units).  Every unnormalised probability then stays <= 2^24, a row sum
// <= N * 2^24 and an O entry <= N * 2^24 * max|V| (fp32 holds that for |V|
// up to ~1e24 at N = 8M), and rows whose max keeps climbing, as with large
// score spreads, rescale O in tensor memory only a few times.
//
// Persistent kernel: one CTA per SM walks work items (query tile, head,
// batch), heaviest causal tiles first, dealt to the CTAs in snake order.  CTA layout (384 threads):
//   warp 0      TMA producer for Q (2 slots) and K (ring of kStagesK)
//   warp 1      TMEM allocator; one thread issues the S = Q K^T MMAs
//   warp 2      TMA producer for V (ring of kStagesV)
//   warp 3      one thread issues the O += P V MMAs.  The two issuers touch
//               disjoint tensor memory and each commit tracks only its own
//               MMAs, so each waits only for what its MMAs need.
//   warps 4-7   softmax group 0, warps 8-11 softmax group 1: the groups take
//               alternate score tiles of the CTA's tile sequence (tile t goes
//               to group t % 2); thread r of the owning group handles query
//               row r (TMEM lane r), so row max and row sum are in-thread
//               reductions.  The running reference max is the only state one
//               tile needs from the previous one: the owner of tile t hands it
//               to the owner of tile t+1 through shared memory as soon as it
//               has its row max, then both groups' exponentials overlap.  Each
//               group keeps its own part of the row sum; the two parts are
//               combined in the item's epilogue.
// The control warpgroup (warps 0-3) keeps kCtrlRegs registers a thread and
// hands the rest of the launch allocation to the two softmax warpgroups,
// which hold a 128-column score row in registers.
// Tensor memory (512 columns): two fp32 128x128 score buffers at columns 0
// and 128, two bf16 probability buffers (128 x 128 bf16 = 64 columns) at 256
// and 320, and the O accumulator (fp32 128 x d) at 384.  Tile t uses score
// and probability buffer t % 2, so each softmax group always works on "its"
// buffers.  P V reads P straight from tensor memory (P never touches shared
// memory).  Tensor pipe order:
//   S0 S1 | S2 PV0 | S3 PV1 | S4 PV2 ...
// S_{t+2} is issued as soon as the owner of tile t has loaded S_t into
// registers; P_t is written once P V_{t-2} has consumed the buffer; neither
// waits for the tensor pipe to drain.
#include "fa_internal.h"
#include "sm103a.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // keys per tile
constexpr int kSBuf = 2;        // score buffers (and probability buffers) in tensor memory
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;                 // 65536 / 384, rounded down to the allocation unit of 8
constexpr int kCtrlRegs = 56;
constexpr int kSoftmaxRegs = (kLaunchRegs * 3 - kCtrlRegs) / 2;   // 224: the shares add up to the launch allocation
static_assert(kSoftmaxRegs % 8 == 0 && kSoftmaxRegs <= 256, "register split");
constexpr uint32_t kBlockBytes = 128u * 128u;   // one 64-column block of a 128-row bf16 tile
constexpr float kRescaleThreshold = 24.0f;   // log2 units; see the header

template <int D>
struct FwdCfg {
  static constexpr int kStagesK = D == 128 ? 3 : 4;
  static constexpr int kStagesV = D == 128 ? 2 : 4;
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;                              // 2 slots
  static constexpr uint32_t kK = kQ + 2u * kTile;
  static constexpr uint32_t kV = kK + kStagesK * kTile;
  static constexpr uint32_t kMref = kV + kStagesV * kTile;     // reference-max hand-off, 128 fp32
  // Row-sum hand-off, 2 x 128 entries: float2 (sum, correction), or, with
  // one O accumulator per softmax group (d = 64), float4 (sum, correction,
  // reference max, unused).
  static constexpr uint32_t kLx = kMref + 512u;
  static constexpr uint32_t kBar = kLx + (D == 64 ? 4096u : 2048u);
  static constexpr uint32_t kBytes = kBar + 512u;
};

// Wait-site ids reported in the status words.
enum : int {
  kSiteQEmpty = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSitePFull, kSiteVFull, kSiteOFree,
  kSiteSFree, kSiteSFull, kSiteORescale, kSiteOLast, kSiteHand, kSiteLx, kSitePPrev, kSiteOStaged,
  // drains on the way out
  kDrainQ = 21, kDrainK, kDrainV, kDrainS, kDrainPV
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[kSBuf], s_free[kSBuf], p_full[kSBuf];
  uint64_t o_done[2];
  uint64_t o_free;
  uint64_t hand[2];         // reference max of tile t published (by tile parity)
  uint64_t lx[2];           // row-sum part of the non-owner group published (by multi-tile item parity)
  uint64_t drain_s, drain_pv;
  uint64_t o_staged[2];     // per Q slot: the finished item's O is staged in the slot (plain instance)
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int b, h, kvh;     // batch, first query head of the tile, kv head
  int qrow;          // Q map row (within batch b) of tile row 0: h * Nq + first query index
  long long row0;    // flattened [B*Hq*Nq] row of tile row 0
  int rows;          // tile rows that are real query rows
  int qbase;         // query index of tile row 0 (per-head tiles), 0 when packed
  int qmin, qmax;    // smallest / largest query position in the tile
  int j0, n;         // key tiles [j0, j0 + n)
  int split;
};

// A query tile is 128 consecutive query rows of one head, or, when packed,
// the rows of all Hq/Hkv heads of one kv group (G * Nq <= 128 rows), so that
// the group reads each K / V tile once.  Query row i stands at key position
// i + Nk - Nq.  Work items are ordered heaviest first: rank r covers query
// tile nqt-1-r of every unit when causal (tile r otherwise), each split of it
// in turn.  An item may own no key tile (a split outside the tile's visible
// range); every role skips such items.
// kGeneral = false compiles the plain self-attention case only (Nq == Nk, no
// window, one split, per-head tiles), so the common path carries none of the
// general path's code.
template <bool kGeneral>
__device__ __forceinline__ Item decode_item(int idx, const FwdArgs& a) {
  const int splits = kGeneral ? a.splits : 1;
  const int rs = idx / a.units;
  const int u = idx - rs * a.units;
  const int rank = rs / splits;
  Item it;
  it.split = rs - rank * splits;
  const int qt = a.causal ? a.nqt - 1 - rank : rank;
  const int G = a.Hq / a.Hkv;
  const int off = kGeneral ? a.Nk - a.Nq : 0;
  if (kGeneral && a.packed) {
    it.kvh = u % a.Hkv;
    it.b = u / a.Hkv;
    it.h = it.kvh * G;
    it.qbase = 0;
    it.rows = G * a.Nq;
    it.qmin = off;
    it.qmax = a.Nq - 1 + off;
  } else {
    it.h = u % a.Hq;
    it.b = u / a.Hq;
    it.kvh = it.h / G;
    it.qbase = qt * kBM;
    it.rows = min(kBM, a.Nq - it.qbase);
    it.qmin = it.qbase + off;
    it.qmax = it.qbase + it.rows - 1 + off;
  }
  it.qrow = it.h * a.Nq + it.qbase;
  it.row0 = (long long)it.b * a.Hq * a.Nq + it.qrow;
  const int ntk = (a.Nk + kBN - 1) / kBN;
  int hi = a.causal ? min(ntk, it.qmax / kBN + 1) : ntk;
  int lo = (kGeneral && a.window > 0) ? max(0, it.qmin - a.window + 1) / kBN : 0;
  if (kGeneral && a.splits > 1) {
    lo = max(lo, it.split * a.split_tiles);
    hi = min(hi, (it.split + 1) * a.split_tiles);
  }
  it.j0 = lo;
  it.n = max(0, hi - lo);
  return it;
}

// Item of this CTA in round k: rounds alternate direction over the CTAs, so
// the CTA that drew a heavy item in one round draws a light one in the next
// (with heaviest-first ranks this balances causal work to within a few %).
__device__ __forceinline__ int item_of_round(int k) {
  const int g = gridDim.x;
  return k * g + ((k & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Walks this CTA's (item, key tile) sequence over the items that own key
// tiles; li counts those items.
template <bool kGeneral>
struct Cursor {
  int item, round, li, j, n_items;
  Item it;
  bool valid;
  __device__ __forceinline__ void seek(const FwdArgs& a) {
    for (;;) {
      item = item_of_round(round);
      valid = item < n_items;
      if (!valid) return;
      it = decode_item<kGeneral>(item, a);
      if (it.n > 0) return;
      ++round;
    }
  }
  __device__ __forceinline__ void init(const FwdArgs& a, int n_items_) {
    n_items = n_items_;
    round = 0;
    li = 0;
    j = 0;
    seek(a);
  }
  __device__ __forceinline__ void next(const FwdArgs& a) {
    if (++j == it.n) {
      j = 0;
      ++li;
      ++round;
      seek(a);
    }
  }
};

template <int D, bool kGeneral>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ TmaMap3 tmQ, const __grid_constant__ TmaMap4 tmK,
                  const __grid_constant__ TmaMap4 tmV, const __grid_constant__ TmaMap4 tmO, const FwdArgs args,
                  const DevStatus st) {
  using L = FwdCfg<D>;
  constexpr int kAtoms = D / 64;
  constexpr int SK = L::kStagesK, SV = L::kStagesV;
  // The MMA issuers run as one lane each (a whole-warp issuer, see
  // issuer_wait, spills in the 56-register control warpgroup).
  constexpr bool kWarpIssue = false;
  // d = 64: each softmax group accumulates its own tiles into its own O
  // (64 columns each, at 384 and 448) relative to its own reference max, so
  // a tile never waits for the other group's max; the item's epilogue
  // combines the two (O = O_0 2^(m_0 - m) + O_1 2^(m_1 - m), likewise the
  // row sums, m = max(m_0, m_1)).  d = 128 has no tensor memory for a second
  // O: one shared O and the reference max handed from tile to tile.
  constexpr bool kIndep = D == 64;
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort;
  // The swizzled operand tiles need a 1024-byte aligned base.  The dynamic
  // shared memory of a kernel without static shared memory starts there; if
  // it ever did not, stop cleanly with an error instead of computing garbage.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(st, kErrDeviceTimeout, 0);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nk = args.Nk;
  const int n_items = args.nqt * args.splits * args.units;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);   // last S of the item done (general instance)
      mbar_init(&bars->o_done[i], 1);
      mbar_init(&bars->hand[i], 128);
      mbar_init(&bars->lx[i], 128);
    }
    for (int s = 0; s < SK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < kSBuf; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 128);
      mbar_init(&bars->p_full[s], 128);
    }
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain_s, 1);
    mbar_init(&bars->drain_pv, 1);
    for (int x = 0; x < 2; ++x) mbar_init(&bars->o_staged[x], 128);
    bars->abort = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (!kGeneral) tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tO = tmem + 384;

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);

  if (warp < 4) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0) {
      // ------------------------------------------------------ Q / K producer
      if (lane == 0) {
        int kt = 0, li = 0;
        int q_issued[2] = {0, 0};
        int o_qbase[2] = {0, 0}, o_h[2] = {0, 0}, o_b[2] = {0, 0};   // O tile of the item in each Q slot
        // Plain instance: the softmax group that finishes item k stages its O
        // in the item's Q slot; this thread writes it out with TMA stores and
        // reloads the slot once they have read it, so that the softmax warps
        // never wait for the store.
        auto store_o = [&](int k) -> bool {
          const int sl = k & 1;
          if (!mbar_wait(&bars->o_staged[sl], (k >> 1) & 1, st, abort_flag, kSiteOStaged)) return false;
          for (int a = 0; a < kAtoms; ++a)
            tma_store_4d(&tmO, sQ + sl * L::kTile + a * kBlockBytes, a * 64, o_qbase[sl], o_h[sl], o_b[sl]);
          bulk_commit_group();
          bulk_wait_read<0>();
          return true;
        };
        bool ok = true;
        for (int round = 0, item = item_of_round(0); ok && item < n_items; item = item_of_round(++round)) {
          const Item it = decode_item<kGeneral>(item, args);
          if (it.n == 0) continue;
          const int slot = li & 1;
          if (li >= 2) {
            if constexpr (kGeneral) {
              if (!mbar_wait(&bars->q_empty[slot], ((li >> 1) - 1) & 1, st, abort_flag, kSiteQEmpty)) { ok = false; break; }
            } else {
              if (!store_o(li - 2)) { ok = false; break; }
            }
          }
          o_qbase[slot] = it.qbase;
          o_h[slot] = it.h;
          o_b[slot] = it.b;
          mbar_arrive_expect_tx(&bars->q_full[slot], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(smem + L::kQ + slot * L::kTile + a * kBlockBytes, &tmQ, &bars->q_full[slot], a * 64,
                        it.qrow, it.b);
          ++q_issued[slot];
          for (int j = 0; j < it.n; ++j, ++kt) {
            const int s = kt % SK, r = kt / SK;
            if (r > 0 && !mbar_wait(&bars->k_empty[s], (r - 1) & 1, st, abort_flag, kSiteKEmpty)) { ok = false; break; }
            mbar_arrive_expect_tx(&bars->k_full[s], L::kTile);
            for (int a = 0; a < kAtoms; ++a)
              tma_load_4d(smem + L::kK + s * L::kTile + a * kBlockBytes, &tmK, &bars->k_full[s], a * 64,
                          (it.j0 + j) * kBN, it.kvh, it.b);
          }
          ++li;   // items with key tiles, in the order the MMA issuers' cursors count them
        }
        if constexpr (!kGeneral) {
          // The last two items' O, then every store complete before the CTA exits.
          for (int k = li >= 2 ? li - 2 : 0; ok && k < li; ++k) ok = store_o(k);
          bulk_wait_all();
        }
        // Every copy issued must have landed before the CTA may exit.
        for (int i = 0; i < 2; ++i)
          if (q_issued[i]) mbar_wait_drain(&bars->q_full[i], (q_issued[i] - 1) & 1, st, kDrainQ);
        for (int s = 0; s < SK && s < kt; ++s) {
          const int last = kt - 1 - ((kt - 1 - s) % SK);   // last tile issued into stage s
          mbar_wait_drain(&bars->k_full[s], (last / SK) & 1, st, kDrainK);
        }
      }
    } else if (warp == 2) {
      // ------------------------------------------------------ V producer
      if (lane == 0) {
        int vt = 0;
        bool ok = true;
        for (int round = 0, item = item_of_round(0); ok && item < n_items; item = item_of_round(++round)) {
          const Item it = decode_item<kGeneral>(item, args);
          for (int j = 0; j < it.n; ++j, ++vt) {
            const int s = vt % SV, r = vt / SV;
            if (r > 0 && !mbar_wait(&bars->v_empty[s], (r - 1) & 1, st, abort_flag, kSiteVEmpty)) { ok = false; break; }
            mbar_arrive_expect_tx(&bars->v_full[s], L::kTile);
            for (int a = 0; a < kAtoms; ++a)
              tma_load_4d(smem + L::kV + s * L::kTile + a * kBlockBytes, &tmV, &bars->v_full[s], a * 64,
                          (it.j0 + j) * kBN, it.kvh, it.b);
          }
        }
        for (int s = 0; s < SV && s < vt; ++s) {
          const int last = vt - 1 - ((vt - 1 - s) % SV);
          mbar_wait_drain(&bars->v_full[s], (last / SV) & 1, st, kDrainV);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------ S issuer
      if (kWarpIssue || lane == 0) {
        constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
        // Operand descriptors, built once: a K stage or a k16 step adds a constant.
        const uint64_t dQ0 = desc_kmajor(sQ, 0, kBlockBytes), dQ1 = desc_kmajor(sQ + L::kTile, 0, kBlockBytes);
        const uint64_t dK0 = desc_kmajor(sK, 0, kBlockBytes);
        Cursor<kGeneral> sc;
        sc.init(args, n_items);
        for (int ts = 0; sc.valid; ++ts, sc.next(args)) {
          const int buf = ts % kSBuf;
          // S_ts reuses score buffer ts % 2 once the owner of tile ts-2 has read it.
          if (ts >= 2 && !issuer_wait<kWarpIssue>(&bars->s_free[buf], ((ts - 2) / kSBuf) & 1, st, abort_flag, kSiteSFree)) break;
          if (sc.j == 0 &&
              !issuer_wait<kWarpIssue>(&bars->q_full[sc.li & 1], (sc.li >> 1) & 1, st, abort_flag, kSiteQFull))
            break;
          const int s = ts % SK;
          if (!issuer_wait<kWarpIssue>(&bars->k_full[s], (ts / SK) & 1, st, abort_flag, kSiteKFull)) break;
          tc_fence_after();
          const uint64_t dq = (sc.li & 1) ? dQ1 : dQ0;
          const uint64_t dk = dK0 + (uint64_t)s * (L::kTile >> 4);
#pragma unroll
          for (int k16 = 0; k16 < D / 16; ++k16)
            issue_ss<kWarpIssue>(tmem + buf * 128, dq + desc_step_kmajor(k16, kBlockBytes), dk + desc_step_kmajor(k16, kBlockBytes),
                        idS, k16 > 0);
          issue_commit<kWarpIssue>(&bars->s_full[buf]);
          issue_commit<kWarpIssue>(&bars->k_empty[s]);
          if (sc.j == sc.it.n - 1) issue_commit<kWarpIssue>(&bars->q_empty[sc.li & 1]);
        }
        // No MMA may still be writing tensor memory when it is freed.
        issue_commit<kWarpIssue>(&bars->drain_s);
        mbar_wait_drain(&bars->drain_s, 0, st, kDrainS);
      }
    } else if (warp == 3) {
      // ------------------------------------------------------ P V issuer
      if (kWarpIssue || lane == 0) {
        constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
        const uint64_t dV0 = desc_mnmajor(sV, 0, kBlockBytes);
        Cursor<kGeneral> pc;
        pc.init(args, n_items);
        for (int t = 0; pc.valid; ++t, pc.next(args)) {
          const int buf = t % kSBuf;
          if (!issuer_wait<kWarpIssue>(&bars->p_full[buf], (t / kSBuf) & 1, st, abort_flag, kSitePFull)) break;
          const int v = t % SV;
          if (!issuer_wait<kWarpIssue>(&bars->v_full[v], (t / SV) & 1, st, abort_flag, kSiteVFull)) break;
          if (pc.j == 0 && pc.li > 0 && !issuer_wait<kWarpIssue>(&bars->o_free, (pc.li - 1) & 1, st, abort_flag, kSiteOFree)) break;
          tc_fence_after();
          const uint64_t dv = dV0 + (uint64_t)v * (L::kTile >> 4);
#pragma unroll
          for (int k16 = 0; k16 < kBN / 16; ++k16)
            issue_ts<kWarpIssue>(tO + (kIndep ? (uint32_t)(t & 1) * 64u : 0u), tmem + 256 + buf * 64 + k16 * 8,
                                 dv + desc_step_mnmajor(k16), idO,
                                 (pc.j >= (kIndep ? 2 : 1) || k16 > 0) ? 1u : 0u);
          issue_commit<kWarpIssue>(&bars->o_done[t & 1]);
          issue_commit<kWarpIssue>(&bars->v_empty[v]);
        }
        issue_commit<kWarpIssue>(&bars->drain_pv);
        mbar_wait_drain(&bars->drain_pv, 0, st, kDrainPV);
      }
    }
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------ softmax
    const int g = (warp - 4) >> 2;               // softmax group 0 or 1: owns tiles t with t % 2 == g
    const int quad = warp & 3;
    const int r = quad * 32 + lane;              // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // One slot per row is enough for the reference max: the owner of tile t+1
    // reads it before it writes its own and only then arrives on the hand
    // barrier the owner of tile t+2 waits for.
    float* mref = reinterpret_cast<float*>(smem + L::kMref);   // [row]
    float2* lxb = reinterpret_cast<float2*>(smem + L::kLx);    // [item parity][row]
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    const uint32_t tOg = kIndep ? tO + (uint32_t)g * 64u : tO;          // this group's O
    const uint32_t tOo = kIndep ? tO + (uint32_t)(1 - g) * 64u : tO;    // the other group's
    float m_g = -INFINITY;                       // reference max this group's row sum is relative to
    float l_g = 0.f;                             // this group's part of the row sum
    // The P V product applies each probability rounded to bf16.  A row's
    // largest probability in a tile is 2^lag with a non-integer lag whenever
    // the reference max lags the row's max, so its rounding (relative 2^-9)
    // would not cancel against the row sum; c_g collects, per tile, that one
    // weight's rounding, and O is normalised by l + c (LSE by l).  On rows
    // dominated by one key this keeps O the convex combination the tensor
    // core formed; the other weights' roundings average out.
    float c_g = 0.f;
    int my_item = -1;                            // item the group's (l_g, c_g, m_g) belong to
    int n_multi = 0;                             // items with >= 2 tiles completed so far
    Cursor<kGeneral> c;
    c.init(args, n_items);
    for (int t = 0; c.valid; ++t, c.next(args)) {
      const int j = c.j, n = c.it.n;
      const int n_multi_before = n_multi;
      const int multi_slot = n_multi & 1;
      if (j == n - 1 && n >= 2) ++n_multi;
      if ((t & 1) != g) continue;                // the other group's tile
      const int buf = t % kSBuf;
      // Position of this thread's query among the keys.
      const int qpos = kGeneral ? (args.packed ? r % args.Nq : c.it.qbase + r) + (Nk - args.Nq) : c.it.qbase + r;
      const uint32_t tS = tmem + buf * 128 + lane_off;
      if (!mbar_wait_warp(&bars->s_full[buf], (t / kSBuf) & 1, st, abort_flag, kSiteSFull)) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) reg_fence(sr[q]);
      tc_fence_before();
      mbar_arrive(&bars->s_free[buf]);   // the MMA may compute S_{t+2} into this buffer now

      const int key0 = (c.it.j0 + j) * kBN;
      const bool windowed = kGeneral && args.window > 0;
      if ((key0 + kBN > Nk) || (args.causal && key0 + kBN - 1 > c.it.qmin) ||
          (windowed && key0 < c.it.qmax - args.window + 1)) {
        // Keys [key0 + lo, key0 + hi) are visible to this row.
        const int hi = min(Nk, args.causal ? qpos + 1 : Nk) - key0;
        const int lo = windowed ? qpos - args.window + 1 - key0 : 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (q * 32 + e >= hi || q * 32 + e < lo) sr[q][e] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          mx0 = fmax3(mx0, __uint_as_float(sr[q][e + 0]), __uint_as_float(sr[q][e + 1]));
          mx1 = fmax3(mx1, __uint_as_float(sr[q][e + 2]), __uint_as_float(sr[q][e + 3]));
          mx2 = fmax3(mx2, __uint_as_float(sr[q][e + 4]), __uint_as_float(sr[q][e + 5]));
          mx3 = fmax3(mx3, __uint_as_float(sr[q][e + 6]), __uint_as_float(sr[q][e + 7]));
        }
      }
      const float s_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_cand = s_max * sl2;
      // Reference max after the previous tile (owned by the other group).  The
      // wait also happens at an item's first tile, where the value is unused:
      // it keeps the two groups' hand-offs strictly alternating, so no hand
      // barrier can run two phases ahead of its waiter.
      float m_prev = -INFINITY;
      bool first_g;                              // the group's first tile of the item
      if constexpr (kIndep) {
        first_g = my_item != c.item;
        if (!first_g) m_prev = m_g;
      } else {
        first_g = j == 0;
        if (t > 0) {
          if (!mbar_wait_warp(&bars->hand[(t - 1) & 1], ((t - 1) >> 1) & 1, st, abort_flag, kSiteHand)) break;
          if (j > 0) m_prev = mref[r];
        }
      }
      const bool need = first_g || (m_cand > m_prev + kRescaleThreshold);
      const float m_new = need ? m_cand : m_prev;
      if constexpr (!kIndep) {
        // Hand the reference on to the owner of tile t+1 right away.
        mref[r] = m_new;
        mbar_arrive(&bars->hand[t & 1]);
      }

      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      if (my_item != c.item) {
        my_item = c.item;
        l_g = 0.f;
        c_g = 0.f;
      } else if (m_g != m_new) {
        const float a = ex2(m_g - m_use);
        l_g *= a;
        c_g *= a;
      }
      m_g = m_new;
      {
        // The tile's largest probability exactly as the loop below forms it,
        // and its bf16 rounding error (0 for a row the tile masks entirely).
        const float p_max = ex2(fmaf(s_max, sl2, -m_use));
        c_g += __uint_as_float(cvt_bf16x2(p_max, 0.f) << 16) - p_max;
      }

      // P = 2^(s*sl2 - m), 32 keys at a time, into probability buffer t % 2
      // once P V_{t-2} has consumed it.
      if (t >= 2 && !mbar_wait_warp(&bars->o_done[t & 1], ((t >> 1) - 1) & 1, st, abort_flag, kSitePPrev)) break;
      tc_fence_after();
      const uint32_t tP = tmem + 256 + buf * 64 + lane_off;
      const uint64_t negm = f2pack(-m_use, -m_use);
      uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint64_t x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint64_t sv = f2pack(__uint_as_float(sr[q][e + 2 * u]), __uint_as_float(sr[q][e + 2 * u + 1]));
            float lo, hi;
            f2unpack(ffma2(sv, sl2x2, negm), lo, hi);
            lo = ex2(lo);
            hi = ex2(hi);
            x[u] = f2pack(lo, hi);
            pk[e / 2 + u] = cvt_bf16x2(lo, hi);
          }
          acc0 = fadd2(acc0, x[0]);
          acc1 = fadd2(acc1, x[1]);
          acc2 = fadd2(acc2, x[2]);
          acc3 = fadd2(acc3, x[3]);
        }
        tmem_st16(tP + q * 16, pk);
      }
      float a0, a1;
      f2unpack(fadd2(fadd2(acc0, acc1), fadd2(acc2, acc3)), a0, a1);
      l_g += a0 + a1;

      if (!first_g && __any_sync(0xffffffffu, need)) {
        // O holds rows relative to the previous reference: rescale it once
        // P V of the previous tile has landed (with one O per group, that is
        // the group's own previous tile, already waited for above).
        const float alpha = need ? ex2(m_prev - m_use) : 1.f;
        if constexpr (!kIndep) {
          if (!mbar_wait_warp(&bars->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, st, abort_flag, kSiteORescale)) break;
        }
        tc_fence_after();
        const uint64_t al2 = f2pack(alpha, alpha);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tOg + lane_off + q * 32, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float lo, hi;
            f2unpack(fmul2(f2pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), al2), lo, hi);
            o[e] = __float_as_uint(lo);
            o[e + 1] = __float_as_uint(hi);
          }
          tmem_st32(tOg + lane_off + q * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[buf]);

      if (j == n - 2) {
        // The other group owns the item's last tile: hand it this group's
        // row-sum part and rounding correction, relative to m_new (which it
        // reads back as m_prev).
        if constexpr (kIndep)
          reinterpret_cast<float4*>(lxb)[multi_slot * 128 + r] = make_float4(l_g, c_g, m_g, 0.f);
        else
          lxb[multi_slot * 128 + r] = make_float2(l_g, c_g);
        mbar_arrive(&bars->lx[multi_slot]);
      }
      if (j == n - 1) {
        // ------------------------------------------------ epilogue of the item
        float l_tot = l_g, c_tot = c_g;
        float m_fin = m_new;                   // the reference the totals and O end up relative to
        float a_g = 1.f, a_o = 0.f;            // weights of this group's and the other group's O
        if (n >= 2) {
          if (!mbar_wait_warp(&bars->lx[multi_slot], (n_multi_before >> 1) & 1, st, abort_flag, kSiteLx)) break;
          if constexpr (kIndep) {
            const float4 other = reinterpret_cast<const float4*>(lxb)[multi_slot * 128 + r];
            m_fin = fmaxf(m_new, other.z);
            const float mf = m_fin == -INFINITY ? 0.f : m_fin;
            a_g = ex2(m_new - mf);
            a_o = ex2(other.z - mf);
            l_tot = l_g * a_g + other.x * a_o;
            c_tot = c_g * a_g + other.y * a_o;
          } else {
            const float2 other = lxb[multi_slot * 128 + r];
            const float a = ex2(m_prev - m_use);
            l_tot += other.x * a;
            c_tot += other.y * a;
          }
        }
        const float l_o = l_tot + c_tot;   // sum of the weights P V applied
        // O row of this thread, in the same reference: one accumulator, or
        // this group's and (items of two or more tiles) the other group's.
        auto load_o = [&](int col, uint32_t (&dst)[32]) {
          tmem_ld32(tOg + lane_off + col, dst);
          if constexpr (kIndep) {
            if (n >= 2) {
              uint32_t oo[32];
              tmem_ld32(tOo + lane_off + col, oo);
              tmem_wait_ld();
              reg_fence(dst);
              reg_fence(oo);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                dst[e] = __float_as_uint(__uint_as_float(dst[e]) * a_g + __uint_as_float(oo[e]) * a_o);
            }
          }
        };
        if (!mbar_wait_warp(&bars->o_done[t & 1], (t >> 1) & 1, st, abort_flag, kSiteOLast)) break;
        tc_fence_after();
        const long long frow = c.it.row0 + r;
        if constexpr (!kGeneral) {
          // Plain instance: every thread writes its O row, normalised to
          // bf16, into the item's Q slot (free: the item's last S has
          // completed), 128-byte swizzled like the tensor map's box, 64
          // columns at a time; the Q / K producer then writes the tile with
          // TMA stores (rows past N are clipped) before it reloads the slot.
          // The group neither stores rows nor waits for the store.
          const float inv_l = 1.f / l_o;
          const uint32_t stage = smem_u32(smem + L::kQ) + (c.li & 1) * L::kTile;
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            uint32_t o[2][32];
            load_o(a * 64, o[0]);
            load_o(a * 64 + 32, o[1]);
            tmem_wait_ld();
            reg_fence(o[0]);
            reg_fence(o[1]);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const uint32_t w0 = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 0]) * inv_l, __uint_as_float(o[q][v * 8 + 1]) * inv_l);
                const uint32_t w1 = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 2]) * inv_l, __uint_as_float(o[q][v * 8 + 3]) * inv_l);
                const uint32_t w2 = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 4]) * inv_l, __uint_as_float(o[q][v * 8 + 5]) * inv_l);
                const uint32_t w3 = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 6]) * inv_l, __uint_as_float(o[q][v * 8 + 7]) * inv_l);
                // Columns a*64 + q*32 + v*8 .. +7: block a, 16-byte chunk q*4 + v.
                st_shared_v4(stage + a * kBlockBytes + swz128(r, q * 4 + v), w0, w1, w2, w3);
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&bars->o_free);   // the next item's first P V may overwrite O now
          if (r < c.it.rows) args.lse[frow] = (m_fin + __log2f(l_tot)) * 0.69314718055994530942f;
          fence_proxy_async_smem();
          mbar_arrive(&bars->o_staged[c.li & 1]);   // the Q / K producer stores it
        } else {
          uint32_t o[D / 32][32];
#pragma unroll
          for (int q = 0; q < D / 32; ++q) load_o(q * 32, o[q]);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < D / 32; ++q) reg_fence(o[q]);
          tc_fence_before();
          mbar_arrive(&bars->o_free);   // the next item's first P V may overwrite O now
          if (r < c.it.rows) {
            if (args.splits == 1) {
              const float inv_l = 1.f / l_o;
              __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(args.o) + frow * D;
#pragma unroll
              for (int q = 0; q < D / 32; ++q) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  uint4 w;
                  w.x = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 0]) * inv_l, __uint_as_float(o[q][v * 8 + 1]) * inv_l);
                  w.y = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 2]) * inv_l, __uint_as_float(o[q][v * 8 + 3]) * inv_l);
                  w.z = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 4]) * inv_l, __uint_as_float(o[q][v * 8 + 5]) * inv_l);
                  w.w = cvt_bf16x2(__uint_as_float(o[q][v * 8 + 6]) * inv_l, __uint_as_float(o[q][v * 8 + 7]) * inv_l);
                  *reinterpret_cast<uint4*>(orow + q * 32 + v * 8) = w;
                }
              }
              args.lse[frow] = (m_fin + __log2f(l_tot)) * 0.69314718055994530942f;
            } else {
              // One key split: O normalised within the split, fp32, and its LSE;
              // a row that sees no key of the split gets O = 0, LSE = -inf.
              const long long prow = (long long)c.it.split * args.B * args.Hq * args.Nq + frow;
              const float inv_l = l_tot > 0.f ? 1.f / l_o : 0.f;
              float4* orow = reinterpret_cast<float4*>(args.o_part + prow * D);
#pragma unroll
              for (int q = 0; q < D / 32; ++q)
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  orow[q * 8 + v] = make_float4(__uint_as_float(o[q][v * 4 + 0]) * inv_l,
                                                __uint_as_float(o[q][v * 4 + 1]) * inv_l,
                                                __uint_as_float(o[q][v * 4 + 2]) * inv_l,
                                                __uint_as_float(o[q][v * 4 + 3]) * inv_l);
              args.lse_part[prow] =
                  l_tot > 0.f ? (m_fin + __log2f(l_tot)) * 0.69314718055994530942f : -INFINITY;
            }
          }
        }
      }
    }
    // A wait that gave up between this tile's probability stores and their
    // wait leaves them in flight: let them land before tensor memory is freed.
    tmem_wait_st();
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

template <int D, bool kGeneral>
static cudaError_t configure_fwd_d() {
  using L = FwdCfg<D>;
  static_assert(L::kBytes <= 232448, "shared memory budget");
  static_assert(sizeof(Bars) <= 512, "barrier block");
  cudaError_t e =
      cudaFuncSetAttribute(fa_fwd_kernel<D, kGeneral>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // The warpgroups' register shares assume this launch allocation; with any
  // other, the softmax warpgroups' increase could never be granted.  The
  // build checks the same count in ptxas's report; this guards a library
  // built some other way.
  cudaFuncAttributes fattr;
  e = cudaFuncGetAttributes(&fattr, fa_fwd_kernel<D, kGeneral>);
  if (e != cudaSuccess) return e;
  return fattr.numRegs == kLaunchRegs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t configure_fwd_kernels() {
  cudaError_t e = configure_fwd_d<64, false>();
  if (e == cudaSuccess) e = configure_fwd_d<64, true>();
  if (e == cudaSuccess) e = configure_fwd_d<128, false>();
  if (e == cudaSuccess) e = configure_fwd_d<128, true>();
  return e;
}

template <int D, bool kGeneral>
static cudaError_t launch_fwd_d(const TmaMap3& tq, const TmaMap4& tk, const TmaMap4& tv,
                                const TmaMap4& to, const FwdArgs& a, const DevStatus& st, int num_sms,
                                cudaStream_t stream) {
  using L = FwdCfg<D>;
  const long long items = (long long)a.nqt * a.splits * a.units;
  const int grid = (int)(items < num_sms ? items : num_sms);
  fa_fwd_kernel<D, kGeneral><<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, to, a, st);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const TmaMap3& tq, const TmaMap4& tk, const TmaMap4& tv,
                       const TmaMap4& to, const FwdArgs& a, const DevStatus& st, int num_sms,
                       cudaStream_t stream) {
  const bool general = a.Nq != a.Nk || a.window > 0 || a.splits > 1 || a.packed;
  if (d == 64)
    return general ? launch_fwd_d<64, true>(tq, tk, tv, to, a, st, num_sms, stream)
                   : launch_fwd_d<64, false>(tq, tk, tv, to, a, st, num_sms, stream);
  return general ? launch_fwd_d<128, true>(tq, tk, tv, to, a, st, num_sms, stream)
                 : launch_fwd_d<128, false>(tq, tk, tv, to, a, st, num_sms, stream);
}

// Merge of the key splits ([Lecture] "推导 FlashAttention 的在线 softmax": both
// parts of a softmax-weighted sum are carried relative to a reference max and
// rescaled by exp(old - new) when the reference changes).  For query row r
// with split results (O_s, LSE_s): m = max_s LSE_s, w_s = exp(LSE_s - m),
// O = sum_s w_s O_s / sum_s w_s, LSE = m + ln sum_s w_s.  Splits that hold no
// key the row may see were either not computed or hold LSE = -inf; both are
// skipped.  One thread per 4 columns of a row.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_merge_kernel(const FwdArgs a) {
  constexpr int kC4 = D / 4;
  const long long R = (long long)a.B * a.Hq * a.Nq;
  const long long total = R * kC4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const long long row = idx / kC4;
    const int c4 = (int)(idx - row * kC4);
    const int qpos = (int)(row % a.Nq) + a.Nk - a.Nq;
    const int klo = a.window > 0 ? max(0, qpos - a.window + 1) : 0;   // visible keys [klo, khi)
    const int khi = a.causal ? min(a.Nk, qpos + 1) : a.Nk;
    const int span = a.split_tiles * kBN;
    const int s0 = klo / span, s1 = (khi - 1) / span;                 // splits holding visible keys
    float m = -INFINITY;
    for (int s = s0; s <= s1; ++s) m = fmaxf(m, a.lse_part[s * R + row]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = s0; s <= s1; ++s) {
      const float ls = a.lse_part[s * R + row];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - m);
      const float4 o = reinterpret_cast<const float4*>(a.o_part + (s * R + row) * D)[c4];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
      den += w;
    }
    const float inv = 1.f / den;
    uint2 out;
    out.x = cvt_bf16x2(acc.x * inv, acc.y * inv);
    out.y = cvt_bf16x2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) + row * D)[c4] = out;
    if (c4 == 0) a.lse[row] = m + __logf(den);
  }
}

cudaError_t launch_fwd_merge(int d, const FwdArgs& a, int num_sms, cudaStream_t stream) {
  const long long total = (long long)a.B * a.Hq * a.Nq * (d / 4);
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)num_sms * 8) blocks = (long long)num_sms * 8;
  if (blocks < 1) blocks = 1;
  if (d == 64)
    fa_fwd_merge_kernel<64><<<(int)blocks, 256, 0, stream>>>(a);
  else
    fa_fwd_merge_kernel<128><<<(int)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
