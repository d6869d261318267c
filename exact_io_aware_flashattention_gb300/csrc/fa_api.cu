// C-ABI layer of libfa_gb300.so: argument validation, TMA tensor maps,
// kernel launches and the device status words.  See include/fa.h for the
// contract of every entry point.
#include "fa.h"

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fa_internal.h"

namespace {

// Most recent CUDA runtime error behind an FA_ERR_LAUNCH / FA_ERR_CUDA return
// on this thread (see fa_last_cuda_error).
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

fa_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = e;
  return FA_ERR_LAUNCH;
}

// Records a failing runtime call and returns FA_ERR_CUDA.
fa_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = e;
  return FA_ERR_CUDA;
}

#define FA_TRY(x)                   \
  do {                              \
    fa_status _s = (x);             \
    if (_s != FA_OK) return _s;     \
  } while (0)

#define FA_TRY_CUDA(x)                                \
  do {                                                \
    const cudaError_t _e = (x);                       \
    if (_e != cudaSuccess) return cuda_status(_e);    \
  } while (0)

// First device-side error: code, block, wait site, thread, and the first
// failed drain (site, block).  Read and cleared by fa_last_device_status.
__device__ int g_status_words[fa::kStatusWords];

// Named range around each public call, for timeline tools (a no-op unless a
// tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

__global__ void wait_selftest_kernel(fa::DevStatus st) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(&bar, 1);
    abort_flag = 0;
    fa::mbar_fence_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up and record
  // FA_ERR_DEVICE_TIMEOUT.
  if (threadIdx.x == 0) fa::mbar_wait(&bar, 0, st, &abort_flag, 99);
  __syncthreads();
}

// The same with the drain wait a kernel does on its way out: nothing ever
// completes `bar`, so the drain gives up and records its site (98).
__global__ void drain_selftest_kernel(fa::DevStatus st) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    fa::mbar_init(&bar, 1);
    fa::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) fa::mbar_wait_drain(&bar, 0, st, 98);
  __syncthreads();
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool unusable = false;   // a kernel's drain gave up: no further launches on this device
  int num_sms = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

unsigned long long default_timeout_ns() {
  static unsigned long long t = [] {
    const char* s = std::getenv("FA_WAIT_TIMEOUT_NS");
    unsigned long long v = s ? std::strtoull(s, nullptr, 10) : 0ull;
    return v ? v : 2000000000ull;  // 2 s: far above any single wait of a correct run
  }();
  return t;
}

// Per-device state, set up once with the device current: its SM count, the
// status words' address, the kernels' shared-memory attributes and the
// forward kernel's register check.  With `launch`, a device on which a drain
// has failed is refused.
fa_status device_state(DeviceState** out, bool launch = true) {
  int dev = -1;
  FA_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (launch && s.unusable) return FA_ERR_DEVICE_DRAIN;
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    FA_TRY_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    FA_TRY_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    FA_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    FA_TRY_CUDA(cudaGetSymbolAddress(&p, g_status_words));
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    {
      const cudaError_t e = fa::configure_kernels();
      if (e != cudaSuccess) return launch_status(e);
    }
    s.num_sms = sms;
    s.status = static_cast<int*>(p);
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

fa::DevStatus dev_status(const DeviceState* s) { return fa::DevStatus{s->status, default_timeout_ns()}; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_shape(int B, int Hq, int Hkv, int N, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return FA_ERR_BAD_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_BAD_SHAPE;
  if (B > 65535 || N > 65535 * 128) return FA_ERR_BAD_SHAPE;
  if ((long long)((N + 127) / 128) * Hq * B >= (1LL << 31)) return FA_ERR_BAD_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_HEADDIM;
  return FA_OK;
}

fa_status check_scale(int causal, float scale) {
  if (causal != 0 && causal != 1) return FA_ERR_BAD_ARGUMENT;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_ARGUMENT;
  return FA_OK;
}

struct Range {
  uintptr_t lo, hi;
};
Range range(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t elems(int B, int H, int N, int d) { return (size_t)B * H * N * d; }

fa_status check_shape_ex(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  FA_TRY(check_shape(B, Hq, Hkv, Nq, d));
  return check_shape(B, Hq, Hkv, Nk, d);
}

// How the forward tiles a problem: per-head 128-row query tiles, or, for few
// query rows (Nq < 128, Hq/Hkv * Nq <= 128, Hq > Hkv), one tile holding the
// rows of all query heads of a kv group; the key tiles split into chunks.
struct FwdGeometry {
  int packed, nqt, units, splits, split_tiles;
};
FwdGeometry fwd_geometry(int B, int Hq, int Hkv, int Nq, int Nk, int num_splits) {
  FwdGeometry g;
  const int G = Hq / Hkv;
  g.packed = (G > 1 && Nq < 128 && G * Nq <= 128) ? 1 : 0;
  g.nqt = g.packed ? 1 : (Nq + 127) / 128;
  g.units = g.packed ? B * Hkv : B * Hq;
  const int ntk = (Nk + 127) / 128;
  g.split_tiles = (ntk + num_splits - 1) / num_splits;
  g.splits = (ntk + g.split_tiles - 1) / g.split_tiles;
  return g;
}

// Split forward workspace: per-split O, fp32 [S, B*Hq*Nq, d], then per-split
// LSE, fp32 [S, B*Hq*Nq], each 256-byte aligned.
struct FwdWsLayout {
  size_t o_off, lse_off, total;
};
FwdWsLayout fwd_ws_layout(int B, int Hq, int Nq, int d, int num_splits) {
  const size_t rows = (size_t)B * Hq * Nq;
  FwdWsLayout w;
  w.o_off = 0;
  w.lse_off = align256((size_t)num_splits * rows * d * 4);
  w.total = w.lse_off + align256((size_t)num_splits * rows * 4);
  return w;
}

// Backward workspace: fp32 dQ accumulator [B,Hq,N,d], then LSE*log2(e) and
// D = rowsum(dO*O), each fp32 [B*Hq, ntp] with ntp = ceil(N/128)*128.
struct WsLayout {
  size_t dq_off, lse2_off, dr_off, total;
};
WsLayout ws_layout(int B, int Hq, int N, int d) {
  const size_t ntp = (size_t)((N + 127) / 128) * 128;
  WsLayout w;
  w.dq_off = 0;
  w.lse2_off = align256(elems(B, Hq, N, d) * 4);
  w.dr_off = w.lse2_off + align256((size_t)B * Hq * ntp * 4);
  w.total = w.dr_off + align256((size_t)B * Hq * ntp * 4);
  return w;
}

// Tensor maps are a pure function of (kind, base address, sizes): a small
// per-thread cache saves re-encoding them when the same buffers come back.
struct TmapKey {
  const void* base;
  int kind, B, H, N, d;
  bool operator==(const TmapKey& o) const {
    return base == o.base && kind == o.kind && B == o.B && H == o.H && N == o.N && d == o.d;
  }
};
struct TmapSlot {
  TmapKey key{nullptr, -1, 0, 0, 0, 0};
  CUtensorMap map;   // the encoded map of either rank
};
constexpr int kTmapSlots = 32;
thread_local TmapSlot t_tmaps[kTmapSlots];

int tmap_slot(const TmapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) >> 8;
  h = h * 0x9E3779B97F4A7C15ull + (uint64_t)k.kind;
  h = h * 0x9E3779B97F4A7C15ull + (uint64_t)(uint32_t)k.N;
  h = h * 0x9E3779B97F4A7C15ull + (uint64_t)(uint32_t)(k.B * 131 + k.H * 7 + k.d);
  return (int)((h >> 40) % kTmapSlots);
}

template <typename Encode>
fa_status cached_tmap(CUtensorMap* m, const TmapKey& key, Encode encode) {
  TmapSlot& slot = t_tmaps[tmap_slot(key)];
  if (slot.key == key) {
    *m = slot.map;
    return FA_OK;
  }
  const fa_status st = encode(m);
  if (st == FA_OK) {
    slot.key = key;
    slot.map = *m;
  }
  return st;
}

fa_status tmap_bf16_encode(CUtensorMap* m, const void* base, int B, int H, int N, int d) {  // rank 4
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2, (cuuint64_t)H * N * d * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_LAUNCH;
}

// Q (or O) [B, Hq, Nq, d] viewed as {d, Hq*Nq, B}: a 128-row box may start at
// any row of a batch (a tile of one head, or the rows of a group of heads).
fa_status tmap_rows_bf16_encode(CUtensorMap* m, const void* base, int B, int H, int N, int d) {  // rank 3
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H * N, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * N * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_LAUNCH;
}

// fp32 dQ accumulator [B*Hq, N, d] viewed as {d, N, B*Hq} with a {32, 128, 1}
// box and 128-byte swizzle, the target of the tiled TMA reduce-add.
fa_status tmap_dq_accum_encode(CUtensorMap* m, void* base, int B, int Hq, int N, int d) {  // rank 3
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)B * Hq};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_LAUNCH;
}

// [B, H, N, d] bf16 as {d, N, H, B}, {64, 128, 1, 1} boxes.
fa_status tmap_bf16(fa::TmaMap4* m, const void* base, int B, int H, int N, int d) {
  return cached_tmap(&m->m, TmapKey{base, 0, B, H, N, d},
                     [&](CUtensorMap* x) { return tmap_bf16_encode(x, base, B, H, N, d); });
}
fa_status tmap_rows_bf16(fa::TmaMap3* m, const void* base, int B, int H, int N, int d) {
  return cached_tmap(&m->m, TmapKey{base, 1, B, H, N, d},
                     [&](CUtensorMap* x) { return tmap_rows_bf16_encode(x, base, B, H, N, d); });
}
fa_status tmap_dq_accum(fa::TmaMap3* m, void* base, int B, int Hq, int N, int d) {
  return cached_tmap(&m->m, TmapKey{base, 2, B, Hq, N, d},
                     [&](CUtensorMap* x) { return tmap_dq_accum_encode(x, base, B, Hq, N, d); });
}

fa_status validate_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B,
                        int Hq, int Hkv, int N, int d, int causal, float scale, const void* workspace,
                        size_t workspace_bytes) {
  if (!q || !k || !v || !dO || !dk || !dv || !workspace) return FA_ERR_NULL_PTR;
  FA_TRY(check_shape(B, Hq, Hkv, N, d));
  FA_TRY(check_scale(causal, scale));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return FA_ERR_MISALIGNED;
  if (workspace_bytes < ws_layout(B, Hq, N, d).total) return FA_ERR_WORKSPACE_TOO_SMALL;
  const size_t qb = elems(B, Hq, N, d) * 2, kb = elems(B, Hkv, N, d) * 2;
  const Range ins[] = {range(q, qb), range(k, kb), range(v, kb), range(dO, qb)};
  const Range outs[] = {range(dk, kb), range(dv, kb), range(workspace, ws_layout(B, Hq, N, d).total)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return FA_ERR_ALIASING;
  if (overlap(outs[0], outs[1]) || overlap(outs[0], outs[2]) || overlap(outs[1], outs[2])) return FA_ERR_ALIASING;
  return FA_OK;
}

fa_status dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B, int Hq, int Hkv,
               int N, int d, int causal, int window, int with_dq, float scale, void* workspace,
               size_t workspace_bytes, void* stream) {
  FA_TRY(validate_dkdv(q, k, v, dO, dk, dv, B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes));
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  fa::TmaMap4 tq, tk, tv, tdo;
  fa::TmaMap3 tdq;
  const WsLayout w = ws_layout(B, Hq, N, d);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FA_TRY(tmap_bf16(&tq, q, B, Hq, N, d));
  FA_TRY(tmap_bf16(&tk, k, B, Hkv, N, d));
  FA_TRY(tmap_bf16(&tv, v, B, Hkv, N, d));
  FA_TRY(tmap_bf16(&tdo, dO, B, Hq, N, d));
  FA_TRY(tmap_dq_accum(&tdq, ws + w.dq_off, B, Hq, N, d));
  fa::BwdArgs a;
  a.lse2 = reinterpret_cast<const float*>(ws + w.lse2_off);
  a.drow = reinterpret_cast<const float*>(ws + w.dr_off);
  a.dq_accum = reinterpret_cast<float*>(ws + w.dq_off);
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.causal = causal;
  a.window = window;
  a.with_dq = with_dq;
  a.v8 = ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31u) == 0;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_status(
      fa::launch_bwd_dkdv(d, tq, tk, tv, tdo, tdq, a, dev_status(ds), ds->num_sms, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int fa_version(void) { return 101; }

const char* fa_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* fa_strerror(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_NULL_PTR: return "a required pointer is NULL";
    case FA_ERR_BAD_SHAPE:
      return "bad shape (B, Hq, Hkv, N must be >= 1, Hq % Hkv == 0, B <= 65535, N <= 8388480, "
             "ceil(N/128)*Hq*B < 2^31)";
    case FA_ERR_UNSUPPORTED_HEADDIM: return "unsupported head dimension (d must be 64 or 128)";
    case FA_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case FA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than fa_bwd_workspace_bytes()";
    case FA_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case FA_ERR_LAUNCH: return "kernel launch or tensor-map encoding failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait ran out";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_BAD_ARGUMENT: return "bad argument (scale must be finite and > 0, causal 0 or 1)";
    case FA_ERR_ALIASING: return "an output overlaps an input or another output";
    case FA_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than fa_bwd_noalloc's built-in buffer (FA_NOALLOC_SCRATCH_BYTES) holds";
    case FA_ERR_DEVICE_DRAIN:
      return "a kernel exited with its own copies or MMAs possibly in flight after a device-side timeout; "
             "no further launches on this device in this process";
  }
  return "unknown status";
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_shape(B, Hq, Hkv, N, d) != FA_OK) return 0;
  return ws_layout(B, Hq, N, d).total;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                 int d, int causal, float scale, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, N, N, d, causal, 0, 1, scale, nullptr, 0, stream);
}

size_t fa_fwd_ex_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits) {
  if (check_shape_ex(B, Hq, Hkv, Nq, Nk, d) != FA_OK || num_splits < 1) return 0;
  if (num_splits == 1) return 0;
  return fwd_ws_layout(B, Hq, Nq, d, num_splits).total;
}

int fa_fwd_ex_default_splits(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window) {
  if (check_shape_ex(B, Hq, Hkv, Nq, Nk, d) != FA_OK) return 1;
  DeviceState* ds = nullptr;
  if (device_state(&ds) != FA_OK) return 1;
  const FwdGeometry g = fwd_geometry(B, Hq, Hkv, Nq, Nk, 1);
  const long long units = (long long)g.units * g.nqt;
  int ntk = (Nk + 127) / 128;
  if (causal && window > 0) ntk = std::min(ntk, (window + 127) / 128 + 1);
  // Key tiles on the busiest SM, counting each item's fixed cost (its Q
  // load, pipeline fill and epilogue) as about two key tiles.
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= std::min(64, ntk); ++s) {
    const long long rounds = (units * s + ds->num_sms - 1) / ds->num_sms;
    const long long cost = rounds * ((ntk + s - 1) / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int causal, int window, int num_splits, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  NvtxRange nv("fa_fwd_ex");
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_PTR;
  FA_TRY(check_shape_ex(B, Hq, Hkv, Nq, Nk, d));
  FA_TRY(check_scale(causal, scale));
  if (window < 0 || (window > 0 && !causal) || (causal && Nq > Nk) || num_splits < 1 || num_splits > 4096)
    return FA_ERR_BAD_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  const FwdGeometry g = fwd_geometry(B, Hq, Hkv, Nq, Nk, num_splits);
  if ((long long)g.nqt * g.splits * g.units >= (1LL << 31)) return FA_ERR_BAD_SHAPE;
  const size_t qb = elems(B, Hq, Nq, d) * 2, kb = elems(B, Hkv, Nk, d) * 2;
  const Range ins[] = {range(q, qb), range(k, kb), range(v, kb)};
  const Range ro = range(o, qb), rl = range(lse, (size_t)B * Hq * Nq * 4);
  for (const Range& i : ins)
    if (overlap(ro, i) || overlap(rl, i)) return FA_ERR_ALIASING;
  if (overlap(ro, rl)) return FA_ERR_ALIASING;
  FwdWsLayout w{};
  if (g.splits > 1) {
    w = fwd_ws_layout(B, Hq, Nq, d, num_splits);
    if (!workspace) return FA_ERR_NULL_PTR;
    if (!aligned16(workspace)) return FA_ERR_MISALIGNED;
    if (workspace_bytes < w.total) return FA_ERR_WORKSPACE_TOO_SMALL;
    const Range rw = range(workspace, w.total);
    for (const Range& i : ins)
      if (overlap(rw, i)) return FA_ERR_ALIASING;
    if (overlap(rw, ro) || overlap(rw, rl)) return FA_ERR_ALIASING;
  }

  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  fa::TmaMap3 tq;
  fa::TmaMap4 tk, tv, to;
  FA_TRY(tmap_rows_bf16(&tq, q, B, Hq, Nq, d));
  FA_TRY(tmap_bf16(&tk, k, B, Hkv, Nk, d));
  FA_TRY(tmap_bf16(&tv, v, B, Hkv, Nk, d));
  FA_TRY(tmap_bf16(&to, o, B, Hq, Nq, d));
  fa::FwdArgs a;
  a.o = o;
  a.lse = lse;
  a.o_part = g.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.o_off) : nullptr;
  a.lse_part = g.splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.lse_off) : nullptr;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.causal = causal;
  a.window = window;
  a.packed = g.packed;
  a.nqt = g.nqt;
  a.units = g.units;
  a.splits = g.splits;
  a.split_tiles = g.split_tiles;
  a.scale_log2 = scale * 1.4426950408889634f;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  FA_TRY(launch_status(fa::launch_fwd(d, tq, tk, tv, to, a, dev_status(ds), ds->num_sms, st)));
  if (g.splits > 1) FA_TRY(launch_status(fa::launch_fwd_merge(d, a, ds->num_sms, st)));
  return FA_OK;
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int Hq, int Hkv, int N, int d,
                            void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nv("fa_bwd_preprocess");
  if (!o || !dO || !lse || !workspace) return FA_ERR_NULL_PTR;
  FA_TRY(check_shape(B, Hq, Hkv, N, d));
  if (!aligned16(o) || !aligned16(dO) || !aligned16(lse) || !aligned16(workspace)) return FA_ERR_MISALIGNED;
  const WsLayout w = ws_layout(B, Hq, N, d);
  if (workspace_bytes < w.total) return FA_ERR_WORKSPACE_TOO_SMALL;
  const size_t qb = elems(B, Hq, N, d) * 2;
  const Range rw = range(workspace, w.total);
  if (overlap(rw, range(o, qb)) || overlap(rw, range(dO, qb)) || overlap(rw, range(lse, (size_t)B * Hq * N * 4)))
    return FA_ERR_ALIASING;
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return launch_status(fa::launch_bwd_preprocess(
      d, o, dO, lse, reinterpret_cast<float*>(ws + w.lse2_off), reinterpret_cast<float*>(ws + w.dr_off),
      reinterpret_cast<float*>(ws + w.dq_off), (long long)B * Hq, N, ds->num_sms, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B, int Hq,
                      int Hkv, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  NvtxRange nv("fa_bwd_dkdv");
  return dkdv(q, k, v, dO, dk, dv, B, Hq, Hkv, N, d, causal, 0, 1, scale, workspace, workspace_bytes, stream);
}



fa_status fa_bwd_dq_convert(void* dq, int B, int Hq, int Hkv, int N, int d, float scale, const void* workspace,
                            size_t workspace_bytes, void* stream) {
  NvtxRange nv("fa_bwd_dq_convert");
  if (!dq || !workspace) return FA_ERR_NULL_PTR;
  FA_TRY(check_shape(B, Hq, Hkv, N, d));
  FA_TRY(check_scale(0, scale));
  if (!aligned16(dq) || !aligned16(workspace)) return FA_ERR_MISALIGNED;
  const WsLayout w = ws_layout(B, Hq, N, d);
  if (workspace_bytes < w.total) return FA_ERR_WORKSPACE_TOO_SMALL;
  if (overlap(range(dq, elems(B, Hq, N, d) * 2), range(workspace, w.total))) return FA_ERR_ALIASING;
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  return launch_status(fa::launch_bwd_dq_convert(reinterpret_cast<const float*>(ws + w.dq_off), dq, scale,
                                                 (long long)elems(B, Hq, N, d), ds->num_sms,
                                                 static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, 0, 0, scale, workspace,
                   workspace_bytes, stream);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                    int deterministic, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nv("fa_bwd_ex");
  if (!o || !dq || !lse) return FA_ERR_NULL_PTR;
  if (window < 0 || (window > 0 && !causal) || (deterministic != 0 && deterministic != 1)) return FA_ERR_BAD_ARGUMENT;
  FA_TRY(validate_dkdv(q, k, v, dO, dk, dv, B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes));
  if (!aligned16(o) || !aligned16(dq) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  const size_t qb = elems(B, Hq, N, d) * 2, kb = elems(B, Hkv, N, d) * 2;
  const Range rdq = range(dq, qb);
  const Range others[] = {range(q, qb),  range(k, kb),  range(v, kb),  range(o, qb), range(dO, qb),
                          range(lse, (size_t)B * Hq * N * 4), range(dk, kb), range(dv, kb),
                          range(workspace, ws_layout(B, Hq, N, d).total)};
  for (const Range& r : others)
    if (overlap(rdq, r)) return FA_ERR_ALIASING;
  const Range ro = range(o, qb);
  const Range rl = range(lse, (size_t)B * Hq * N * 4), rw = range(workspace, ws_layout(B, Hq, N, d).total);
  if (overlap(ro, range(dk, kb)) || overlap(ro, range(dv, kb)) || overlap(ro, rw)) return FA_ERR_ALIASING;
  if (overlap(rl, range(dk, kb)) || overlap(rl, range(dv, kb)) || overlap(rl, rw)) return FA_ERR_ALIASING;
  if (!deterministic) {
    FA_TRY(fa_bwd_preprocess(o, dO, lse, B, Hq, Hkv, N, d, workspace, workspace_bytes, stream));
    FA_TRY(dkdv(q, k, v, dO, dk, dv, B, Hq, Hkv, N, d, causal, window, 1, scale, workspace, workspace_bytes, stream));
    return fa_bwd_dq_convert(dq, B, Hq, Hkv, N, d, scale, workspace, workspace_bytes, stream);
  }
  // Deterministic: LSE*log2(e) and D only (no accumulator), dK/dV without
  // dQ partials, then dQ per query tile in a fixed order.
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  const WsLayout w = ws_layout(B, Hq, N, d);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  FA_TRY(launch_status(fa::launch_bwd_preprocess(d, o, dO, lse, reinterpret_cast<float*>(ws + w.lse2_off),
                                                 reinterpret_cast<float*>(ws + w.dr_off), nullptr, (long long)B * Hq,
                                                 N, ds->num_sms, st)));
  FA_TRY(dkdv(q, k, v, dO, dk, dv, B, Hq, Hkv, N, d, causal, window, 0, scale, workspace, workspace_bytes, stream));
  fa::TmaMap4 tq, tk, tv, tdo;
  FA_TRY(tmap_bf16(&tq, q, B, Hq, N, d));
  FA_TRY(tmap_bf16(&tk, k, B, Hkv, N, d));
  FA_TRY(tmap_bf16(&tv, v, B, Hkv, N, d));
  FA_TRY(tmap_bf16(&tdo, dO, B, Hq, N, d));
  fa::DqArgs a;
  a.lse2 = reinterpret_cast<const float*>(ws + w.lse2_off);
  a.drow = reinterpret_cast<const float*>(ws + w.dr_off);
  a.dq = dq;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.causal = causal;
  a.window = window;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_status(fa::launch_bwd_dq(d, tq, tk, tv, tdo, a, dev_status(ds), ds->num_sms, st));
}

fa_status fa_last_device_status(void* stream, int* detail) {
  NvtxRange nv("fa_last_device_status");
  FA_TRY_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds, false));
  int words[fa::kStatusWords] = {};
  FA_TRY_CUDA(cudaMemcpy(words, ds->status, sizeof(words), cudaMemcpyDeviceToHost));
  const int zero[fa::kStatusWords] = {};
  FA_TRY_CUDA(cudaMemcpy(ds->status, zero, sizeof(zero), cudaMemcpyHostToDevice));
  if (words[4] != 0 || ds->unusable) {
    // A block exited with copies or MMAs possibly still in flight: nothing
    // more is launched on this device by this process.
    {
      std::lock_guard<std::mutex> lock(g_mu);
      ds->unusable = true;
    }
    if (detail && words[4] != 0) {
      detail[0] = words[5];
      detail[1] = words[4];
      detail[2] = -1;
    }
    return FA_ERR_DEVICE_DRAIN;
  }
  if (detail) {
    detail[0] = words[1];
    detail[1] = words[2];
    detail[2] = words[3];
  }
  return static_cast<fa_status>(words[0]);
}

fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return FA_ERR_BAD_ARGUMENT;
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  fa::DevStatus st{ds->status, timeout_ns};
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
  return launch_status(cudaGetLastError());
}

fa_status fa_selftest_drain_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return FA_ERR_BAD_ARGUMENT;
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  fa::DevStatus st{ds->status, timeout_ns};
  drain_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
  return launch_status(cudaGetLastError());
}

}  // extern "C"

// ---------------------------------------------------------------------------
// fa_bwd_noalloc: fa_bwd with its scratch in a buffer compiled into the
// library, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace {

// The scratch lives here, in the library's own device image: every device
// that loads the library holds these FA_NOALLOC_SCRATCH_BYTES until exit.
// In host code this name is only a stand-in for the symbol, not a device
// address; the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current.
fa_status noalloc_scratch(void** out) {
  int dev = -1;
  FA_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    FA_TRY_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    if (p == nullptr) return FA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                    int d, int causal, float scale, void* stream) {
  NvtxRange nv("fa_bwd_noalloc");
  FA_TRY(check_shape(B, Hq, Hkv, N, d));
  if (ws_layout(B, Hq, N, d).total > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL_PTR;
  FA_TRY(check_scale(causal, scale));
  DeviceState* ds = nullptr;
  FA_TRY(device_state(&ds));
  void* scratch = nullptr;
  FA_TRY(noalloc_scratch(&scratch));
  // fa_bwd clears the dQ accumulator in its first kernel, so whatever the
  // previous call left in the scratch does not matter.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, scratch,
                (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
