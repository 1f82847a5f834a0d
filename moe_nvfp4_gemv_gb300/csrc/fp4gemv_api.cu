// fp4gemv_api.cu -- the C ABI of libfp4gemv (see include/fp4gemv.h).
//
// Host side only: argument validation (before any launch), launch-shape
// selection (token tile, cluster split of K, ring depth), TMA descriptor
// encoding and the launches themselves.  All arithmetic runs in the kernels.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <cstring>

#include "fp4gemv.h"
#include "fp4gemv_plan.h"
#include "launch.h"

namespace fp4 {
// Per-device error state (one copy per device context of this library image):
// the error word, then the wait limit the kernels' bounded waits use (see
// common.cuh; 0 = the built-in 2 s).
struct DeviceErrorState {
  uint32_t word;
  uint32_t unused;
  unsigned long long wait_limit_ns;
};
__device__ DeviceErrorState g_dev_state = {0u, 0u, 0ull};
static_assert(offsetof(DeviceErrorState, wait_limit_ns) == 8, "the kernels read the limit 8 bytes past the word");
}  // namespace fp4

namespace {

using fp4::GemvParams;
using fp4::KernelInfo;
using fp4::LaunchCfg;

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_skip_stage{-1};  // test hook (fp4gemv_debug_skip_stage)

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Encoded tensor maps are cached per host thread: decode calls re-use the
// same weight and activation buffers, and encoding costs about as much host
// time as the launch itself.  A map depends only on its key (base address,
// shape, strides, box, element type); the cache holds no device state, so a
// stale entry is impossible -- a different buffer is a different key.
struct MapKey {
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  int rank, dtype;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

bool encode_cached(CUtensorMap* m, const MapKey& key) {
  constexpr int kEntries = 64;
  struct Entry {
    MapKey key;
    CUtensorMap map;
    bool used;
  };
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i) {
    if (cache[i].used && cache[i].key == key) {
      *m = cache[i].map;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, static_cast<CUtensorMapDataType>(key.dtype), key.rank, const_cast<void*>(key.base), key.dims,
         key.strides, key.box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.key = key;
  e.map = *m;
  e.used = true;
  return true;
}

// 2-D row-major tensor [outer, inner] with a 128-byte-swizzled box.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.dims[0] = inner;
  k.dims[1] = outer;
  k.strides[0] = row_bytes;
  k.box[0] = box_inner;
  k.box[1] = box_outer;
  k.rank = 2;
  k.dtype = static_cast<int>(dt);
  return encode_cached(m, k);
}

// Activations x [M, K] (bf16, row stride ldx) viewed as [K/64, M, 64]: one
// box {64, rows, atoms} holds `atoms` 64-wide K atoms of `rows` tokens, each
// atom a [rows x 128-byte] 128B-swizzled block -- the layout the MMA reads.
// The register-fed kernel loads a 256-K stage (4 atoms), the tcgen05 kernel
// a 128-K slice (2).
bool encode_x_atoms(CUtensorMap* m, const void* x, int K, int M, int64_t ldx, uint32_t rows, uint32_t atoms) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = x;
  k.dims[0] = 64;
  k.dims[1] = static_cast<uint64_t>(M);
  k.dims[2] = static_cast<uint64_t>(K / 64);
  k.strides[0] = static_cast<uint64_t>(ldx) * 2;
  k.strides[1] = 128;
  k.box[0] = 64;
  k.box[1] = rows;
  k.box[2] = atoms;
  k.rank = 3;
  k.dtype = static_cast<int>(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return encode_cached(m, k);
}

struct DeviceState {
  std::atomic<uint32_t*> err{nullptr};
  std::atomic<int> sms{0};
};
DeviceState g_dev[kMaxDevices];

fp4gemv_status device_state(uint32_t** err, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
  DeviceState& d = g_dev[dev];
  uint32_t* e = d.err.load(std::memory_order_acquire);
  if (!e) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, fp4::g_dev_state) != cudaSuccess) return FP4GEMV_ERR_CUDA;
    e = &static_cast<fp4::DeviceErrorState*>(p)->word;
    d.err.store(e, std::memory_order_release);
  }
  int n = d.sms.load(std::memory_order_acquire);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP4GEMV_ERR_CUDA;
    d.sms.store(n, std::memory_order_release);
  }
  if (err) *err = e;
  if (sms) *sms = n;
  return FP4GEMV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fp4gemv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP4GEMV_OK : FP4GEMV_ERR_CUDA; }

int pick_nt(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

// Pseudo-modes of the register-fed NVFP4 kernel (chunks of <= 16 tokens).
constexpr int kRfBase = 100;
constexpr int kDenseFp4Rf = kRfBase + fp4::kDenseFp4;
constexpr int kMoeGateUpRf = kRfBase + fp4::kMoeGateUp;
constexpr int kMoeDownRf = kRfBase + fp4::kMoeDown;
constexpr int kMoeDownRf3 = kRfBase + 10 + fp4::kMoeDown;  // budgeted for three CTAs per SM
constexpr int kDenseFp4RfCoop = kRfBase + 20 + fp4::kDenseFp4;  // 3 .. 12 tokens, cooperative f16 conversion
constexpr int kDenseFp4Slab = kRfBase + 30 + fp4::kDenseFp4;    // 1 .. 8 tokens, activations resident in smem

cudaError_t kernel_info(int mode, int nt, KernelInfo* info) {
  GemvParams dummy;
  LaunchCfg cfg{};
  switch (mode) {
    case kDenseFp4Rf:
    case kMoeGateUpRf:
    case kMoeDownRf: return fp4::launch_rf(mode - kRfBase, nt, dummy, cfg, info);
    case kMoeDownRf3: return fp4::launch_rf_occ3(fp4::kMoeDown, nt, dummy, cfg, info);
    case kDenseFp4RfCoop: return fp4::launch_rf_coop(fp4::kDenseFp4, nt, dummy, cfg, info);
    case kDenseFp4Slab: return fp4::launch_slab(2, dummy, cfg, info);
    case fp4::kDenseFp4: return fp4::launch_dense_fp4(nt, dummy, cfg, info);
    case fp4::kDenseBf16: return fp4::launch_dense_bf16(nt, dummy, cfg, info);
    default: return fp4::launch_moe(mode, nt, dummy, cfg, info);
  }
}

cudaError_t kernel_launch(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  switch (mode) {
    case kDenseFp4Rf:
    case kMoeGateUpRf:
    case kMoeDownRf: return fp4::launch_rf(mode - kRfBase, nt, p, cfg, nullptr);
    case kMoeDownRf3: return fp4::launch_rf_occ3(fp4::kMoeDown, nt, p, cfg, nullptr);
    case kDenseFp4RfCoop: return fp4::launch_rf_coop(fp4::kDenseFp4, nt, p, cfg, nullptr);
    case kDenseFp4Slab: return fp4::launch_slab(p.slab_r, p, cfg, nullptr);
    case fp4::kDenseFp4: return fp4::launch_dense_fp4(nt, p, cfg, nullptr);
    case fp4::kDenseBf16: return fp4::launch_dense_bf16(nt, p, cfg, nullptr);
    default: return fp4::launch_moe(mode, nt, p, cfg, nullptr);
  }
}

// Ring depth and dynamic shared memory: two CTAs per SM when the kernel's
// tensor-memory footprint allows it (<= 256 columns), else one.
// CTAs per SM of the tcgen05 kernel: two when its tensor memory (512
// columns per SM) allows.
int tc_ctas_per_sm(const KernelInfo& info) { return info.tmem_cols <= 256 ? 2 : 1; }

// Ring of the tcgen05 kernel for a launch of S-rank clusters, within one
// CTA's share of shared memory.  NVFP4 (fp4w): weight stages of 16 KB codes
// + sf_slots 2 KB scale groups (they hide HBM latency) beside nx activation
// slots (they hide L2's): nx = 4 or 3, whichever leaves more weight stages
// (4 on a tie), 2 if neither leaves two.  nx = 3 only with three tensor-
// memory slots: the kernel's parity waits on an activation slot need either
// an even nx (each warpgroup owns its slots) or nx = tensor-memory slots.
// BF16: stages of weights and activations together.  The split-K inbox
// (push mode) follows the ring when S > 1; with one rank it reuses the
// ring, drained by then.
struct TcRing {
  int nstages = 0, nx = 0, wstage = 0, inbox_off = 0;
  size_t smem = 0;
};
TcRing size_ring(const KernelInfo& info, bool fp4w, int sf_slots, int S) {
  TcRing r;
  const int per_sm = tc_ctas_per_sm(info);
  const int inbox = S > 1 ? info.inbox_bytes : 0;
  const int avail = (per_sm == 2 ? 110 * 1024 : 220 * 1024) - 1024 - inbox;
  int bytes = 0;
  if (fp4w) {
    r.wstage = 16384 + 2048 * sf_slots;
    auto stages = [&](int nx) {
      const int n = (avail - nx * info.x_slice_bytes) / r.wstage;
      return n > fp4::kMaxStages ? fp4::kMaxStages : n;
    };
    r.nx = fp4::kMaxXSlots;  // 4
    if (info.tmem_slots == 3 && stages(3) > stages(4)) r.nx = 3;
    if (stages(r.nx) < 2) r.nx = 2;
    r.nstages = stages(r.nx);
    if (r.nstages < 2) r.nstages = 2;
    bytes = r.nstages * r.wstage + r.nx * info.x_slice_bytes;
  } else {
    r.wstage = info.stage_bytes;
    r.nstages = avail / info.stage_bytes;
    if (r.nstages > fp4::kMaxStages) r.nstages = fp4::kMaxStages;
    if (r.nstages < 2) r.nstages = 2;
    bytes = r.nstages * info.stage_bytes;
  }
  if (bytes < info.red_bytes) bytes = info.red_bytes;  // pull mode: partials reuse the ring
  if (bytes < info.inbox_bytes) bytes = info.inbox_bytes;
  r.inbox_off = S > 1 ? bytes : 0;
  r.smem = 1024 + static_cast<size_t>(bytes) + inbox;
  // one CTA per SM: ask for more than half of the SM's shared memory
  if (per_sm == 1 && r.smem < 120 * 1024) r.smem = 120 * 1024;
  return r;
}

// Ring of the register-fed kernel: a stage is the 16 KB weight tile, 2 KB per
// scale group the call needs and the activations (info.stage_bytes); two
// CTAs per SM, each with as many stages as its share of shared memory holds
// (a deeper ring keeps more weight bytes in flight per SM).
constexpr int kRfBudget = 110 * 1024;  // shared memory per register-fed CTA, two per SM (with margin)

void size_ring_rf(const KernelInfo& info, int wtile_bytes, int sf_groups, int* nstages, size_t* smem,
                  int* stage_bytes, int* x_off, int kBudget = kRfBudget) {
  *x_off = wtile_bytes + sf_groups * 2048;
  *stage_bytes = (*x_off + info.stage_bytes + 1023) / 1024 * 1024;
  int ns = (kBudget - 1024 - info.inbox_bytes) / *stage_bytes;
  if (ns > fp4::kMaxStages) ns = fp4::kMaxStages;
  if (ns < 2) ns = 2;
  *nstages = ns;
  *smem = 1024 + static_cast<size_t>(ns) * *stage_bytes + info.inbox_bytes;
}

// Cluster split of K.  A CTA costs its ring stages plus a fixed overhead
// (launch, prologue, first-load latency, cluster reduction, epilogue) of about
// kFixedStages stages; minimise waves x (stages + fixed), ties to the smaller
// split.  Every rank keeps a non-empty K range.
constexpr int kFixedStages = 4;
constexpr int kStageK4 = fp4::kStageK4;

// Tile height and K split of the dense register-fed kernel.  A tile is 16 cw
// rows (cw = 6 .. 8 consumer warps; with silu_mul 8 cw gate + 8 cw up rows,
// cw even), split over S = 1, 2, 4 or 8 cluster ranks along K.  The default
// is 128-row tiles split by pick_split; a lower tile is taken only when its
// grid fits on the GPU at once (cap[S] CTAs in whole clusters) and its CTAs
// are at least 8 % shorter: a stage costs a fixed part (barrier hand-offs,
// activations) plus a part that scales with the tile height, and a CTA adds
// kFixedStages stages (prologue, first loads, reduction, epilogue).  This
// evens out grids such as 224 tiles of 128 rows on 304 CTA slots.
double rf_cta_cost(int cw, int K, int s) {
  const int kslab = ((K + s - 1) / s + 63) / 64 * 64;
  return (static_cast<double>(kslab) / kStageK4) * (0.45 + 0.55 * cw / 8.0) + kFixedStages;
}

void pick_rf_geometry(int n_out, bool paired, int K, int s_default, const int (&cap)[9], int* cw_out, int* s_out) {
  *cw_out = 8;
  *s_out = s_default;
  const long tiles8 = paired ? (n_out + 63) / 64 : (n_out + 127) / 128;
  if (tiles8 * s_default > cap[s_default]) return;  // the default runs in waves: keep it
  double best = rf_cta_cost(8, K, s_default) * 0.92;
  for (int cw = 7; cw >= 6; --cw) {
    if (paired && cw % 2 != 0) continue;
    const int feats = paired ? 8 * cw : 16 * cw;
    const long tiles = (n_out + feats - 1) / feats;
    for (int s = 1; s <= 8; s *= 2) {
      if (s > 1 && K / s < kStageK4) break;
      const int kslab = ((K + s - 1) / s + 63) / 64 * 64;
      if (static_cast<long>(s - 1) * kslab >= K) break;  // every rank keeps a non-empty K range
      if (tiles * s > cap[s]) continue;
      const double cost = rf_cta_cost(cw, K, s);
      if (cost < best) {
        best = cost;
        *cw_out = cw;
        *s_out = s;
      }
    }
  }
}

// Co-resident CTAs of the dense register-fed kernel in clusters of 1 .. 8
// (per device and token tile, queried once).
struct RfCap {
  std::atomic<int> v[2][9];
};
RfCap g_rf_cap[kMaxDevices];

fp4gemv_status rf_capacity(int nt, int (&cap)[9]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
  const int i = nt == 8 ? 0 : 1;
  cap[0] = 0;
  for (int s = 1; s <= 8; ++s) {
    int n = g_rf_cap[dev].v[i][s].load(std::memory_order_acquire);
    if (n == 0) {
      // (size_ring_rf never exceeds the budget, so this is the launches' worst
      // case).  A size the query cannot answer counts as fitting nothing: the
      // plan then keeps the default tiles for it.  The error is cleared so a
      // later launch check does not report it.
      if (fp4::rf_max_clusters(fp4::kDenseFp4, nt, s, kRfBudget, &n) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      if (n < 0) n = 0;
      g_rf_cap[dev].v[i][s].store(n == 0 ? -1 : n, std::memory_order_release);
    }
    cap[s] = n < 0 ? 0 : n * s;  // CTAs
  }
  return FP4GEMV_OK;
}

int pick_split(int tiles, int K, int stage_k, int slots) {
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= 8; s *= 2) {
    if (s > 1 && K / s < stage_k) break;
    const long ctas = static_cast<long>(tiles) * s;
    const long waves = (ctas + slots - 1) / slots;
    const int kslab = ((K + s - 1) / s + 63) / 64 * 64;
    if (s > 1 && static_cast<long>(s - 1) * kslab >= K) break;
    const long stages = (kslab + stage_k - 1) / stage_k;
    const long fixed = kFixedStages * kStageK4 / stage_k;  // the same time in this kernel's stages
    const long cost = waves * (stages + fixed);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// A single wave of more CTAs than SMs (two CTAs per SM) puts two on some SMs
// and one on the rest, and the call ends with the doubled SMs.  Between no
// split and a split of two, compare the busiest SM's work, an SM running
// two CTAs at once delivering 1.5x one CTA's throughput (8B gate_up at 32
// tokens, 224 tiles: 37.5 -> 36.0 us with the split).
int balance_split(int S, int tiles, int K, int stage_k, int sms, int per_sm) {
  if (S != 1 || per_sm != 2 || tiles <= sms || tiles > 2 * sms || K / 2 < stage_k) return S;
  const double fixed = kFixedStages * kStageK4 / stage_k;
  const int kslab2 = ((K + 1) / 2 + 63) / 64 * 64;
  const double c1 = 2 * ((K + stage_k - 1) / stage_k + fixed) / 1.5;
  const int n2 = (2 * tiles + sms - 1) / sms;
  const double c2 = n2 * ((kslab2 + stage_k - 1) / stage_k + fixed) / (n2 > 1 ? 1.5 : 1.0);
  return c2 < c1 ? 2 : 1;
}

// The tcgen05 kernel's plan for an N x K weight (NVFP4 or BF16): tiles of
// 128 features (64 with silu_mul), the K split, the scale groups a weight
// stage holds (one 128-row group; with silu_mul the gate box's and the up
// box's, a third when an up box straddles two) and the ring.
struct TcPlan {
  KernelInfo info{};
  int per_sm = 2, tiles = 0, S = 1, kslab = 0, sf_slots = 1;
  TcRing ring;
};
bool plan_tc(int kmode, int NT, bool fp4w, int N, int K, bool silu, int sms, TcPlan* tp) {
  if (kernel_info(kmode, NT, &tp->info) != cudaSuccess) return false;
  tp->per_sm = tc_ctas_per_sm(tp->info);
  const int n_out = silu ? N / 2 : N;
  const int box_rows = silu ? 64 : 128;
  tp->tiles = (n_out + box_rows - 1) / box_rows;
  const int stage_k = fp4w ? fp4::kStageK4 : fp4::kStageK16;
  int S0 = pick_split(tp->tiles, K, stage_k, sms * tp->per_sm);
  if (fp4w) S0 = balance_split(S0, tp->tiles, K, stage_k, sms, tp->per_sm);
  tp->kslab = ((K + S0 - 1) / S0 + 63) / 64 * 64;
  tp->S = (K + tp->kslab - 1) / tp->kslab;  // every cluster rank gets a non-empty K range
  tp->sf_slots = silu ? ((N / 2) % 64 == 0 ? 2 : 3) : 1;
  tp->ring = size_ring(tp->info, fp4w, tp->sf_slots, tp->S);
  return true;
}

// The register-fed dense kernel's plan (tile height 16 cw, split, scale
// groups per stage) for N x K on a GPU with `sms` SMs and cap[] co-resident
// CTAs per cluster size.
void plan_rf(int N, int K, bool silu, int sms, const int (&cap)[9], int* cw, int* s0, int* sf_groups) {
  const int n_out = silu ? N / 2 : N;
  const int s_default = pick_split((n_out + (silu ? 63 : 127)) / (silu ? 64 : 128), K, fp4::kStageK4, sms * 2);
  pick_rf_geometry(n_out, silu, K, s_default, cap, cw, s0);
  // 128-row scale groups a stage holds: a box of h rows starting at an
  // offset o (mod h) stays in one group for every tile iff h divides 128
  // and o is a multiple of h
  const int h = silu ? 8 * *cw : 16 * *cw;
  const bool even = 128 % h == 0;
  *sf_groups = silu ? (even ? 1 : 2) + ((even && (N / 2) % h == 0) ? 1 : 2) : (even ? 1 : 2);
}

// The slab kernel's plan (M <= 8): tiles of 128 rows (two 16-row blocks per
// consumer warp, four consumer warps; with silu_mul 64 gate + 64 up rows),
// three CTAs per SM, and the largest K split S in 1, 2, 4, 8 whose grid still
// runs in one wave (tiles x S <= 3 x SMs) -- for 1 .. kSlabMaxM tokens and
// weights of at least kSlabMinTiles tiles per SM, provided the grid then
// holds at least kSlabMinFill CTAs per SM and the CTA's activation slab and
// two 256-K weight stages fit a third of the SM's shared memory.  Measured on
// the Llama-3-8B layers: gate_up at 1 .. 4 tokens 9-11 % faster than the
// register-fed kernel alone and ~1 % on a whole decode step; qkv (48 tiles,
// split 8) 5 % faster alone but slower inside a step next to the register-
// fed kernels (their 110 KB CTAs and these 70 KB ones pack badly at the
// hand-over); at 8 tokens the larger slab made it slower; on grids of fewer
// CTAs (o_proj, down: 32 tiles) the register-fed kernel's 8-warp CTAs are as
// fast or faster, and more splits (clusters of 16) or several waves were
// slower.  False: the register-fed kernel serves the call.
constexpr int kSlabOcc = 3;
constexpr double kSlabMinFill = 2.4;
constexpr double kSlabMinTiles = 1.2;  // tiles per SM before the split
constexpr int kSlabMaxM = 4;
constexpr int kSmemPerSm = 228 * 1024;   // shared memory per SM
constexpr int kSmemPerCta = 2048;        // per-CTA reservation + the kernel's static shared memory

struct SlabPlan {
  int r = 2, cw = 4, S = 1, kslab = 0, sf_groups = 1, nstages = 0, stage_bytes = 0, slab_bytes = 0, occ = 0;
  size_t smem = 0;
};

// regs[r - 1]: registers per thread of the kernel with r row blocks per warp
// (with the threads and the shared memory they bound the CTAs per SM).
bool plan_slab(int M, int N, int K, bool silu, int sms, int inbox_bytes, const int (&regs)[2], SlabPlan* sp) {
  if (M < 1 || M > kSlabMaxM || sms < 1) return false;
  const int r = 2, cw = 4, occ = kSlabOcc;
  const int warp_regs = (regs[r - 1] * 32 + 255) / 256 * 256;  // registers allocated per warp
  if (static_cast<long>(occ) * (cw + 1) * warp_regs > 65536) return false;
  const int trows = 16 * r * cw;
  const int h = silu ? trows / 2 : trows;  // rows per box, h | 128, boxes start on multiples of h
  const long tiles = ((silu ? N / 2 : N) + h - 1) / h;
  const int groups = silu ? 1 + ((N / 2) % h == 0 ? 1 : 2) : 1;
  const int stage = (trows * 128 + groups * 2048 + 1023) / 1024 * 1024;
  const int dyn = kSmemPerSm / occ - kSmemPerCta;
  if (tiles < kSlabMinTiles * sms) return false;
  for (int S = 8; S >= 1; S /= 2) {
    if (tiles * S > static_cast<long>(occ) * sms) continue;         // more than one wave
    if (tiles * S < kSlabMinFill * sms) return false;                // too few CTAs to fill the SMs
    const int kslab = ((K + S - 1) / S + 63) / 64 * 64;
    if (S > 1 && (kslab < 256 || static_cast<long>(S - 1) * kslab >= K)) continue;
    const int nst = (kslab + 255) / 256;
    if (nst > fp4::kSlabMaxStages) return false;
    const int slab = (M * nst * 512 + 1023) / 1024 * 1024;
    // Two stages: with three CTAs per SM that is 6 stages (~110 KB) in
    // flight per SM; deeper rings measured slower (gate_up 15.4 -> 16.0 us at
    // M = 1), their burst of first loads delaying the previous grid's end.
    const int ns = 2;
    if (1024 + slab + ns * stage + inbox_bytes > dyn) return false;
    sp->r = r;
    sp->cw = cw;
    sp->kslab = kslab;
    sp->S = (K + kslab - 1) / kslab;  // every cluster rank gets a non-empty K range
    sp->sf_groups = groups;
    sp->nstages = ns;
    sp->stage_bytes = stage;
    sp->slab_bytes = slab;
    sp->occ = occ;
    sp->smem = 1024 + static_cast<size_t>(slab) + static_cast<size_t>(ns) * stage + inbox_bytes;
    return true;
  }
  return false;
}

// The slab kernel for MoE gate_up: 128-row tiles (a routed [up; gate] group
// of 64 features, or a shared-expert pair of 64-row gate and up boxes), the
// CTA's activation rows resident, two scale groups per weight stage.  Two
// forms:
//   split:   one tile per CTA, routed chunks of up to fp4::kSlabChunk pairs,
//            H split over a cluster so that the CTAs of every expert the
//            call can touch (at most min(P, E) routed chunks plus the shared
//            expert's) run in one wave at three CTAs per SM.  One token of
//            the E = 128, top-8, H = 4096, I = SI = 1536 block (216 tiles):
//            a split of two; the register-fed kernel ran those 216 whole-H
//            CTAs in one uneven wave.
//   grouped: the whole H per CTA, T = 1 or 2 of its column's tiles in turn
//            over the same activation rows, many waves of CTAs.  Measured
//            on that block (us per call, L2-cold, 8 routings; against the
//            register-fed kernel's chunks of 8): a sweep of chunk, tiles per
//            CTA and CTAs per SM put the best at one tile per CTA for 2
//            tokens (32.2 vs 39.7), two tiles per CTA from 4 tokens (4: 56.6
//            vs 64.4; 8: 102.3 vs 115.3; 16: 164.6 vs 176.6), pairs of 2 at
//            three CTAs per SM up to 16 tokens and pairs of 4 at two CTAs
//            per SM (a deeper ring) from 32 (255 vs 265); fewer, longer
//            CTAs were slower at every size (each CTA's stream is bounded
//            by its ring, so the GPU needs many of them).  Where that grid
//            fills a wave badly (below): 3 tokens 46.3 (55.6), 5: 71.5
//            (81.1), 6: 85.2 (97.8), 7: 90.6 (100.0).  The ring takes as many stages as fit (2 .. 8); a
//            chunk that leaves room for fewer than two is halved.
struct SlabMoePlan {
  int S = 1, kslab = 0, T = 0, groups = 0, chunk = fp4::kSlabChunk, slab_bytes = 0, stage_bytes = 0, nstages = 2,
      occ = kSlabOcc;
  size_t smem = 0;
};

bool plan_slab_moe(int M, int topk, int E, int H, int I, int SI, int sms, int regs, SlabMoePlan* sp) {
  const int cw = fp4::kSlabMaxCW, occ3 = kSlabOcc;
  const int warp_regs = (regs * 32 + 255) / 256 * 256;
  if (static_cast<long>(occ3) * (cw + 1) * warp_regs > 65536 || sms < 1 || M > 64) return false;
  const long P = static_cast<long>(M) * topk;
  const int stage = 128 * 128 + 2 * 2048;  // codes + two scale groups (shared-expert gate and up boxes)
  const int tiles = I / 64 > (SI + 63) / 64 ? I / 64 : (SI + 63) / 64;
  {  // split form
    const long routed_cols = P < E ? P : E;
    const long shared_cols = (M + fp4::kSlabChunk - 1) / fp4::kSlabChunk;
    const long ctas1 = routed_cols * (I / 64) + shared_cols * ((SI + 63) / 64);
    const int rows = static_cast<int>(P < fp4::kSlabChunk ? P : fp4::kSlabChunk);  // B rows of a chunk, at most
    const int dyn = kSmemPerSm / occ3 - kSmemPerCta;
    for (int S = 8; S >= 1; S /= 2) {
      if (ctas1 * S > static_cast<long>(occ3) * sms) continue;  // more than one wave
      const int kslab = ((H + S - 1) / S + 63) / 64 * 64;
      if (S > 1 && (kslab < 256 || static_cast<long>(S - 1) * kslab >= H)) continue;
      const int nst = (kslab + 255) / 256;
      if (nst > fp4::kSlabMaxStages) break;
      const int slab = (rows * nst * 512 + 1023) / 1024 * 1024;
      const size_t smem = 1024 + static_cast<size_t>(slab) + 2 * static_cast<size_t>(stage) + fp4::SlabInboxBytes;
      if (smem > static_cast<size_t>(dyn)) break;  // a smaller split only needs more
      sp->S = (H + kslab - 1) / kslab;
      sp->kslab = kslab;
      sp->T = 0;
      sp->groups = static_cast<int>(tiles) * sp->S;
      sp->chunk = fp4::kSlabChunk;
      sp->slab_bytes = slab;
      sp->stage_bytes = stage;
      sp->nstages = 2;
      sp->occ = occ3;
      sp->smem = smem;
      return true;
    }
  }
  // grouped form
  const int nst = (H + 255) / 256;
  if (nst > fp4::kSlabMaxStages) return false;
  int occ = M >= 32 ? 2 : 3;
  int T = M <= 2 ? 1 : 2;
  int chunk0 = M >= 32 ? 4 : M <= 2 ? 1 : 2;
  if (M >= 3 && M < 32) {
    // Two exceptions by the CTAs that stream (the expected distinct experts
    // of P uniform draws, at least ceil(P / c) chunks of c pairs, plus the
    // shared expert's ceil(M / c) chunks, times the tile groups): two tiles
    // of pairs of 2 filling less than 0.7 of a wave at three per SM take
    // pairs of 4 at two per SM (deeper rings) if those fit one wave; more
    // than 0.9 and at most 1.35 waves take one tile per CTA.
    const double distinct = E * (1.0 - std::pow(1.0 - 1.0 / E, static_cast<double>(P)));
    auto ctas = [&](int T_, int c) {
      return (std::max(distinct, static_cast<double>((P + c - 1) / c)) + (M + c - 1) / c) * ((tiles + T_ - 1) / T_);
    };
    const double f = ctas(2, 2) / (3.0 * sms);
    if (f < 0.7 && ctas(2, 4) <= 2.0 * sms) T = 2, chunk0 = 4, occ = 2;
    else if (f > 0.9 && f <= 1.35) T = 1;
  }
  for (int chunk = chunk0; chunk >= 1; chunk /= 2) {
    const int rows = static_cast<int>(P < chunk ? P : chunk);
    const int slab = (rows * nst * 512 + 1023) / 1024 * 1024;
    const long room = static_cast<long>(kSmemPerSm / occ - kSmemPerCta) - 1024 - slab - fp4::SlabInboxBytes;
    long ns = room / stage;
    if (ns > fp4::kMaxStages) ns = fp4::kMaxStages;
    if (ns > static_cast<long>(T) * nst) ns = static_cast<long>(T) * nst;
    if (ns < 2) continue;
    sp->S = 1;
    sp->kslab = H;
    sp->T = T;
    sp->groups = (tiles + T - 1) / T;
    sp->chunk = chunk;
    sp->slab_bytes = slab;
    sp->stage_bytes = stage;
    sp->nstages = static_cast<int>(ns);
    sp->occ = occ;
    sp->smem = 1024 + static_cast<size_t>(slab) + static_cast<size_t>(ns) * stage + fp4::SlabInboxBytes;
    return true;
  }
  return false;
}

std::atomic<int> g_slab_moe_regs[kMaxDevices];

// The slab kernel for down_combine: the whole K per CTA (its activation
// rows resident), chunks of up to 8 pairs of one expert, T row tiles per CTA
// streamed in turn over the same rows; one scale group per 128-row weight
// stage, as many stages as fit (2 .. 8).  The combine is a kernel of its own
// after it.  T and the CTAs per SM follow the number of CTAs that stream:
// the host does not see the ids, so it takes the expected number of distinct
// experts of P = M topk uniform draws (at least P / 8 chunks) plus the shared
// expert's token chunks as the columns, times ceil(tiles / T):
//   one tile per CTA at two CTAs per SM if those fit in one wave (deeper
//   rings), else two tiles at two per SM if they fit, else two tiles at
//   three per SM, except when those fill more than 0.9 and at most 1.35
//   waves (then one tile at three per SM: twice as many CTAs of half the
//   length, and no nearly empty second wave of long ones).
// When that grid still holds more than one wave, the persistent form
// (k_moe_down_persist.cuh) serves the call instead: three CTAs per SM take
// the (tile group, column) items from a counter, so no slot idles while
// another wave finishes; its items hold 4 tiles when that still gives every
// slot 1.6 items or more on average, else 2 tiles when that does, else 1
// (an item's start costs a few microseconds -- the activation rows'
// round trip and the ring's restart -- so the longest items that still
// spread evenly).
// Measured on the E = 128, top-8, H = 4096, I = SI = 1536 block (us per
// call, L2-flushed by rotation, 8 routings; sweeps of T = 1 .. 4, chunks of
// 2, 4, 8 and two or three CTAs per SM): one CTA per item 1 token 14.9,
// 2 tokens 24.6, 3: 30.7; persistent 4 tokens 41.3 (one CTA per item:
// 42.3), 5: 45.0, 6: 55.0, 8: 61.2 (66.6), 16: 91.5 (103.3), 32: 131.3
// (148.3), 64: 177.2 (196.4; persistent with 2-tile items 183.2).
struct SlabDownPlan {
  int T = 2, groups = 1, chunk = 8, slab_bytes = 0, stage_bytes = 0, nstages = 2, occ = 3;
  bool persist = false;
  size_t smem = 0;
};

constexpr int kSmemPerCtaDown = 4096;  // reservation + static shared memory

bool plan_slab_down(int M, int topk, int E, int H, int I, int SI, int sms, int regs, SlabDownPlan* sp) {
  const int cw = fp4::kSlabMaxCW;
  const int warp_regs = (regs * 32 + 255) / 256 * 256;
  if (sms < 1 || M < 1 || M > 64) return false;
  const long P = static_cast<long>(M) * topk;
  int chunk = fp4::kSlabNT;
  const int tiles = (H + 127) / 128;
  const double distinct = E * (1.0 - std::pow(1.0 - 1.0 / E, static_cast<double>(P)));
  auto columns = [&](int cn) {
    return std::max(distinct, static_cast<double>((P + cn - 1) / cn)) + static_cast<double>((M + cn - 1) / cn);
  };
  double cols = columns(chunk);
  auto ctas = [&](int T) { return cols * ((tiles + T - 1) / T); };
  int T = 2, occ = 3;
  const double f = ctas(2) / (3.0 * sms);  // waves of two-tile CTAs at three per SM
  if (ctas(1) <= 2.0 * sms) T = 1, occ = 2;
  else if (ctas(2) <= 2.0 * sms) T = 2, occ = 2;
  else if (f > 0.9 && f <= 1.35) T = 1, occ = 3;
  // More CTAs than one wave: the persistent grid instead, three CTAs per
  // SM; chunks of 4 pairs when there are no more pairs than experts (few
  // experts then take more than 4, and the half-height slab leaves room for
  // a deeper ring); items of the most tiles (4, 2, 1) that still give every
  // CTA slot 1.6 items or more on average.
  const bool persist = ctas(T) > static_cast<double>(occ) * sms;
  if (persist) {
    occ = 3;
    if (P <= E) {
      chunk = 4;
      cols = columns(chunk);
    }
    const double slots = 3.0 * sms;
    T = ctas(4) >= 1.6 * slots ? 4 : ctas(2) >= 1.6 * slots ? 2 : 1;
  }
  if (static_cast<long>(occ) * (cw + 1) * warp_regs > 65536) return false;
  const int rows = static_cast<int>(P < chunk ? P : chunk);
  const int kmax = I > SI ? I : SI;
  const int nst = (kmax + 255) / 256;
  if (nst > fp4::kSlabMaxStages) return false;
  const int slab = (rows * nst * 512 + 1023) / 1024 * 1024;
  const int stage = 128 * 128 + 2048;
  const long room = static_cast<long>(kSmemPerSm / occ - kSmemPerCtaDown) - 1024 - slab;
  int ns = static_cast<int>(room / stage);
  if (ns > fp4::kMaxStages) ns = fp4::kMaxStages;
  if (!persist && ns > T * ((I + 255) / 256)) ns = T * ((I + 255) / 256);  // (no deeper than a routed CTA's stream)
  if (ns < 2) return false;
  sp->groups = (tiles + T - 1) / T;
  sp->T = (tiles + sp->groups - 1) / sp->groups;
  sp->persist = persist;
  sp->chunk = chunk;
  sp->slab_bytes = slab;
  sp->stage_bytes = stage;
  sp->nstages = ns;
  sp->occ = occ;
  sp->smem = 1024 + static_cast<size_t>(slab) + static_cast<size_t>(ns) * stage;
  return true;
}
std::atomic<int> g_slab_down_regs[kMaxDevices];

// Registers per thread of both slab-kernel variants (queried once per device).
std::atomic<int> g_slab_regs[kMaxDevices][2];

fp4gemv_status slab_registers(int (&regs)[2]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
  for (int r = 1; r <= 2; ++r) {
    int v = g_slab_regs[dev][r - 1].load(std::memory_order_acquire);
    if (v == 0) {
      if (fp4::slab_regs(r, &v) != cudaSuccess || v <= 0) return FP4GEMV_ERR_CUDA;
      g_slab_regs[dev][r - 1].store(v, std::memory_order_release);
    }
    regs[r - 1] = v;
  }
  return FP4GEMV_OK;
}

// sf_kbp: 16-wide K blocks per 128-row group of the scale buffer (0: the
// exact roundup(K / 16, 4); more for buffers padded along K).
fp4gemv_status dense_launch(int mode, const void* x, int64_t ldx, const void* w, const uint8_t* w_sf,
                            const float* gs, void* out, int64_t ldo, int M, int N, int K, int silu_mul, int pdl,
                            cudaStream_t stream, int sf_kbp = 0) {
  const bool fp4w = mode == fp4::kDenseFp4;
  const int kbp_exact = ((K / 16) + 3) / 4 * 4;
  if (sf_kbp != 0 && (sf_kbp < kbp_exact || sf_kbp % 4 != 0)) return FP4GEMV_ERR_INVALID_ARG;
  // Order of the checks: flags and sizes, then alignment, then null
  // pointers (a null pointer passes the alignment test), so a call with
  // null pointers and a bad size reports the size.
  if ((silu_mul != 0 && silu_mul != 1) || (pdl != 0 && pdl != 1)) return FP4GEMV_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return FP4GEMV_ERR_INVALID_ARG;
  if (M > FP4GEMV_MAX_M || N % 16 != 0 || (silu_mul && N % 32 != 0) || K % 64 != 0) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (fp4w && K < 256) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  const int n_out = silu_mul ? N / 2 : N;
  if (ldx < K || ldo < n_out) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ldx * 2) % 16 != 0 || !aligned(w, 16) || !aligned(out, 16) || ldo % 8 != 0)
    return FP4GEMV_ERR_MISALIGNED;
  if (fp4w && !aligned(w_sf, 16)) return FP4GEMV_ERR_MISALIGNED;
  if (gs && !aligned(gs, 4)) return FP4GEMV_ERR_MISALIGNED;
  if (!x || !w || !out || (fp4w && (!w_sf || !gs))) return FP4GEMV_ERR_INVALID_ARG;

  uint32_t* err = nullptr;
  int sms = 0;
  fp4gemv_status st = device_state(&err, &sms);
  if (st != FP4GEMV_OK) return st;

  // NVFP4 weights and M <= 16: the register-fed kernel (8- or 16-token tile);
  // otherwise the tcgen05 kernel (at 32 tokens the register-fed kernel is
  // bound by its MMA count and no faster).  3 .. 12 tokens: the variant whose
  // consumer warps convert each stage's activations to f16 together
  // (measured on the Llama-3-8B layers against the bf16 route: gate_up 29.6
  // -> 25.9 us at 9 tokens, 29.9 -> 27.0 at 12; at 16 tokens the conversion
  // and its per-stage barrier cost what the cheaper dequantization saves).
  const bool rf = fp4w && M <= 16;
  int kmode = rf ? (M >= 3 && M <= 12 ? kDenseFp4RfCoop : kDenseFp4Rf) : mode;
  const int NT = rf ? (M <= 8 ? 8 : 16) : pick_nt(M);
  int nstages = 0, stage_bytes = 0, x_off = 0;
  size_t smem = 0;
  // 1 .. 8 tokens: the slab kernel when the CTA's activations fit in shared
  // memory, else the register-fed kernel.
  bool slab = false;
  SlabPlan sp;
  if (rf && M <= 8) {
    int regs[2];
    st = slab_registers(regs);
    if (st != FP4GEMV_OK) return st;
    slab = plan_slab(M, N, K, silu_mul != 0, sms, fp4::SlabInboxBytes, regs, &sp);
    if (slab) kmode = kDenseFp4Slab;
  }
  // A tile is `box_rows` weight rows per box: 128 output features (tcgen05),
  // or with silu_mul 64 features (64 gate rows + the 64 matching up rows, two
  // boxes); the register-fed kernel's tiles are 16 cw rows (see
  // pick_rf_geometry).
  int cw = 8, S0 = 1, kslab = 0;
  TcPlan tp;  // tcgen05 kernel
  TcRing& tr = tp.ring;
  if (slab) {
    cw = sp.cw;
    nstages = sp.nstages;
    smem = sp.smem;
    stage_bytes = sp.stage_bytes;
    x_off = sp.slab_bytes;
    kslab = sp.kslab;
  } else if (rf) {
    KernelInfo info{};
    if (kernel_info(kmode, NT, &info) != cudaSuccess) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
    int cap[9];
    st = rf_capacity(NT, cap);
    if (st != FP4GEMV_OK) return st;
    int sf_groups = 1;
    plan_rf(N, K, silu_mul != 0, sms, cap, &cw, &S0, &sf_groups);
    size_ring_rf(info, 16 * cw * 128, sf_groups, &nstages, &smem, &stage_bytes, &x_off);
    kslab = ((K + S0 - 1) / S0 + 63) / 64 * 64;
  } else {
    if (!plan_tc(kmode, NT, fp4w, N, K, silu_mul != 0, sms, &tp)) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
    nstages = tr.nstages;
    smem = tr.smem;
    kslab = tp.kslab;
  }
  const int tile_rows = slab ? 16 * sp.r * cw : 16 * cw;
  const int box_rows = rf ? (silu_mul ? tile_rows / 2 : tile_rows) : (silu_mul ? 64 : 128);
  const int tiles = (n_out + box_rows - 1) / box_rows;
  const int S = (K + kslab - 1) / kslab;  // every cluster rank gets a non-empty K range
  const int sf_slots = tp.sf_slots;

  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  if (fp4w) {
    if (!encode_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K / 2, N, K / 2, 128, box_rows))
      return FP4GEMV_ERR_CUDA;
  } else {
    if (!encode_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, K, N, static_cast<uint64_t>(K) * 2, 64, box_rows))
      return FP4GEMV_ERR_CUDA;
  }
  if (slab) {
    // (activations read with plain loads)
  } else if (fp4w) {
    if (!encode_x_atoms(&p.tm_x, x, K, M, ldx, NT, rf ? 4 : 2)) return FP4GEMV_ERR_CUDA;
  } else {
    if (!encode_2d(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, static_cast<uint64_t>(ldx) * 2, 64, NT))
      return FP4GEMV_ERR_CUDA;
  }
  p.sf = w_sf;
  p.x = static_cast<const uint16_t*>(x);
  p.ldx = ldx;
  p.gs = gs;
  p.out = static_cast<uint16_t*>(out);
  p.ldo = ldo;
  p.M = M;
  p.n_out = n_out;
  p.n_half = N / 2;
  p.silu = silu_mul;
  p.K = K;
  p.k_split = kslab;
  p.rows_w = N;
  p.kbp = sf_kbp ? sf_kbp : kbp_exact;
  p.nstages = nstages;
  p.nx = tr.nx;
  p.wstage = tr.wstage;
  p.sf_slots = sf_slots;
  p.inbox_off = tr.inbox_off;
  p.stage_bytes = stage_bytes;
  p.x_off = x_off;
  p.cw = cw;
  p.slab_r = slab ? sp.r : 0;
  p.skip_stage = g_skip_stage.load(std::memory_order_relaxed);
  p.err = err;

  LaunchCfg cfg{};
  cfg.grid = dim3(tiles * S, 1, 1);
  cfg.cluster = S;
  cfg.smem = smem;
  cfg.pdl = pdl;
  cfg.stream = stream;
  return from_cuda(kernel_launch(kmode, NT, p, cfg));
}

}  // namespace

extern "C" {

fp4gemv_status fp4gemv_plan_rf(int N, int K, int silu_mul, int sms, const int* cap, fp4gemv_rf_plan* out) {
  if (!cap || !out || sms < 1 || (silu_mul != 0 && silu_mul != 1) || N < 1 || K < 1) return FP4GEMV_ERR_INVALID_ARG;
  if (N % 16 != 0 || (silu_mul && N % 32 != 0) || K % 64 != 0 || K < 256) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  int c[9];
  for (int s = 0; s < 9; ++s) c[s] = s == 0 ? 0 : cap[s];
  int cw = 8, s0 = 1, groups = 1;
  plan_rf(N, K, silu_mul != 0, sms, c, &cw, &s0, &groups);
  const int feats = silu_mul ? 8 * cw : 16 * cw;
  const int n_out = silu_mul ? N / 2 : N;
  const int kslab = ((K + s0 - 1) / s0 + 63) / 64 * 64;
  const int split = (K + kslab - 1) / kslab;
  out->tile_rows = 16 * cw;
  out->split = split;
  out->ctas = (n_out + feats - 1) / feats * split;
  out->scale_groups = groups;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_plan_slab(int M, int N, int K, int silu_mul, int sms, const int* regs, fp4gemv_slab_plan* out) {
  if (!regs || !out || sms < 1 || (silu_mul != 0 && silu_mul != 1) || M < 1 || N < 1 || K < 1)
    return FP4GEMV_ERR_INVALID_ARG;
  if (M > 8 || N % 16 != 0 || (silu_mul && N % 32 != 0) || K % 64 != 0 || K < 256) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  const int rg[2] = {regs[0], regs[1]};
  if (rg[0] < 1 || rg[1] < 1) return FP4GEMV_ERR_INVALID_ARG;
  SlabPlan sp;
  if (!plan_slab(M, N, K, silu_mul != 0, sms, fp4::SlabInboxBytes, rg, &sp)) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  const int trows = 16 * sp.r * sp.cw;
  const int feats = silu_mul ? trows / 2 : trows;
  const int n_out = silu_mul ? N / 2 : N;
  out->row_blocks = sp.r;
  out->warps = sp.cw;
  out->tile_rows = trows;
  out->split = sp.S;
  out->ctas = (n_out + feats - 1) / feats * sp.S;
  out->k_slab = sp.kslab;
  out->stages = sp.nstages;
  out->slab_bytes = sp.slab_bytes;
  out->ctas_per_sm = sp.occ;
  out->smem_bytes = sp.smem;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_plan_moe_slab(int M, int topk, int E, int H, int I, int SI, int sms, int regs,
                                     fp4gemv_moe_slab_plan* out) {
  if (!out || sms < 1 || regs < 1 || M < 1 || topk < 1 || E < 1 || H < 1 || I < 1 || SI < 1)
    return FP4GEMV_ERR_INVALID_ARG;
  if (static_cast<long>(M) * topk > 1024 || H % 64 != 0 || H < 256 || I % 64 != 0 || SI % 64 != 0)
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  SlabMoePlan sp;
  if (!plan_slab_moe(M, topk, E, H, I, SI, sms, regs, &sp)) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  out->split = sp.S;
  out->k_slab = sp.kslab;
  out->tiles_per_cta = sp.T;
  out->groups = sp.groups;
  out->chunk_pairs = sp.chunk;
  out->columns = M * topk + (M + sp.chunk - 1) / sp.chunk;
  out->tiles = I / 64 > (SI + 63) / 64 ? I / 64 : (SI + 63) / 64;
  out->slab_bytes = sp.slab_bytes;
  out->stage_bytes = sp.stage_bytes;
  out->stages = sp.nstages;
  out->ctas_per_sm = sp.occ;
  out->smem_bytes = sp.smem;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_plan_moe_down_slab(int M, int topk, int E, int H, int I, int SI, int sms, int regs,
                                          fp4gemv_moe_down_slab_plan* out) {
  if (!out || sms < 1 || regs < 1 || M < 1 || topk < 1 || E < 1 || H < 1 || I < 1 || SI < 1)
    return FP4GEMV_ERR_INVALID_ARG;
  if (static_cast<long>(M) * topk > 1024 || H % 64 != 0 || I % 64 != 0 || I < 256 || SI % 64 != 0 || SI < 256)
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  SlabDownPlan sp;
  if (M > 64 || !plan_slab_down(M, topk, E, H, I, SI, sms, regs, &sp)) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  out->tiles_per_cta = sp.T;
  out->groups = sp.groups;
  out->columns = M * topk + (M + sp.chunk - 1) / sp.chunk;
  out->chunk_pairs = sp.chunk;
  out->slab_bytes = sp.slab_bytes;
  out->stage_bytes = sp.stage_bytes;
  out->stages = sp.nstages;
  out->ctas_per_sm = sp.occ;
  out->persistent = sp.persist ? 1 : 0;
  out->smem_bytes = sp.smem;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_plan_tc(int M, int N, int K, int silu_mul, int bf16_weights, int sms, fp4gemv_tc_plan* out) {
  if (!out || sms < 1 || (silu_mul != 0 && silu_mul != 1) || (bf16_weights != 0 && bf16_weights != 1) || M < 1 ||
      N < 1 || K < 1)
    return FP4GEMV_ERR_INVALID_ARG;
  const bool fp4w = bf16_weights == 0;
  if (M > FP4GEMV_MAX_M || N % 16 != 0 || (silu_mul && N % 32 != 0) || K % 64 != 0 || (fp4w && K < 256) ||
      (fp4w && M <= 16))
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  const int NT = pick_nt(M);
  TcPlan tp;
  if (!plan_tc(fp4w ? fp4::kDenseFp4 : fp4::kDenseBf16, NT, fp4w, N, K, silu_mul != 0, sms, &tp))
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  out->tokens_tile = NT;
  out->ctas_per_sm = tp.per_sm;
  out->tiles = tp.tiles;
  out->split = tp.S;
  out->k_slab = tp.kslab;
  out->weight_stages = tp.ring.nstages;
  out->act_slots = tp.ring.nx;
  out->scale_slots = fp4w ? tp.sf_slots : 0;
  out->inbox_in_ring = tp.S == 1 ? 1 : 0;
  out->smem_bytes = tp.ring.smem;
  return FP4GEMV_OK;
}

size_t fp4gemv_scale_bytes(int rows, int K) {
  if (rows < 1 || K < 16) return 0;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((K / 16 + 3) / 4 * 4);
}

fp4gemv_status fp4gemv_nvfp4_gemv(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                  const float* global_scale, void* out, int64_t ldo, int M, int N, int K,
                                  int silu_mul, int pdl, cudaStream_t stream) {
  return dense_launch(fp4::kDenseFp4, x, ldx, w, w_sf, global_scale, out, ldo, M, N, K, silu_mul, pdl, stream);
}

fp4gemv_status fp4gemv_nvfp4_gemv_padded(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                         int sf_k_blocks, const float* global_scale, void* out, int64_t ldo, int M,
                                         int N, int K, int silu_mul, int pdl, cudaStream_t stream) {
  return dense_launch(fp4::kDenseFp4, x, ldx, w, w_sf, global_scale, out, ldo, M, N, K, silu_mul, pdl, stream,
                      sf_k_blocks);
}

fp4gemv_status fp4gemv_bf16_gemv(const void* x, int64_t ldx, const void* w, void* out, int64_t ldo, int M, int N,
                                 int K, int silu_mul, int pdl, cudaStream_t stream) {
  return dense_launch(fp4::kDenseBf16, x, ldx, w, nullptr, nullptr, out, ldo, M, N, K, silu_mul, pdl, stream);
}

fp4gemv_status fp4gemv_dequantize_rows_padded(const uint8_t* w, const uint8_t* w_sf, int sf_k_blocks, void* out,
                                              int rows, int K, cudaStream_t stream) {
  if (rows < 1 || K < 1) return FP4GEMV_ERR_INVALID_ARG;
  if (rows % 16 != 0 || K % 256 != 0) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (sf_k_blocks != 0 && (sf_k_blocks < K / 16 || sf_k_blocks % 4 != 0)) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(out, 16) || !aligned(w_sf, 4)) return FP4GEMV_ERR_MISALIGNED;
  if (!w || !w_sf || !out) return FP4GEMV_ERR_INVALID_ARG;
  fp4gemv_status st = device_state(nullptr, nullptr);
  if (st != FP4GEMV_OK) return st;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return from_cuda(fp4::launch_dequantize_rows(w, w_sf, out, rows, K, sf_k_blocks, stream));
}

fp4gemv_status fp4gemv_dequantize_rows(const uint8_t* w, const uint8_t* w_sf, void* out, int rows, int K,
                                       cudaStream_t stream) {
  return fp4gemv_dequantize_rows_padded(w, w_sf, 0, out, rows, K, stream);
}

fp4gemv_status fp4gemv_dequant_gemm(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                    const float* global_scale, void* w_bf16, void* out, int64_t ldo, int M, int N,
                                    int K, int pdl, cudaStream_t stream) {
  if (pdl != 0 && pdl != 1) return FP4GEMV_ERR_INVALID_ARG;
  if (M > FP4GEMV_MAX_M || N % 16 != 0 || K % 256 != 0) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  // Validate the GEMM half first so nothing launches on a bad argument.
  if (M < 1 || ldx < K || ldo < N) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(global_scale, 4) || !aligned(x, 16) || (ldx * 2) % 16 != 0 || !aligned(out, 16) || ldo % 8 != 0 ||
      !aligned(w_bf16, 16))
    return FP4GEMV_ERR_MISALIGNED;
  if (!global_scale || !w_bf16 || !x || !out) return FP4GEMV_ERR_INVALID_ARG;
  fp4gemv_status st = fp4gemv_dequantize_rows(w, w_sf, w_bf16, N, K, stream);
  if (st != FP4GEMV_OK) return st;
  // The GEMM reads the weight the previous launch writes, so it is launched
  // without early weight prefetch.
  (void)pdl;
  return dense_launch(fp4::kDenseBf16, x, ldx, w_bf16, nullptr, global_scale, out, ldo, M, N, K, 0, 0, stream);
}

size_t fp4gemv_w4a4_workspace_bytes(int M, int K) {
  if (M < 1 || K < 1) return 0;
  return (static_cast<size_t>(M) * K * 2 + 15) / 16 * 16;
}

fp4gemv_status fp4gemv_quantize_act(const void* x, int64_t ldx, const float* gsi, uint8_t* x_fp4, uint8_t* x_sf,
                                    void* x_deq, int M, int K, cudaStream_t stream) {
  if (M < 1 || K < 1 || ldx < K) return FP4GEMV_ERR_INVALID_ARG;
  if (K % 16 != 0) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || (ldx * 2) % 16 != 0 || !aligned(x_fp4, 8) || !aligned(gsi, 4) || !aligned(x_deq, 16))
    return FP4GEMV_ERR_MISALIGNED;
  if (!x || !gsi || !x_fp4 || !x_sf) return FP4GEMV_ERR_INVALID_ARG;
  fp4gemv_status st = device_state(nullptr, nullptr);
  if (st != FP4GEMV_OK) return st;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return from_cuda(fp4::launch_quantize_act(x, ldx, gsi, x_fp4, x_sf, x_deq, M, K, 0, stream));
}

namespace {

// The W4A4 GEMM on the exact bf16 dequantisation of the activations (in the
// workspace): the dense NVFP4 GEMM with alpha as its global scale, in
// launches of at most FP4GEMV_MAX_M rows.
fp4gemv_status w4a4_gemm_on(const uint16_t* xd, const uint8_t* w, const uint8_t* w_sf, const float* alpha,
                            void* out, int64_t ldo, int M, int N, int K, int pdl, cudaStream_t stream) {
  for (int m0 = 0; m0 < M; m0 += FP4GEMV_MAX_M) {
    const int mc = std::min(FP4GEMV_MAX_M, M - m0);
    fp4gemv_status st = dense_launch(fp4::kDenseFp4, xd + static_cast<int64_t>(m0) * K, K, w, w_sf, alpha,
                                     static_cast<uint16_t*>(out) + static_cast<int64_t>(m0) * ldo, ldo, mc, N, K, 0,
                                     pdl, stream);
    if (st != FP4GEMV_OK) return st;
  }
  return FP4GEMV_OK;
}

fp4gemv_status w4a4_check(const uint8_t* w, const uint8_t* w_sf, const float* alpha, void* out, int64_t ldo, int M,
                          int N, int K, void* workspace, size_t workspace_bytes, int pdl) {
  if (pdl != 0 && pdl != 1) return FP4GEMV_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldo < N) return FP4GEMV_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % 64 != 0 || K < 256) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < fp4gemv_w4a4_workspace_bytes(M, K)) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(w_sf, 16) || !aligned(out, 16) || ldo % 8 != 0 || !aligned(workspace, 16) ||
      !aligned(alpha, 4))
    return FP4GEMV_ERR_MISALIGNED;
  if (!w || !w_sf || !alpha || !out || !workspace) return FP4GEMV_ERR_INVALID_ARG;
  return FP4GEMV_OK;
}

}  // namespace

fp4gemv_status fp4gemv_w4a4_gemm(const uint8_t* x_fp4, const uint8_t* x_sf, const uint8_t* w, const uint8_t* w_sf,
                                 const float* alpha, void* out, int64_t ldo, int M, int N, int K, void* workspace,
                                 size_t workspace_bytes, int pdl, cudaStream_t stream) {
  fp4gemv_status st = w4a4_check(w, w_sf, alpha, out, ldo, M, N, K, workspace, workspace_bytes, pdl);
  if (st != FP4GEMV_OK) return st;
  if (!aligned(x_fp4, 8)) return FP4GEMV_ERR_MISALIGNED;
  if (!x_fp4 || !x_sf) return FP4GEMV_ERR_INVALID_ARG;
  st = device_state(nullptr, nullptr);
  if (st != FP4GEMV_OK) return st;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  st = from_cuda(fp4::launch_dequantize_act(x_fp4, x_sf, workspace, M, K, stream));
  if (st != FP4GEMV_OK) return st;
  return w4a4_gemm_on(static_cast<const uint16_t*>(workspace), w, w_sf, alpha, out, ldo, M, N, K, pdl, stream);
}

fp4gemv_status fp4gemv_w4a4_linear(const void* x, int64_t ldx, const float* gsi, const uint8_t* w,
                                   const uint8_t* w_sf, const float* alpha, void* out, int64_t ldo, int M, int N,
                                   int K, uint8_t* x_fp4, uint8_t* x_sf, void* workspace, size_t workspace_bytes,
                                   int pdl, cudaStream_t stream) {
  fp4gemv_status st = w4a4_check(w, w_sf, alpha, out, ldo, M, N, K, workspace, workspace_bytes, pdl);
  if (st != FP4GEMV_OK) return st;
  if (ldx < K) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ldx * 2) % 16 != 0 || !aligned(x_fp4, 8) || !aligned(gsi, 4)) return FP4GEMV_ERR_MISALIGNED;
  if (!x || !gsi || !x_fp4 || !x_sf) return FP4GEMV_ERR_INVALID_ARG;
  st = device_state(nullptr, nullptr);
  if (st != FP4GEMV_OK) return st;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  st = from_cuda(fp4::launch_quantize_act(x, ldx, gsi, x_fp4, x_sf, workspace, M, K, pdl, stream));
  if (st != FP4GEMV_OK) return st;
  return w4a4_gemm_on(static_cast<const uint16_t*>(workspace), w, w_sf, alpha, out, ldo, M, N, K, pdl, stream);
}

fp4gemv_status fp4gemv_moe_gate_up(const void* x, const int32_t* ids, int M, int topk, const uint8_t* w1,
                                   const uint8_t* w1_sf, const float* alpha, int E, int H, int I, void* act,
                                   const uint8_t* wsh, const uint8_t* ssh, const float* gssh, int SI, void* sact,
                                   int pdl, cudaStream_t stream) {
  if (pdl != 0 && pdl != 1) return FP4GEMV_ERR_INVALID_ARG;
  if (M < 1 || topk < 1 || E < 1 || H < 1 || I < 1 || SI < 1) return FP4GEMV_ERR_INVALID_ARG;
  if (static_cast<long>(M) * topk > 1024 || H % 64 != 0 || H < 256 || I % 64 != 0 || SI % 64 != 0)
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(w1, 16) || !aligned(w1_sf, 16) || !aligned(wsh, 16) || !aligned(ssh, 16) ||
      !aligned(act, 16) || !aligned(sact, 16) || !aligned(ids, 4) || !aligned(alpha, 4) || !aligned(gssh, 4))
    return FP4GEMV_ERR_MISALIGNED;
  if (!x || !ids || !w1 || !w1_sf || !alpha || !act || !wsh || !ssh || !gssh || !sact) return FP4GEMV_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  int sms = 0;
  fp4gemv_status st = device_state(&err, &sms);
  if (st != FP4GEMV_OK) return st;
  // The slab kernel when it has a plan (plan_slab_moe: up to 64 tokens,
  // split or grouped form); else the register-fed kernel for up to 64
  // tokens: expert chunks hold at most 8 pairs (more pairs routed to one
  // expert form further chunks) and the shared expert runs ceil(M / 8)
  // chunks; the tcgen05 kernel beyond.
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
    int regs = g_slab_moe_regs[dev].load(std::memory_order_acquire);
    if (regs == 0) {
      if (fp4::slab_moe_regs(fp4::kMoeGateUp, &regs) != cudaSuccess || regs <= 0) return FP4GEMV_ERR_CUDA;
      g_slab_moe_regs[dev].store(regs, std::memory_order_release);
    }
    SlabMoePlan sp;
    if (plan_slab_moe(M, topk, E, H, I, SI, sms, regs, &sp)) {
      GemvParams p;
      std::memset(&p, 0, sizeof(p));
      if (!encode_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w1, H / 2, static_cast<uint64_t>(E) * 2 * I, H / 2, 128,
                     128))
        return FP4GEMV_ERR_CUDA;
      if (!encode_2d(&p.tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, wsh, H / 2, 2 * static_cast<uint64_t>(SI), H / 2, 128,
                     64))
        return FP4GEMV_ERR_CUDA;
      p.sf = w1_sf;
      p.sf2 = ssh;
      p.x = static_cast<const uint16_t*>(x);
      p.x2 = p.x;
      p.ldx = p.ldx2 = H;
      p.gs = gssh;
      p.alpha = alpha;
      p.ids = ids;
      p.out = static_cast<uint16_t*>(act);
      p.ldo = I;
      p.out2 = static_cast<uint16_t*>(sact);
      p.ldo2 = SI;
      p.M = M;
      p.n_out = I;
      p.n_half = SI;
      p.K = H;
      p.K2 = H;
      p.k_split = sp.kslab;
      p.E = E;
      p.topk = topk;
      p.P = M * topk;
      p.rows_per_expert = 2 * I;
      p.rows_w = 2 * SI;
      p.shared_n_out = SI;
      p.routed_tiles = I / 64;
      p.shared_tiles = (SI + 63) / 64;
      p.kbp = p.kbp2 = ((H / 16) + 3) / 4 * 4;
      p.sf_expert_bytes = static_cast<uint32_t>(fp4gemv_scale_bytes(2 * I, H));
      p.nstages = sp.nstages;
      p.stage_bytes = sp.stage_bytes;
      p.x_off = sp.slab_bytes;
      p.cw = fp4::kSlabMaxCW;
      p.slab_r = 2;
      p.chunk = sp.chunk;
      p.tiles_per_cta = sp.T;  // 0: the split form
      if (sp.T > 0) p.routed_tiles = p.shared_tiles = sp.groups;  // (grouped: resolve_work's tile is the group)
      p.skip_stage = -1;
      p.err = err;
      LaunchCfg cfg{};
      cfg.grid = dim3(sp.groups, p.P + (M + sp.chunk - 1) / sp.chunk, 1);
      cfg.cluster = sp.S;
      cfg.smem = sp.smem;
      cfg.pdl = pdl;
      cfg.stream = stream;
      g_launches.fetch_add(1, std::memory_order_relaxed);
      return from_cuda(fp4::launch_slab_moe(fp4::kMoeGateUp, p, cfg));
    }
  }
  const bool rf = M <= 64;
  const int kmode = rf ? kMoeGateUpRf : fp4::kMoeGateUp;
  const int NT = rf ? 8 : 32;
  KernelInfo info{};
  if (kernel_info(kmode, NT, &info) != cudaSuccess) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  int nstages = 0, stage_bytes = 0, x_off = 0;
  size_t smem = 0;
  // scale groups per stage: routed tiles one; shared-expert tiles the gate
  // box's and the up box's (SI is a multiple of 64, so neither straddles)
  TcRing tr;
  if (rf) {
    size_ring_rf(info, 128 * 128, 2, &nstages, &smem, &stage_bytes, &x_off);
  } else {
    tr = size_ring(info, true, 2, 1);
    nstages = tr.nstages;
    smem = tr.smem;
  }
  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w1, H / 2, static_cast<uint64_t>(E) * 2 * I, H / 2, 128, 128))
    return FP4GEMV_ERR_CUDA;
  // shared expert: [gate | up] halves read as paired 64-row boxes
  if (!encode_2d(&p.tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, wsh, H / 2, 2 * static_cast<uint64_t>(SI), H / 2, 128, 64))
    return FP4GEMV_ERR_CUDA;
  p.sf = w1_sf;
  p.sf2 = ssh;
  p.x = static_cast<const uint16_t*>(x);
  p.x2 = p.x;
  p.ldx = p.ldx2 = H;
  p.gs = gssh;
  p.alpha = alpha;
  p.ids = ids;
  p.out = static_cast<uint16_t*>(act);
  p.ldo = I;
  p.out2 = static_cast<uint16_t*>(sact);
  p.ldo2 = SI;
  p.M = M;
  p.n_out = I;
  p.n_half = SI;
  p.K = H;
  p.K2 = H;
  p.E = E;
  p.topk = topk;
  p.P = M * topk;
  p.rows_per_expert = 2 * I;
  p.rows_w = 2 * SI;
  p.shared_n_out = SI;
  p.routed_tiles = I / 64;             // one [up; gate] 128-row group (64 features) per tile
  p.shared_tiles = (SI + 63) / 64;     // 64 features per paired tile
  p.kbp = p.kbp2 = ((H / 16) + 3) / 4 * 4;
  p.sf_expert_bytes = static_cast<uint32_t>(fp4gemv_scale_bytes(2 * I, H));
  p.nstages = nstages;
  p.nx = tr.nx;
  p.wstage = tr.wstage;
  p.sf_slots = 2;
  p.inbox_off = tr.inbox_off;
  p.stage_bytes = stage_bytes;
  p.x_off = x_off;
  p.skip_stage = -1;
  p.err = err;
  const int shared_cols = (M + NT - 1) / NT;
  LaunchCfg cfg{};
  cfg.grid = dim3(p.routed_tiles > p.shared_tiles ? p.routed_tiles : p.shared_tiles, p.P + shared_cols, 1);
  cfg.cluster = 1;
  cfg.smem = smem;
  cfg.pdl = pdl;
  cfg.stream = stream;
  return from_cuda(kernel_launch(kmode, NT, p, cfg));
}

size_t fp4gemv_moe_down_combine_workspace_bytes(int M, int topk, int H) {
  if (M < 1 || topk < 1 || H < 1) return 0;
  const size_t counters = ((static_cast<size_t>(H) + 127) / 128 * 8 + 8 + 15) / 16 * 16;  // (+ the work counter)
  const size_t y = (static_cast<size_t>(M) * topk * H * 2 + 15) / 16 * 16;
  const size_t ysh = (static_cast<size_t>(M) * H * 2 + 15) / 16 * 16;
  return counters + y + ysh;
}

fp4gemv_status fp4gemv_moe_down_combine(const void* act, const int32_t* ids, const float* tw, int M, int topk,
                                        const uint8_t* w2, const uint8_t* w2_sf, const float* alpha2, int E, int H,
                                        int I, const void* sact, const uint8_t* wsd, const uint8_t* ssd,
                                        const float* gssd, int SI, void* out, void* workspace,
                                        size_t workspace_bytes, int pdl, cudaStream_t stream) {
  if (pdl != 0 && pdl != 1) return FP4GEMV_ERR_INVALID_ARG;
  if (M < 1 || topk < 1 || E < 1 || H < 1 || I < 1 || SI < 1) return FP4GEMV_ERR_INVALID_ARG;
  if (static_cast<long>(M) * topk > 1024 || H % 64 != 0 || I % 64 != 0 || I < 256 || SI % 64 != 0 || SI < 256)
    return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < fp4gemv_moe_down_combine_workspace_bytes(M, topk, H)) return FP4GEMV_ERR_INVALID_ARG;
  if (!aligned(act, 16) || !aligned(w2, 16) || !aligned(w2_sf, 16) || !aligned(wsd, 16) || !aligned(ssd, 16) ||
      !aligned(sact, 16) || !aligned(out, 16) || !aligned(workspace, 16) || !aligned(ids, 4) || !aligned(tw, 4) ||
      !aligned(alpha2, 4) || !aligned(gssd, 4))
    return FP4GEMV_ERR_MISALIGNED;
  if (!act || !ids || !tw || !w2 || !w2_sf || !alpha2 || !sact || !wsd || !ssd || !gssd || !out || !workspace)
    return FP4GEMV_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  int sms = 0;
  fp4gemv_status st = device_state(&err, &sms);
  if (st != FP4GEMV_OK) return st;
  // Up to 64 tokens the slab kernel when its plan fits (plan_slab_down),
  // then the combine kernel; otherwise (CTAs that would stream fewer than
  // two 256-K stages, or activation rows too long for the slab) the
  // register-fed kernel for up to 64 tokens,
  // chunks of at most 8 pairs (as gate_up), the tcgen05 kernel beyond.  From
  // 8 tokens the register-fed grid holds many short CTAs (K = I is a few
  // stages): the variant budgeted for three CTAs per SM (72 KB ring) hides
  // more of their fixed costs.
  SlabDownPlan sdp;
  bool slab = false;
  if (M <= 64) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4GEMV_ERR_CUDA;
    int regs = g_slab_down_regs[dev].load(std::memory_order_acquire);
    if (regs == 0) {
      if (fp4::slab_moe_regs(fp4::kMoeDown, &regs) != cudaSuccess || regs <= 0) return FP4GEMV_ERR_CUDA;
      g_slab_down_regs[dev].store(regs, std::memory_order_release);
    }
    slab = plan_slab_down(M, topk, E, H, I, SI, sms, regs, &sdp);
  }
  const bool rf = M <= 64;
  const bool occ3 = rf && M >= 8;
  const int kmode = rf ? (occ3 ? kMoeDownRf3 : kMoeDownRf) : fp4::kMoeDown;
  const int NT = rf ? 8 : 32;
  KernelInfo info{};
  if (kernel_info(kmode, NT, &info) != cudaSuccess) return FP4GEMV_ERR_UNSUPPORTED_SHAPE;
  int nstages = 0, stage_bytes = 0, x_off = 0;
  size_t smem = 0;
  TcRing tr;  // one scale group per stage (128-row tiles)
  if (rf) {
    size_ring_rf(info, 128 * 128, 1, &nstages, &smem, &stage_bytes, &x_off, occ3 ? 72 * 1024 : kRfBudget);
  } else {
    tr = size_ring(info, true, 1, 1);
    nstages = tr.nstages;
    smem = tr.smem;
  }
  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_2d(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, I / 2, static_cast<uint64_t>(E) * H, I / 2, 128, 128))
    return FP4GEMV_ERR_CUDA;
  if (!encode_2d(&p.tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, wsd, SI / 2, H, SI / 2, 128, 128)) return FP4GEMV_ERR_CUDA;
  const size_t counters = ((static_cast<size_t>(H) + 127) / 128 * 8 + 8 + 15) / 16 * 16;  // (+ the work counter)
  const size_t ybytes = (static_cast<size_t>(M) * topk * H * 2 + 15) / 16 * 16;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<unsigned long long*>(ws);
  static std::atomic<uint32_t> epoch{0};
  uint32_t ep = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  if (ep == 0) ep = epoch.fetch_add(1, std::memory_order_relaxed) + 1;  // 0 is the reset value
  p.epoch = ep;
  p.out = reinterpret_cast<uint16_t*>(ws + counters);
  p.ldo = H;
  p.out2 = reinterpret_cast<uint16_t*>(ws + counters + ybytes);
  p.ldo2 = H;
  p.out3 = static_cast<uint16_t*>(out);
  p.sf = w2_sf;
  p.sf2 = ssd;
  p.x = static_cast<const uint16_t*>(act);
  p.ldx = I;
  p.x2 = static_cast<const uint16_t*>(sact);
  p.ldx2 = SI;
  p.gs = gssd;
  p.alpha = alpha2;
  p.ids = ids;
  p.tw = tw;
  p.M = M;
  p.n_out = H;
  p.shared_n_out = H;
  p.K = I;
  p.K2 = SI;
  p.E = E;
  p.topk = topk;
  p.P = M * topk;
  p.rows_per_expert = H;
  p.rows_w = H;
  p.routed_tiles = (H + 127) / 128;
  p.shared_tiles = p.routed_tiles;
  p.kbp = ((I / 16) + 3) / 4 * 4;
  p.kbp2 = ((SI / 16) + 3) / 4 * 4;
  p.sf_expert_bytes = static_cast<uint32_t>(fp4gemv_scale_bytes(H, I));
  p.nstages = nstages;
  p.nx = tr.nx;
  p.wstage = tr.wstage;
  p.sf_slots = 1;
  p.inbox_off = tr.inbox_off;
  p.stage_bytes = stage_bytes;
  p.x_off = x_off;
  p.skip_stage = -1;
  p.err = err;
  if (slab) {
    p.skip_stage = g_skip_stage.load(std::memory_order_relaxed);  // (test hook)
    p.nstages = sdp.nstages;
    p.stage_bytes = sdp.stage_bytes;
    p.x_off = sdp.slab_bytes;
    p.cw = fp4::kSlabMaxCW;
    p.slab_r = 2;
    p.tiles_per_cta = sdp.T;
    p.chunk = sdp.chunk;
    p.routed_tiles = p.shared_tiles = sdp.groups;  // (slab grid: a CTA's first tile is blockIdx.x * T)
    const int ncols = p.P + (M + sdp.chunk - 1) / sdp.chunk;
    const long items = static_cast<long>(sdp.groups) * ncols;
    LaunchCfg cfg{};
    cfg.grid = sdp.persist ? dim3(static_cast<unsigned>(std::min<long>(items, static_cast<long>(sdp.occ) * sms)), 1, 1)
                           : dim3(sdp.groups, ncols, 1);
    cfg.cluster = 1;
    cfg.smem = sdp.smem;
    cfg.pdl = pdl;
    cfg.stream = stream;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    st = from_cuda(sdp.persist ? fp4::launch_moe_down_persist(p, cfg) : fp4::launch_slab_moe(fp4::kMoeDown, p, cfg));
    if (st != FP4GEMV_OK) return st;
    // The combine runs as a kernel of its own, launched early (PDL) and
    // waiting for the slab grid: measured, the slab CTAs' per-tile arrival
    // (fence, counter, the last CTA's combine) cost 20 % of the call.
    const long citems = static_cast<long>(M) * (H / 8);
    LaunchCfg ccfg{};
    ccfg.grid = dim3(static_cast<unsigned>(std::min<long>((citems + 127) / 128, 4L * sms)), 1, 1);
    ccfg.cluster = 1;
    ccfg.smem = 0;
    ccfg.pdl = 1;
    ccfg.stream = stream;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return from_cuda(fp4::launch_moe_combine(p, ccfg));
  }
  const int shared_cols = (M + NT - 1) / NT;
  LaunchCfg cfg{};
  cfg.grid = dim3(p.routed_tiles, p.P + shared_cols, 1);
  cfg.cluster = 1;
  cfg.smem = smem;
  cfg.pdl = pdl;
  cfg.stream = stream;
  return from_cuda(kernel_launch(kmode, NT, p, cfg));
}

fp4gemv_status fp4gemv_get_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FP4GEMV_ERR_CUDA;
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, fp4::g_dev_state, sizeof(v)) != cudaSuccess) return FP4GEMV_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(fp4::g_dev_state, &zero, sizeof(zero)) != cudaSuccess) return FP4GEMV_ERR_CUDA;
  if (v & fp4::FP4_ERR_TIMEOUT) return FP4GEMV_ERR_TIMEOUT;
  if (v & fp4::FP4_ERR_BADIDX) return FP4GEMV_ERR_BAD_INDEX;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns;
  if (cudaMemcpyToSymbol(fp4::g_dev_state, &v, sizeof(v), offsetof(fp4::DeviceErrorState, wait_limit_ns)) !=
      cudaSuccess)
    return FP4GEMV_ERR_CUDA;
  return FP4GEMV_OK;
}

fp4gemv_status fp4gemv_debug_skip_stage(int stage) {
  if (stage < -1) return FP4GEMV_ERR_INVALID_ARG;
  g_skip_stage.store(stage, std::memory_order_relaxed);
  return FP4GEMV_OK;
}

const char* fp4gemv_status_string(fp4gemv_status s) {
  switch (s) {
    case FP4GEMV_OK: return "FP4GEMV_OK";
    case FP4GEMV_ERR_INVALID_ARG: return "FP4GEMV_ERR_INVALID_ARG";
    case FP4GEMV_ERR_UNSUPPORTED_SHAPE: return "FP4GEMV_ERR_UNSUPPORTED_SHAPE";
    case FP4GEMV_ERR_MISALIGNED: return "FP4GEMV_ERR_MISALIGNED";
    case FP4GEMV_ERR_CUDA: return "FP4GEMV_ERR_CUDA";
    case FP4GEMV_ERR_TIMEOUT: return "FP4GEMV_ERR_TIMEOUT";
    case FP4GEMV_ERR_BAD_INDEX: return "FP4GEMV_ERR_BAD_INDEX";
  }
  return "FP4GEMV_ERR_UNKNOWN";
}

uint64_t fp4gemv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
