// ggrn_api.cu -- the C ABI declared in include/ggrn.h: argument validation,
// kernel-family selection, launch, decode graphs and status strings.
//
// Selection follows the shape and the layout, the way the ONNX-contrib
// README's implementation variants are picked per call from device
// capabilities, shapes and dtypes ("com.microsoft.GatedRMSNorm" README,
// Implementation variants); here every family runs on every sm_103a device,
// so only the shape and the alignment decide.  A group size that is not a
// multiple of the warp or of the vector width needs no special contract
// ("gated_group_rmsnorm" Mojo module page, Parallelization).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/ggrn.h"
#include "ggrn_internal.h"
#include "ggrn_slots.h"

// Device status word of the library (one per device): kernels whose bounded
// waits run out set bits here (see ggrn_fault_status).
__device__ unsigned int g_ggrn_fault;

// Unit-claim words of the streaming kernel's dynamic schedule (epoch << 32 |
// next unit; see claim_resolve).  The host gives each word to one running
// launch at a time (ggrn_slots.h: launches of one stream share a word, a word
// passes to another stream once its last launch there has completed, and a
// launch that finds none free takes the static schedule).  Zero (epoch 0,
// never given to a launch) at module load.
constexpr int kSchedSlots = 64;
// Claimed indices are 32-bit: larger launches take the static schedule.
constexpr int64_t kMaxClaimUnits = int64_t{1} << 30;
__device__ unsigned long long g_ggrn_sched[kSchedSlots];

namespace ggrn {
namespace {

// The CUDA error behind the last GGRN_ERR_CUDA of this thread.
thread_local cudaError_t tl_last_cuda_error = cudaSuccess;

// Address of this device's status word (looked up once per device).
unsigned int* fault_word() {
  static std::mutex mu;
  static unsigned int* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_ggrn_fault) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(ptr);
  }
  return cache[dev];
}

// Address of this device's claim words (looked up once per device).
unsigned long long* sched_words() {
  static std::mutex mu;
  static unsigned long long* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_ggrn_sched) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned long long*>(ptr);
  }
  return cache[dev];
}

// Ownership of the claim words of one device (see ggrn_slots.h): the stream
// of each word's last launch and an event recorded after it.
struct SlotTable {
  std::mutex mu;
  ClaimSlot slot[kSchedSlots];
  cudaEvent_t ev[kSchedSlots] = {};
  unsigned next = 0;
};

// Has the launch behind a slot's event completed?  A query that finds it
// still running reports cudaErrorNotReady, which the runtime also keeps as
// the thread's last error: that is cleared again, and a query is not made
// while an earlier error is pending (it stays for the caller to read).
bool slot_done(cudaEvent_t ev) {
  if (!ev || cudaPeekAtLastError() != cudaSuccess) return false;
  const cudaError_t q = cudaEventQuery(ev);
  if (q == cudaErrorNotReady) cudaGetLastError();
  return q == cudaSuccess;
}

SlotTable* slot_table() {
  static SlotTable tables[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  return &tables[dev];
}

// A new claim epoch per launch (nonzero; wraps after 2^32 - 1 launches).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e;
  do {
    e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  } while (e == 0);
  return e;
}

constexpr int kDefaultSMs = 152;
constexpr int kTeamBlock = 256;
constexpr int kTeamMaxVec = 128;     // TEAM covers groups of up to 128 vectors
constexpr int kWideVpl = 4;
constexpr int kWideMaxThreads = 1024;
// automatic selection takes WIDE_CLUSTER for groups of at least this many
// 16-byte vectors when every CTA of every cluster fits on the GPU at once
constexpr int64_t kWideClusterAutoVecs = 256;
constexpr int kStraddleMaxVpl = 4;   // chunk of at most 128 vectors per warp
constexpr int kStraddleBlock = 256;
constexpr int kScalarBlock = 256;
constexpr int64_t kMaxGrid = 0x7fffffff;
constexpr int kStreamWarps = 8;  // consumer warps per CTA (target)
constexpr int64_t kStreamSmemPerSM = 226 * 1024;  // shared memory the CTAs of one SM share
// Ring stages (at most; the shared-memory budget may allow fewer).
constexpr int64_t kStreamMaxStages = 2;
constexpr int64_t kStreamMinUnitsPerSlot = 12;        // units per CTA slot to stream (see plan_stream)
constexpr int64_t kStreamMinUnitsPerSlot32 = 6;       // 32-lane teams, one group each
constexpr int64_t kStreamMinUnitsPerSlotNarrow = 36;  // teams of at most 4 lanes, one group each
constexpr int64_t kStreamMinUnitsPerSlotPaired = 3;   // paired 4 x 7 teams
constexpr int64_t kStreamMaxWeightBytes = 64 * 1024;

int elem_size(int dtype) { return dtype == kF32 ? 4 : 2; }

int sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();  // clear the "no device" error this query may set
    return kDefaultSMs;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = kDefaultSMs;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Byte extent of a [rows, width] matrix with row stride `stride` elements;
// false when it does not fit in int64.
bool extent_bytes(int64_t rows, int64_t width, int64_t stride, int es, int64_t* out) {
  if (rows == 0) {
    *out = 0;
    return true;
  }
  __int128 n = static_cast<__int128>(rows - 1) * stride + width;
  n *= es;
  if (n > static_cast<__int128>(INT64_MAX)) return false;
  *out = static_cast<int64_t>(n);
  return true;
}

bool ranges_overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  if (na == 0 || nb == 0) return false;
  uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

// Checks shared by every entry point (pointers are only checked when rows > 0).
// `out_optional`: ggrn_plan accepts out == NULL (an output not allocated yet).
int validate(const Args& a, bool out_optional = false) {
  if (a.dtype != kF32 && a.dtype != kF16 && a.dtype != kBF16) return GGRN_ERR_DTYPE;
  if (a.mode != kMamba2 && a.mode != kOnnx) return GGRN_ERR_DTYPE;
  if (a.mode == kOnnx && a.dtype == kBF16) return GGRN_ERR_DTYPE;
  if (a.rows < 0 || a.width <= 0 || a.gs <= 0 || a.width % a.gs != 0) return GGRN_ERR_SHAPE;
  if (a.rows > 1 && (a.ys < a.width || a.gts < a.width || a.os < a.width)) return GGRN_ERR_SHAPE;
  if (a.rows == 0) return GGRN_OK;
  const int es = elem_size(a.dtype);
  int64_t ny, ng, no;
  const int64_t ys = a.rows > 1 ? a.ys : a.width, gts = a.rows > 1 ? a.gts : a.width,
                os = a.rows > 1 ? a.os : a.width;
  if (!extent_bytes(a.rows, a.width, ys, es, &ny) || !extent_bytes(a.rows, a.width, gts, es, &ng) ||
      !extent_bytes(a.rows, a.width, os, es, &no))
    return GGRN_ERR_SHAPE;
  if (a.rows > INT64_MAX / (a.width / a.gs)) return GGRN_ERR_SHAPE;
  if (!a.y || !a.gate || !a.w || (!a.out && !out_optional)) return GGRN_ERR_NULL;
  const int wes = a.mode == kMamba2 ? 4 : es;
  if (!aligned(a.y, es) || !aligned(a.gate, es) || !aligned(a.out, es) || !aligned(a.w, wes))
    return GGRN_ERR_ALIGN;
  if (!a.out) return GGRN_OK;
  const int64_t nw = (a.mode == kMamba2 ? a.width : a.gs) * wes;
  if (ranges_overlap(a.out, no, a.y, ny) || ranges_overlap(a.out, no, a.gate, ng) ||
      ranges_overlap(a.out, no, a.w, nw))
    return GGRN_ERR_OVERLAP;
  return GGRN_OK;
}

// May the 16-byte vector families load this call's buffers?
bool vector_layout_ok(const Args& a) {
  const int es = elem_size(a.dtype);
  if (!aligned(a.y, 16) || !aligned(a.gate, 16) || !aligned(a.out, 16) || !aligned(a.w, 16))
    return false;
  if (a.rows > 1 &&
      ((a.ys * es) % 16 != 0 || (a.gts * es) % 16 != 0 || (a.os * es) % 16 != 0))
    return false;
  return true;
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Multiplier for the kernels' floor(item / d) (see div_by in
// ggrn_kernels.cuh): floor(2^64 / d) + 1, valid while every item index is
// below 2^32; 0 (plain division) otherwise or for d < 2.
uint64_t div_magic(int64_t items, int64_t d) {
  if (d < 2 || items > static_cast<int64_t>(UINT32_MAX)) return 0;
  return UINT64_MAX / static_cast<uint64_t>(d) + 1;
}

// One item (a group, or a pair of groups) per team; grid capped at the
// launch limit (the kernels stride over the remaining items).
int plan_team(const Args& a, Plan* p) {
  const int es = elem_size(a.dtype);
  const int E = 16 / es;
  int Q = 1;
  if (a.gs % E != 0) {
    // groups of an odd number of half vectors go in pairs (whole vectors),
    // when the row holds an even number of them
    if ((2 * a.gs) % E != 0 || (a.width / a.gs) % 2 != 0) return GGRN_ERR_UNSUPPORTED;
    Q = 2;
  }
  const int64_t nvec = Q * a.gs / E;
  if (nvec > kTeamMaxVec || (Q == 2 && nvec < 4)) return GGRN_ERR_UNSUPPORTED;
  p->path = kTeam;
  p->elems_per_vec = E;
  p->items_groups = Q;
  p->nvec = static_cast<int>(nvec);
  // Four vectors per lane (fewer for tiny groups) and as many lanes as that
  // needs: the per-item costs (indexing, butterfly, normaliser) then spread
  // over at least 32 elements per lane, and a warp serves 32/lanes items.
  p->vpl = nvec >= 4 ? 4 : next_pow2(static_cast<int>(nvec));
  p->lanes = next_pow2(static_cast<int>(ceil_div(nvec, p->vpl)));
  p->groups = a.width / a.gs;
  p->items_per_row = p->groups / Q;
  p->items = a.rows * p->items_per_row;
  p->div_magic = div_magic(p->items, p->items_per_row);
  // Spread small problems over the SMs: shrink the block (down to one warp)
  // while that keeps the grid under one CTA per SM.
  const int sms = sm_count();
  int block = kTeamBlock;
  const int64_t per_warp = 32 / p->lanes;
  while (block > 32 && ceil_div(p->items, (block / 32) * per_warp) < sms) block /= 2;
  p->block = block;
  p->grid = std::min<int64_t>(kMaxGrid, std::max<int64_t>(1, ceil_div(p->items, (block / 32) * per_warp)));
  if (p->items == 0) p->grid = 0;
  p->smem = 0;
  return GGRN_OK;
}

// WIDE: one CTA per group, `vpl` vectors per thread (4 for throughput; 1, 2
// or 4 for launches with few groups, where the per-thread latency decides).
int plan_wide(const Args& a, Plan* p, int vpl = kWideVpl) {
  const int es = elem_size(a.dtype);
  const int E = 16 / es;
  if (a.gs % E != 0) return GGRN_ERR_UNSUPPORTED;
  const int64_t nvec = a.gs / E;
  const int64_t threads = ceil_div(ceil_div(nvec, vpl), 32) * 32;
  if (threads > kWideMaxThreads) return GGRN_ERR_UNSUPPORTED;
  p->path = kWide;
  p->elems_per_vec = E;
  p->nvec = static_cast<int>(nvec);
  p->lanes = static_cast<int>(threads);
  p->vpl = vpl;
  p->block = static_cast<int>(threads);
  p->groups = a.width / a.gs;
  p->items = a.rows * p->groups;
  p->div_magic = div_magic(p->items, p->groups);
  p->grid = std::min<int64_t>(kMaxGrid, p->items);
  p->smem = 0;
  return GGRN_OK;
}

// Vectors per thread of WIDE: 1 up to two groups per SM, 2 up to four, then
// 4, as the CTA size limit allows (5120-wide groups: at 256 rows 1 vector per
// thread 1.98 TB/s against 1.57 with 4; at 1024 rows 4 is best).  One vector
// per thread stops at 640 threads: a lone 7680-wide group (batch-1 decode
// with one group) takes 2.34 us per call in a 21-call graph with 480 threads
// of 2 vectors against 2.59 with 960 of 1, while a lone 5120-wide group is
// faster with 640 threads of 1 (2.05 against 2.15).
constexpr int64_t kWideOneVecMaxThreads = 640;
int wide_vpl(const Args& a, int64_t items, int64_t sms) {
  const int64_t nvec = a.gs / (16 / elem_size(a.dtype));
  int v = items <= 2 * sms ? 1 : (items <= 4 * sms ? 2 : 4);
  if (v == 1 && nvec > kWideOneVecMaxThreads) v = 2;
  while (v < 4 && ceil_div(nvec, v) > kWideMaxThreads) v *= 2;
  return v;
}

// WIDE_CLUSTER: a cluster of CTAs per group, one 16-byte vector per thread;
// up to kWideClusterMax CTAs of about kWideClusterVecs vectors each.
// (Measured on lone 2048..7680-wide bf16 groups: 2 or 4 CTAs of 256..512
// threads, and 16-CTA clusters of 64 or 96 threads, were no faster.)
constexpr int kWideClusterMax = 8;     // the portable cluster size
constexpr int kWideClusterVecs = 128;  // vectors per CTA sought
int plan_wide_cluster(const Args& a, Plan* p) {
  const int es = elem_size(a.dtype);
  const int E = 16 / es;
  if (a.gs % E != 0) return GGRN_ERR_UNSUPPORTED;
  const int64_t nvec = a.gs / E;
  if (nvec < 2) return GGRN_ERR_UNSUPPORTED;
  const int64_t cn = std::max<int64_t>(
      2, std::min<int64_t>(kWideClusterMax, ceil_div(nvec, kWideClusterVecs)));
  const int64_t per = ceil_div(nvec, cn);
  const int64_t threads = ceil_div(per, 32) * 32;
  // the kernel has 32 slots: one per warp of the cluster
  if (cn * (threads / 32) > 32) return GGRN_ERR_UNSUPPORTED;
  p->path = kWideCluster;
  p->elems_per_vec = E;
  p->nvec = static_cast<int>(nvec);
  p->vpl = 1;
  p->lanes = static_cast<int>(threads);
  p->block = static_cast<int>(threads);
  p->cluster_ctas = static_cast<int>(cn);
  p->cluster_vecs = static_cast<int>(per);
  p->groups = a.width / a.gs;
  p->items = a.rows * p->groups;
  p->div_magic = div_magic(p->items, p->groups);
  if (p->items > kMaxGrid / cn) return GGRN_ERR_UNSUPPORTED;
  p->grid = p->items * cn;
  p->smem = 0;
  return GGRN_OK;
}

int plan_straddle(const Args& a, Plan* p) {
  const int es = elem_size(a.dtype);
  const int E = 16 / es;
  // whole vectors only: group size above the vector and not a multiple of
  // it, width a multiple of it (rows then start and end on vector bounds)
  if (a.gs % E == 0 || a.gs < E || a.width % E != 0) return GGRN_ERR_UNSUPPORTED;
  const int64_t g = gcd64(a.gs, E);
  const int64_t lcm = a.gs / g * E;                 // elements per period
  const int64_t period_vecs = lcm / E;
  if (period_vecs > 32 * kStraddleMaxVpl) return GGRN_ERR_UNSUPPORTED;
  // Choose vectors per lane and periods per chunk (one warp per chunk) for
  // the best use of the warp's 32*VPL vector slots over a row.
  const int64_t row_vecs = ceil_div(a.width, E);
  const int64_t periods_per_row = ceil_div(a.width, lcm);
  double best = -1.0;
  int best_vpl = 0;
  int64_t best_k = 0;
  for (int vpl = 1; vpl <= kStraddleMaxVpl; vpl *= 2) {
    const int64_t slots = 32 * vpl;
    const int64_t kmax = std::min<int64_t>(slots / period_vecs, periods_per_row);
    for (int64_t k = 1; k <= kmax; ++k) {
      const int64_t chunks = ceil_div(periods_per_row, k);
      const double use = static_cast<double>(row_vecs) / static_cast<double>(chunks * slots);
      if (use > best + 1e-9) {
        best = use;
        best_vpl = vpl;
        best_k = k;
      }
    }
  }
  if (best_vpl == 0) return GGRN_ERR_UNSUPPORTED;
  p->path = kStraddle;
  p->elems_per_vec = E;
  p->vpl = best_vpl;
  p->straddle_g = static_cast<int>(g);
  p->chunk_elems = best_k * lcm;
  p->chunks_per_row = ceil_div(a.width, p->chunk_elems);
  p->chunk_groups = static_cast<int>(std::min<int64_t>(p->chunk_elems, a.width) / a.gs);
  p->nvec = static_cast<int>(ceil_div(std::min<int64_t>(p->chunk_elems, a.width), E));
  p->gs_magic = static_cast<uint32_t>((uint64_t{1} << 32) / static_cast<uint64_t>(a.gs) + 1);
  p->warp_smem = 2 * 32 * best_vpl + p->chunk_groups;
  p->block = kStraddleBlock;
  p->lanes = 32;
  p->groups = a.width / a.gs;
  p->items = a.rows * p->chunks_per_row;
  p->div_magic = div_magic(p->items, p->chunks_per_row);
  const int64_t warps = kStraddleBlock / 32;
  p->grid = std::min<int64_t>(kMaxGrid, ceil_div(p->items, warps));
  p->smem = static_cast<int>(warps * p->warp_smem * sizeof(float));
  return GGRN_OK;
}

int plan_scalar(const Args& a, Plan* p) {
  p->path = kScalar;
  p->elems_per_vec = 1;
  p->vpl = 1;
  p->lanes = a.gs <= 16 ? 1 : 32;
  p->groups = a.width / a.gs;
  p->items = a.rows * p->groups;
  p->div_magic = div_magic(p->items, p->groups);
  p->block = kScalarBlock;
  const int64_t teams_per_block = (kScalarBlock / 32) * (32 / p->lanes);
  p->grid = std::min<int64_t>(kMaxGrid, ceil_div(p->items, teams_per_block));
  p->smem = 0;
  p->nvec = 0;
  return GGRN_OK;
}

// Shared memory of the streaming kernels: choose CTAs per SM (2, else 1) and
// ring stages (2..max_stages) for stage slots of `stage_bytes`, staging the
// weight (`wb` bytes) when it is a 16-byte multiple and leaves room for the
// ring.  False when not even two stages fit.
bool stream_smem(int64_t stage_bytes, int64_t wb, int64_t wpad, int64_t max_stages, int* cps,
                 int* ns, int64_t* wstage) {
  *cps = 0;
  *ns = 0;
  *wstage = 0;
  for (int staged = 1; staged >= 0 && *ns < 2; --staged) {
    const int64_t warea = staged ? ceil_div(wb + wpad, 128) * 128 : 0;
    if (staged && (wb % 16 != 0 || wb > kStreamMaxWeightBytes)) continue;
    for (int c = 2; c >= 1; --c) {
      const int64_t budget = kStreamSmemPerSM / c - 1024 - warea - 512;
      const int64_t n = std::min<int64_t>(max_stages, budget / (2 * stage_bytes));
      if (n >= 2) {
        *cps = c;
        *ns = static_cast<int>(n);
        *wstage = staged ? wb : 0;
        break;
      }
    }
  }
  return *ns >= 2;
}

// Size of the short first unit of each CTA slot of a streaming launch
// (groups for flat units, rows for row units; 0: none).  A first stage of
// fewer bytes lands sooner, so compute starts sooner while the ring fills.
// Measured over 3 x 400 launches (GB/s, each within 0.1 %): flat units, half
// the unit: prefill 960-wide groups 5914 -> 5970, gated-DeltaNet heads 6934
// -> 6944; row units, one row fewer: odd span 6372 -> 6390 (half: 6370).
// Shorter last units as well were slower everywhere (prefill 5751).
int64_t stream_head_size(int mode, int64_t mid, int Q) {
  const int64_t hs = mode == 0 ? (mid / 2) / Q * Q : mid - 1;
  return hs > 0 && hs < mid ? hs : 0;
}

// STREAM: persistent CTAs fed by bulk copies of row chunks ("units" of ug
// whole groups).  A team takes an item of Q groups: Q = 1 when a group's
// bytes are a multiple of 16 (or of 8, with 8-byte shared-memory vectors),
// Q = 2 when they are an odd multiple of 8 (a pair of groups is then whole
// 16-byte vectors).  Eligible when an item spans 4..128 shared-memory
// vectors, every unit is a 16-byte multiple, and (unless forced) there are
// enough units per CTA slot (kStreamMinUnitsPerSlot and its variants).
int plan_stream(const Args& a, Plan* p, bool forced, bool one_cta = false) {
  // the consumers place groups within a unit in 32-bit arithmetic
  if (a.width >= (int64_t{1} << 30)) return GGRN_ERR_UNSUPPORTED;
  const int es = elem_size(a.dtype);
  const int64_t gbytes = a.gs * es;
  int sv = 0, Q = 1;
  if (gbytes % 16 == 0) {
    sv = 16;
  } else if (gbytes % 8 == 0) {
    sv = 16;
    Q = 2;
  } else {
    return GGRN_ERR_UNSUPPORTED;
  }
  const int se = sv / es;
  const int64_t nvec = Q * a.gs / se;     // vectors per item
  if (nvec < 4 || nvec > 128) return GGRN_ERR_UNSUPPORTED;
  int lanes = next_pow2(static_cast<int>(ceil_div(nvec, 4)));
  int vpl = 4;
  // Consumer warps and ring depth by team width, from a sweep of 4-16 warps,
  // 1-2 CTAs per SM and 2-4 stages over groups of 64..960 elements (claimed
  // units): narrow groups (teams of at most 4 lanes) run best with 6 warps
  // and three stages, two CTAs per SM (+1.5 to 1.9 % at 64 and 128); 8- and
  // 16-lane teams with 8 warps and two stages.  One group per warp (32-lane
  // teams) ran best with 16 warps and three stages in one CTA per SM until
  // the consumer loop lost a fifth of its instructions; since then 8 warps
  // and two stages in each of two CTAs per SM (two independent rings, the
  // weight staged in each) measure faster on the 960-wide prefill groups:
  // 6271 -> 6305 GB/s at 4096 rows, 6633 -> 6767 at 8192, 7125 -> 7225 at
  // 32768 (alternating runs on one box; not staging the weight: 6056 at 4096).
  // Where two such CTAs do not fit on an SM (wide rows, whose staged weight
  // is large), the one-CTA shape is planned instead (`one_cta`, below).
  int target_warps = kStreamWarps;
  int64_t max_stages = kStreamMaxStages;
  const bool wide_team = Q == 1 && lanes == 32;
  if (wide_team && one_cta) {
    target_warps = 16;
    max_stages = 3;
  } else if (Q == 1 && lanes <= 4) {
    target_warps = 6;
    max_stages = 3;
  }
  if (Q == 2 && nvec > 16 && nvec <= 28) {
    // a pair of 17..28 vectors (25 for the 100-wide bf16 odd span): 4 lanes x
    // 7 vectors leave fewer slots idle than 8 x 4 (28 vs 32 for 25).  With
    // the earlier, longer consumer loop as many consumer warps as the
    // registers allow in one CTA per SM hid the per-lane latency best (odd
    // span: 15 warps 6.42 TB/s, 12 warps 6.03); with the current one, 6
    // warps in each of two CTAs per SM (two rings of two-row units) measure
    // faster: 7101 -> 7148 GB/s at 65536 rows, 6559 -> 6718 at 16384
    // (alternating runs on one box)
    lanes = 4;
    vpl = 7;
    target_warps = one_cta ? stream_max_warps(a.mode, vpl) : 6;
  }
  const bool paired7 = vpl == 7;
  const int wmax = stream_max_warps(a.mode, vpl);
  const int64_t gpw = (32 / lanes) * Q;   // groups per warp pass
  const int64_t gpr = a.width / a.gs;
  const int64_t total = a.rows * gpr;
  if (gpr % Q != 0) return GGRN_ERR_UNSUPPORTED;  // items never cross a row
  const bool flat = a.rows <= 1 || (a.ys == a.width && a.gts == a.width && a.os == a.width);
  int W = 0, mode = 0;
  int64_t ug = 0, units = 0, upr = 0, rpu = 0;
  if (flat) {
    // consecutive groups of the contiguous [rows * width] data
    mode = 0;
    W = target_warps;
    ug = W * gpw;
    units = ceil_div(total, ug);
    const int64_t last = total - (units - 1) * ug;
    if ((ug * gbytes) % 16 != 0 || (last * gbytes) % 16 != 0) return GGRN_ERR_UNSUPPORTED;
  } else {
    // units inside a row: ug = W * gpw must divide the row's groups
    for (int w = 4; w <= wmax; ++w) {
      const int64_t u = w * gpw;
      if (gpr % u != 0 || (u * gbytes) % 16 != 0) continue;
      if (W == 0 || std::abs(w - target_warps) <= std::abs(W - target_warps)) W = w;
    }
    if (W != 0) {
      mode = 1;
      ug = W * gpw;
      upr = gpr / ug;
      units = a.rows * upr;
    } else {
      // short rows: whole rows per unit, each row copied on its own
      if ((a.width * es) % 16 != 0) return GGRN_ERR_UNSUPPORTED;
      mode = 2;
      rpu = std::max<int64_t>(1, (target_warps * gpw) / gpr);
      W = static_cast<int>(ceil_div(rpu * gpr, gpw));
      if (W > wmax) return GGRN_ERR_UNSUPPORTED;
      ug = rpu * gpr;
      units = ceil_div(a.rows, rpu);
    }
  }
  const uint32_t stage_bytes = static_cast<uint32_t>(ceil_div(ug * gbytes, 128) * 128);
  // The weight is staged in shared memory once per CTA when its bytes are a
  // 16-byte multiple and it leaves room for the ring.
  const int64_t wb = a.mode == kMamba2 ? a.width * 4 : a.gs * es;
  // MAMBA2 consumers read the staged weight for every slot of a team, also
  // the slots past the last item's vectors (their results are not stored),
  // up to (vpl * lanes - nvec) vectors of f32 columns beyond the row's end:
  // the weight area is that much longer
  const int64_t wpad = a.mode == kMamba2 ? (int64_t{vpl} * lanes - nvec) * se * 4 : 0;
  int cps, ns;
  int64_t wstage;
  if (!stream_smem(stage_bytes, wb, wpad, max_stages, &cps, &ns, &wstage))
    return GGRN_ERR_UNSUPPORTED;
  const int64_t warea = wstage ? ceil_div(wstage + wpad, 128) * 128 : 0;
  // the two-CTA shapes of 32-lane teams and 4 x 7 pairs need both CTAs on an
  // SM: with one, the SM would run only their 6-8 consumer warps
  if (!one_cta && (wide_team || paired7) && cps < 2) return plan_stream(a, p, forced, true);
  const int64_t gmax = static_cast<int64_t>(sm_count()) * cps;
  // Automatic selection streams only with enough units per CTA slot: below
  // that the ring's fill and drain cost more than the register-resident TEAM
  // kernel loses.  Measured crossovers (TEAM vs STREAM, GB/s, forced and
  // automatic sweeps on one box): 960-wide prefill groups, 32-lane teams in
  // two CTAs per SM, 6 per slot (1536 rows 4926 vs 4828, 1824 rows 5280 vs
  // 5336, 2128 rows 5396 vs 5520, 3040 rows 5786 vs 5801); 128-wide fp16
  // heads, 4-lane teams, 36 per slot (8192 rows 6355 vs 6248, 16384 rows
  // 6790 vs 6800, 24576 rows 6923 vs 7002); the odd span's paired 4 x 7
  // teams in two CTAs per SM, 3 per slot (1520 rows 4017 vs 3690, 2048 rows
  // 4057 vs 4417, 4096 rows 4730 vs 5390); other team widths 12 per slot.
  int64_t min_per_slot = kStreamMinUnitsPerSlot;
  if (Q == 1 && lanes == 32) min_per_slot = kStreamMinUnitsPerSlot32;
  if (Q == 1 && lanes <= 4) min_per_slot = kStreamMinUnitsPerSlotNarrow;
  if (Q == 2 && vpl == 7) min_per_slot = kStreamMinUnitsPerSlotPaired;
  if (!forced && units < min_per_slot * gmax) return GGRN_ERR_UNSUPPORTED;
  // static schedule: equal units per CTA, so the last wave ends together
  const int64_t per_cta = ceil_div(units, gmax);
  p->path = kStream;
  p->elems_per_vec = se;
  p->smem_vec_bytes = sv;
  p->items_groups = Q;
  p->nvec = static_cast<int>(nvec);
  p->vpl = vpl;
  p->lanes = lanes;
  p->consumer_warps = W;
  p->ug = static_cast<int>(ug);
  p->units_per_row = upr;
  p->unit_mode = mode;
  p->rows_per_unit = static_cast<int>(rpu);
  p->total_groups = total;
  p->groups = gpr;
  p->items = units;
  p->stage_bytes = stage_bytes;
  p->stages = ns;
  p->ctas_per_sm = cps;
  // dynamic schedule (claimed units): every CTA slot of the device
  p->grid = std::min(units, gmax);
  p->grid_static = ceil_div(units, per_cta);
  p->block = (W + 1) * 32;
  p->w_smem_bytes = static_cast<uint32_t>(wstage);
  p->w_area_bytes = static_cast<uint32_t>(warea);
  // ring, weight, a 16-byte zero block, barriers full/empty/weight/permute,
  // unit of each stage and its placement
  p->smem = static_cast<int>(2 * static_cast<int64_t>(ns) * stage_bytes + warea + 16 +
                             8 * (2 * ns + 2) + 8 * ns + 16 * ns);
  p->div_magic = mode == 1 ? div_magic(units, upr) : 0;
  p->div_magic2 = div_magic(total, gpr);
  // a group's row past its unit's first row is floor(c / gpr) for the
  // group's index c from that row's start, c < gpr + ug; one multiply-high
  // gives it exactly while (gpr + ug) * gpr < 2^32 (div_small)
  p->groups_magic = (gpr >= 2 && (gpr + ug) * gpr < (int64_t{1} << 32))
                        ? static_cast<uint32_t>((uint64_t{1} << 32) / static_cast<uint64_t>(gpr) + 1)
                        : 0;
  // Teams of 4 lanes, 8 to a warp: an 8-lane phase of a shared-memory load
  // holds two teams, each reading 4 consecutive 16-byte slots of its item.
  // Consecutive items start d slots apart (mod the 8 slots of a 128-byte
  // bank row); two teams on items d apart overlap unless d = 4.  So the
  // teams sharing a phase take items 4 apart (d odd) or 2 apart (d = 2, 6):
  // the odd span (pairs of 200 bf16, d = 1) went from 8.1 to about 4
  // wavefronts per load and 6450 -> 6546 GB/s.  For d = 0 (the 128-wide
  // fp16 heads) only walking the second team's vectors from its second one
  // would help; that removed the conflicts but cost 5.8 % more instructions
  // and measured 2 % slower, so those teams stay in order.  (Lanes taking
  // vectors {0, 1, 4, 5} then {2, 3, 6, 7} of each 128 bytes, the odd team
  // the other set first, two base addresses a lane and no extra work a load,
  // also removes them: 6898 against 7058 GB/s on the heads.)
  p->team_map = kTeamsInOrder;
  if (lanes == 4 && sv == 16) {
    const int64_t d = (gbytes * Q / 16) % 8;
    if (d % 2 == 1) p->team_map = kTeamsApart4;
    else if (d == 2 || d == 6) p->team_map = kTeamsApart2;
  }
  // a short first unit for each CTA slot (flat units keep starting on
  // 16-byte boundaries and holding whole items)
  const int64_t mid = mode == 0 ? ug : rpu;
  const int64_t n = mode == 0 ? total : a.rows;
  const int64_t hs = mode == 1 ? 0 : stream_head_size(mode, mid, Q);
  p->head_units = 0;
  p->head_size = static_cast<int>(mid);
  if (hs > 0 && (mode != 0 || (hs * gbytes) % 16 == 0) && n - gmax * hs >= gmax * mid) {
    p->head_units = gmax;
    p->head_size = static_cast<int>(hs);
    p->items = gmax + ceil_div(n - gmax * hs, mid);
    p->grid = std::min(p->items, gmax);
    p->grid_static = ceil_div(p->items, ceil_div(p->items, gmax));
  }
  return GGRN_OK;
}

int make_plan(const Args& a, int path, Plan* p) {
  *p = Plan();
  const bool vec_ok = vector_layout_ok(a);
  switch (path) {
    case kAuto: {
      if (vec_ok) {
        // streaming for groups of whole 16-byte vectors, and for paired
        // items of 17..28 vectors (the low-waste 4 x 7 layout); other paired
        // items leave a quarter of the lane slots idle and measured faster on
        // the register-resident families
        if (plan_stream(a, p, false) == GGRN_OK && p->smem_vec_bytes == 16 &&
            (p->items_groups == 1 || p->vpl == 7))
          return GGRN_OK;
        *p = Plan();
        // Few groups (decode: one row of a few groups): a CTA per group with
        // as few vectors per thread as the CTA size allows, so each group's
        // chain of loads, reduction and stores is short (decode 960-wide:
        // 2.45 -> 1.57 us per call in a 21-call graph, against TEAM's warp
        // of 30 elements per lane).
        const int64_t items = a.rows * (a.width / a.gs);
        const int64_t sms = sm_count();
        // A few wide groups (a batch-1 step of a norm with one wide group):
        // a cluster of CTAs per group, the partial sums of squares combined
        // through distributed shared memory, so each CTA's chain of loads
        // is short.
        if (a.gs / (16 / elem_size(a.dtype)) >= kWideClusterAutoVecs &&
            plan_wide_cluster(a, p) == GGRN_OK && p->grid <= sms)
          return GGRN_OK;
        *p = Plan();
        if (items <= sms) {
          if (plan_wide(a, p, wide_vpl(a, items, sms)) == GGRN_OK) return GGRN_OK;
          *p = Plan();
        }
        if (plan_team(a, p) == GGRN_OK) return GGRN_OK;
        if (plan_wide(a, p, wide_vpl(a, items, sms)) == GGRN_OK) return GGRN_OK;
        if (plan_straddle(a, p) == GGRN_OK) return GGRN_OK;
      }
      return plan_scalar(a, p);
    }
    case kTeam:
      if (!vec_ok) return GGRN_ERR_ALIGN;
      return plan_team(a, p);
    case kWide:
      if (!vec_ok) return GGRN_ERR_ALIGN;
      return plan_wide(a, p);
    case kStraddle:
      if (!vec_ok) return GGRN_ERR_ALIGN;
      return plan_straddle(a, p);
    case kScalar:
      return plan_scalar(a, p);
    case kStream:
      if (!vec_ok) return GGRN_ERR_ALIGN;
      return plan_stream(a, p, true);
    case kWideCluster:
      if (!vec_ok) return GGRN_ERR_ALIGN;
      return plan_wide_cluster(a, p);
    default:
      return GGRN_ERR_ARG;
  }
}

Args make_args(const void* y, const void* gate, const void* w, void* out, int64_t rows,
               int64_t width, int64_t gs, int64_t ys, int64_t gts, int64_t os, float eps,
               int dtype, int mode) {
  Args a;
  a.y = y;
  a.gate = gate;
  a.w = w;
  a.out = out;
  a.rows = rows;
  a.width = width;
  a.gs = gs;
  // A single row has no row stride to speak of.
  a.ys = rows > 1 ? ys : width;
  a.gts = rows > 1 ? gts : width;
  a.os = rows > 1 ? os : width;
  a.eps = eps;
  a.dtype = dtype;
  a.mode = mode;
  return a;
}

// Is work enqueued on `s` being recorded into a graph?  (An error of the
// query counts as yes: the static schedule is always safe.)
bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

int launch(const Args& a, const Plan& plan, cudaStream_t s) {
  if (plan.grid == 0) return GGRN_OK;
  Plan p = plan;
  KParams k = make_params(a, p);
  SlotTable* table = nullptr;
  std::unique_lock<std::mutex> hold;  // held from the slot's choice to its event
  int slot = -1;
  if (p.path == kStream || p.path == kWideCluster) {
    k.fault = fault_word();
    if (!k.fault) return GGRN_ERR_CUDA;
  }
  if (p.path == kStream) {
    // A graph replays its launches with the parameters they were recorded
    // with, the claim epoch included: recorded launches take the static
    // schedule.
    if (!capturing(s) && p.items <= kMaxClaimUnits) {
      unsigned long long* words = sched_words();
      table = slot_table();
      if (!words || !table) return GGRN_ERR_CUDA;
      hold = std::unique_lock<std::mutex>(table->mu);
      const uintptr_t sid = reinterpret_cast<uintptr_t>(s);
      slot = pick_claim_slot(table->slot, kSchedSlots, sid, s == cudaStreamPerThread,
                             table->next, [&](int i) { return slot_done(table->ev[i]); });
      if (slot >= 0 && !table->ev[slot] &&
          cudaEventCreateWithFlags(&table->ev[slot], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        table->ev[slot] = nullptr;
        slot = -1;
      }
      if (slot >= 0) {
        table->next = static_cast<unsigned>(slot + 1) % kSchedSlots;
        k.epoch = next_epoch();
        k.sched = words + slot;
      }
    }
    if (slot < 0) p.grid = p.grid_static;
  }
  cudaError_t e;
  switch (a.dtype) {
    case kF32: e = launch_f32(k, p, a.mode, s); break;
    case kF16: e = launch_f16(k, p, a.mode, s); break;
    default: e = launch_bf16(k, p, a.mode, s); break;
  }
  if (e != cudaSuccess) {
    tl_last_cuda_error = e;
    return GGRN_ERR_CUDA;
  }
  if (slot >= 0) {
    // the slot is this stream's until the event after its launch completes;
    // should the record fail, the slot counts as busy until a later record
    // on it succeeds
    table->slot[slot].owner = reinterpret_cast<uintptr_t>(s);
    table->slot[slot].used = true;
    e = cudaEventRecord(table->ev[slot], s);
    if (e != cudaSuccess) {
      cudaEventDestroy(table->ev[slot]);
      table->ev[slot] = nullptr;
      tl_last_cuda_error = e;
      return GGRN_ERR_CUDA;
    }
  }
  return GGRN_OK;
}

int forward_impl(const Args& a, int path, cudaStream_t s) {
  int st = validate(a);
  if (st != GGRN_OK || a.rows == 0) return st;
  Plan p;
  st = make_plan(a, path, &p);
  if (st != GGRN_OK) return st;
  return launch(a, p, s);
}

struct DecodeGraph {
  cudaGraphExec_t exec = nullptr;  // the captured chain (two or more calls)
  bool direct = false;             // one call: launched as ggrn_forward would
  Args call;
};

}  // namespace

Args call_args(const void* y, const void* gate, const void* w, void* out, int64_t rows,
                int64_t width, int64_t gs, int64_t ys, int64_t gts, int64_t os, float eps,
                int dtype, int mode) {
  return make_args(y, gate, w, out, rows, width, gs, ys, gts, os, eps, dtype, mode);
}

int validate_call(const Args& a) { return validate(a); }

int forward_call(const Args& a, cudaStream_t s) { return forward_impl(a, kAuto, s); }

int plan_family(const Args& a, int path, int vpl, Plan* p) {
  *p = Plan();
  switch (path) {
    case kTeam:
    case kWide:
    case kStraddle:
      if (!vector_layout_ok(a)) return GGRN_ERR_ALIGN;
      if (path == kTeam) return plan_team(a, p);
      if (path == kWide) return plan_wide(a, p, vpl);
      return plan_straddle(a, p);
    case kScalar:
      return plan_scalar(a, p);
    default:
      return GGRN_ERR_ARG;
  }
}

int launch_plan(const Args& a, const Plan& p, cudaStream_t s) { return launch(a, p, s); }

void record_cuda_error(cudaError_t e) { tl_last_cuda_error = e; }

unsigned int* device_fault_word() { return fault_word(); }

KParams make_params(const Args& a, const Plan& p) {
  KParams k;
  k.y = a.y;
  k.gate = a.gate;
  k.w = a.w;
  k.out = a.out;
  k.items = p.items;
  k.groups = p.groups;
  k.items_per_row = p.items_per_row;
  k.width = a.width;
  k.gs = a.gs;
  k.ys = a.ys;
  k.gts = a.gts;
  k.os = a.os;
  k.chunk_elems = p.chunk_elems;
  k.chunks_per_row = p.chunks_per_row;
  k.nvec = p.nvec;
  k.chunk_groups = p.chunk_groups;
  k.warp_smem = p.warp_smem;
  k.gs_magic = p.gs_magic;
  k.div_magic = p.div_magic;
  k.div_magic2 = p.div_magic2;
  k.groups_magic = p.groups_magic;
  k.units = p.items;
  k.units_per_row = p.units_per_row;
  k.total_groups = p.total_groups;
  k.consumer_warps = p.consumer_warps;
  k.stages = p.stages;
  k.stage_bytes = p.stage_bytes;
  k.w_smem_bytes = p.w_smem_bytes;
  k.w_area_bytes = p.w_area_bytes;
  k.ug = p.ug;
  k.unit_mode = p.unit_mode;
  k.rows_per_unit = p.rows_per_unit;
  k.head_units = p.head_units;
  k.head_size = p.head_size;
  k.team_map = p.team_map;
  k.cluster_ctas = p.cluster_ctas;
  k.cluster_vecs = p.cluster_vecs;
  k.rows = a.rows;
  k.fault = nullptr;
  k.no_copies = 0;
  k.sched = nullptr;
  k.epoch = 0;
  k.eps = a.eps;
  k.gs_f = static_cast<float>(a.gs);
  return k;
}

}  // namespace ggrn

using namespace ggrn;

extern "C" int ggrn_forward(const void* y, const void* gate, const void* w, void* out,
                            int64_t rows, int64_t width, int64_t group_size,
                            int64_t y_row_stride, int64_t gate_row_stride,
                            int64_t out_row_stride, float eps, int dtype, int mode,
                            void* cuda_stream) {
  const Args a = make_args(y, gate, w, out, rows, width, group_size, y_row_stride,
                           gate_row_stride, out_row_stride, eps, dtype, mode);
  return forward_impl(a, kAuto, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int ggrn_forward_path(const void* y, const void* gate, const void* w, void* out,
                                 int64_t rows, int64_t width, int64_t group_size,
                                 int64_t y_row_stride, int64_t gate_row_stride,
                                 int64_t out_row_stride, float eps, int dtype, int mode,
                                 int path, void* cuda_stream) {
  if (path < kAuto || path > kWideCluster) return GGRN_ERR_ARG;
  const Args a = make_args(y, gate, w, out, rows, width, group_size, y_row_stride,
                           gate_row_stride, out_row_stride, eps, dtype, mode);
  return forward_impl(a, path, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int ggrn_forward_inproj(const void* inproj, int64_t inproj_row_stride, int64_t y_col,
                                   int64_t gate_col, const void* w, void* out,
                                   int64_t out_row_stride, int64_t rows, int64_t width,
                                   int64_t group_size, float eps, int dtype, int mode,
                                   void* cuda_stream) {
  if (rows < 0 || width <= 0) return GGRN_ERR_SHAPE;
  if (rows == 0) return GGRN_OK;
  if (!inproj) return GGRN_ERR_NULL;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return GGRN_ERR_DTYPE;
  // both column ranges inside a row of the packed buffer
  if (y_col < 0 || gate_col < 0 || y_col > inproj_row_stride - width ||
      gate_col > inproj_row_stride - width)
    return GGRN_ERR_SHAPE;
  const int es = elem_size(dtype);
  const char* base = static_cast<const char*>(inproj);
  const Args a = make_args(base + y_col * es, base + gate_col * es, w, out, rows, width, group_size,
                           inproj_row_stride, inproj_row_stride, out_row_stride, eps, dtype, mode);
  return forward_impl(a, kAuto, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int ggrn_plan(const void* y, const void* gate, const void* w, const void* out,
                         int64_t rows, int64_t width, int64_t group_size, int64_t y_row_stride,
                         int64_t gate_row_stride, int64_t out_row_stride, int dtype, int mode,
                         int path, ggrn_plan_info* info) {
  if (!info) return GGRN_ERR_ARG;
  if (path < kAuto || path > kWideCluster) return GGRN_ERR_ARG;
  std::memset(info, 0, sizeof(*info));
  const Args a = make_args(y, gate, w, const_cast<void*>(out), rows, width, group_size,
                           y_row_stride, gate_row_stride, out_row_stride, 0.0f, dtype, mode);
  int st = validate(a, /*out_optional=*/true);
  if (st != GGRN_OK) return st;
  Plan p;
  st = make_plan(a, path, &p);
  if (st != GGRN_OK) return st;
  info->path = p.path;
  info->team_lanes = p.lanes;
  info->vec_per_lane = p.vpl;
  info->elems_per_vec = p.elems_per_vec;
  info->grid_blocks = p.grid;
  info->block_threads = p.block;
  info->smem_bytes = p.smem;
  info->items = p.items;
  return GGRN_OK;
}

extern "C" int ggrn_graph_create(const ggrn_call* calls, int32_t n, void** graph) {
  if (!graph || n <= 0 || !calls) return GGRN_ERR_ARG;
  *graph = nullptr;
  // Validate and plan every call before capturing anything.
  for (int32_t i = 0; i < n; ++i) {
    const ggrn_call& c = calls[i];
    const Args a = make_args(c.y, c.gate, c.w, c.out, c.rows, c.width, c.group_size,
                             c.y_row_stride, c.gate_row_stride, c.out_row_stride, c.eps, c.dtype,
                             c.mode);
    int st = validate(a);
    if (st != GGRN_OK) return st;
    Plan p;
    if (a.rows > 0 && (st = make_plan(a, kAuto, &p)) != GGRN_OK) return st;
  }
  // symbol lookups before the capture starts
  if (!fault_word() || !sched_words()) return GGRN_ERR_CUDA;
  if (n == 1) {
    // A graph of one small kernel costs more to launch than the kernel
    // itself (decode: 4.1 against 3.4-3.7 us per call): a one-call chain is
    // launched directly on each replay, with the same buffers.
    DecodeGraph* dg = new DecodeGraph();
    dg->direct = true;
    const ggrn_call& c = calls[0];
    dg->call = make_args(c.y, c.gate, c.w, c.out, c.rows, c.width, c.group_size,
                         c.y_row_stride, c.gate_row_stride, c.out_row_stride, c.eps, c.dtype,
                         c.mode);
    *graph = dg;
    return GGRN_OK;
  }
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return GGRN_ERR_CUDA;
  int status = GGRN_OK;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    return GGRN_ERR_CUDA;
  }
  for (int32_t i = 0; i < n && status == GGRN_OK; ++i) {
    const ggrn_call& c = calls[i];
    const Args a = make_args(c.y, c.gate, c.w, c.out, c.rows, c.width, c.group_size,
                             c.y_row_stride, c.gate_row_stride, c.out_row_stride, c.eps, c.dtype,
                             c.mode);
    status = forward_impl(a, kAuto, s);
  }
  cudaError_t e = cudaStreamEndCapture(s, &g);
  if (status == GGRN_OK && e != cudaSuccess) status = GGRN_ERR_CUDA;
  DecodeGraph* dg = nullptr;
  if (status == GGRN_OK) {
    dg = new DecodeGraph();
    if (cudaGraphInstantiate(&dg->exec, g, 0) != cudaSuccess) {
      status = GGRN_ERR_CUDA;
      delete dg;
      dg = nullptr;
    }
  }
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  if (status == GGRN_OK) *graph = dg;
  return status;
}

extern "C" int ggrn_graph_launch(void* graph, void* cuda_stream) {
  if (!graph) return GGRN_ERR_ARG;
  DecodeGraph* dg = static_cast<DecodeGraph*>(graph);
  if (dg->direct) return forward_impl(dg->call, kAuto, static_cast<cudaStream_t>(cuda_stream));
  return cudaGraphLaunch(dg->exec, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
             ? GGRN_OK
             : GGRN_ERR_CUDA;
}

extern "C" int ggrn_graph_destroy(void* graph) {
  if (!graph) return GGRN_OK;
  DecodeGraph* dg = static_cast<DecodeGraph*>(graph);
  const cudaError_t e = dg->direct ? cudaSuccess : cudaGraphExecDestroy(dg->exec);
  delete dg;
  return e == cudaSuccess ? GGRN_OK : GGRN_ERR_CUDA;
}

extern "C" const char* ggrn_status_string(int status) {
  switch (status) {
    case GGRN_OK: return "ok";
    case GGRN_ERR_NULL: return "a required pointer is NULL";
    case GGRN_ERR_SHAPE: return "invalid shape: rows < 0, width <= 0, group_size <= 0, width not a "
                                "multiple of group_size, row stride < width, or size overflow";
    case GGRN_ERR_ALIGN: return "pointers or row strides not aligned for the requested path";
    case GGRN_ERR_DTYPE: return "unsupported dtype/mode (ONNX semantics admit float32 and float16)";
    case GGRN_ERR_OVERLAP: return "out overlaps y, gate or w";
    case GGRN_ERR_CUDA: return "CUDA runtime error";
    case GGRN_ERR_UNSUPPORTED: return "the requested path does not cover this shape";
    case GGRN_ERR_ARG: return "invalid argument (path id, NULL out-parameter or call list)";
    case GGRN_ERR_LIMIT: return "beyond the fixed limit of ggrn_forward_noalloc (more streamed "
                                "units than its claim counter can address)";
    default: return "unknown status";
  }
}

extern "C" int ggrn_version(void) { return 100; }

extern "C" int ggrn_fault_status(uint32_t* flags, int clear) {
  if (!flags) return GGRN_ERR_ARG;
  *flags = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return GGRN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_ggrn_fault, sizeof(v)) != cudaSuccess) return GGRN_ERR_CUDA;
  *flags = v;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_ggrn_fault, &zero, sizeof(zero)) != cudaSuccess) return GGRN_ERR_CUDA;
  }
  return GGRN_OK;
}

extern "C" const char* ggrn_last_cuda_error(void) {
  return cudaGetErrorName(tl_last_cuda_error);
}

// ---------------------------------------------------------------------------
// ggrn_forward_noalloc: the streaming kernel with its claim counter in a
// fixed array of this file (no counterpart in the pages; see include/ggrn.h).
// ---------------------------------------------------------------------------

// The entry point's scratch: GGRN_NOALLOC_SCRATCH_BYTES in this module, one
// copy on every device that loads the library, held until the process exits.
// Word 0 is the unit-claim counter of the call in flight; every call clears
// it on its own stream before its kernel starts, so calls that overlap on the
// GPU share it and race.
static __device__ __align__(256) unsigned long long
    g_ggrn_noalloc_scratch[GGRN_NOALLOC_SCRATCH_BYTES / sizeof(unsigned long long)];

namespace ggrn {
namespace {

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// (once per device, on the first call there, with that device current) and
// passed to the kernel.
unsigned long long* noalloc_scratch() {
  static std::mutex mu;
  static unsigned long long* cache[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    tl_last_cuda_error = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_ggrn_noalloc_scratch);
    if (e != cudaSuccess) {
      tl_last_cuda_error = e;
      return nullptr;
    }
    cache[dev] = static_cast<unsigned long long*>(ptr);
  }
  return cache[dev];
}

}  // namespace
}  // namespace ggrn

extern "C" int ggrn_forward_noalloc(const void* y, const void* gate, const void* w, void* out,
                                    int64_t rows, int64_t width, int64_t group_size,
                                    int64_t y_row_stride, int64_t gate_row_stride,
                                    int64_t out_row_stride, float eps, int dtype, int mode,
                                    void* cuda_stream) {
  const Args a = make_args(y, gate, w, out, rows, width, group_size, y_row_stride,
                           gate_row_stride, out_row_stride, eps, dtype, mode);
  int st = validate(a);
  if (st != GGRN_OK || a.rows == 0) return st;
  if (!vector_layout_ok(a)) return GGRN_ERR_ALIGN;
  Plan p;
  st = plan_stream(a, &p, /*forced=*/true);
  if (st != GGRN_OK) return st;
  // The counter hands out 32-bit unit indices.
  if (p.items > GGRN_NOALLOC_MAX_UNITS) return GGRN_ERR_LIMIT;
  unsigned long long* scratch = noalloc_scratch();
  if (!scratch) return GGRN_ERR_CUDA;
  unsigned int* fault = fault_word();
  if (!fault) return GGRN_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // Claims start at 0 under epoch 0 (a cleared word reads as installed).
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(unsigned long long), s);
  if (e == cudaSuccess) {
    KParams k = make_params(a, p);
    k.fault = fault;
    k.sched = scratch;
    k.epoch = 0;
    switch (a.dtype) {
      case kF32: e = launch_f32(k, p, a.mode, s); break;
      case kF16: e = launch_f16(k, p, a.mode, s); break;
      default: e = launch_bf16(k, p, a.mode, s); break;
    }
  }
  if (e != cudaSuccess) {
    tl_last_cuda_error = e;
    return GGRN_ERR_CUDA;
  }
  return GGRN_OK;
}

extern "C" int ggrn_selftest_wait_timeout(const void* y, const void* gate, const void* w,
                                          void* out, int64_t rows, int64_t width,
                                          int64_t group_size, int dtype, void* cuda_stream) {
  const Args a = make_args(y, gate, w, out, rows, width, group_size, width, width, width, 1e-5f,
                           dtype, kMamba2);
  int st = validate(a);
  if (st != GGRN_OK) return st;
  if (rows == 0) return GGRN_ERR_SHAPE;
  if (!vector_layout_ok(a)) return GGRN_ERR_ALIGN;
  Plan p;
  if ((st = plan_stream(a, &p, /*forced=*/true)) != GGRN_OK) return st;
  KParams k = make_params(a, p);
  k.fault = fault_word();
  if (!k.fault) return GGRN_ERR_CUDA;
  k.no_copies = 1;
  const cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e;
  switch (a.dtype) {
    case kF32: e = launch_f32(k, p, a.mode, s); break;
    case kF16: e = launch_f16(k, p, a.mode, s); break;
    default: e = launch_bf16(k, p, a.mode, s); break;
  }
  if (e != cudaSuccess) {
    tl_last_cuda_error = e;
    return GGRN_ERR_CUDA;
  }
  return GGRN_OK;
}
