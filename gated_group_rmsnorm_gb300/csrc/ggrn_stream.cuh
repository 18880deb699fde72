// ggrn_stream.cuh -- the TMA streaming family of the fused gated
// group-RMSNorm (sm_103a).
//
// Persistent CTAs.  One producer lane moves whole row chunks ("units": a run
// of whole groups, contiguous in y, gate and out) from HBM into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk, the TMA engine),
// each stage completing on an mbarrier that counts the bytes.  W consumer
// warps wait for a stage, compute every group of it from shared memory
// (teams of `L` lanes per group as in k_team; a segmented butterfly reduces
// each team), store the outputs straight to HBM with evict-first 16- or
// 8-byte stores, and release the stage.  Bytes in flight per SM are the
// stages the producer runs ahead, independent of registers, and the copy
// engine issues them without spending the consumers' issue slots.
//
// Shared-memory vectors of SV bytes (16 or 8: the largest that divides a
// group's bytes) let groups that are not a multiple of the 16-byte vector
// (the odd span of 100 bf16 = 200 bytes) be read at group granularity with no
// straddling: the bulk copy itself moves 16-byte-multiple chunks.
//
// Schedule: each CTA takes its first NS units statically (CTA b: units b,
// b + grid, ...), then claims units one at a time from a word in device
// memory shared by the CTAs of the launch, so that CTAs that run slower
// (memory-channel contention varies) take fewer units and all finish within
// about one unit of each other.  The claim of the next unit is issued while
// the producer waits for a free stage.  Launches recorded into a CUDA graph
// keep the static interleaved schedule (no claim word).
//
// Waits are bounded: after kWaitLimit polls a thread records a fault bit in
// the library's device status word and stops; the producer lane then waits
// (again bounded) until every copy it issued has landed, so no copy targets
// the shared memory of a finished CTA.
#pragma once

#include "ggrn_kernels.cuh"

// Per-CTA timeline of streaming launches, compiled in only with
// -DGGRN_TIMELINE (a separate profiling build of the library): for each of the
// last 64 launches (by claim epoch) and each CTA, the global-timer stamps of
// entry, release of the dependency wait, the first stage seen by consumer
// warp 0 and the end of the CTA's last consumer warp, and the units it took.
#ifdef GGRN_TIMELINE
constexpr int kTimelineLaunches = 64;
constexpr int kTimelineCtas = 320;
static __device__ unsigned long long g_ggrn_timeline[kTimelineLaunches][kTimelineCtas][5];
__device__ __forceinline__ unsigned long long timeline_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define GGRN_TIMELINE_AT(p, field) \
  g_ggrn_timeline[(p).epoch % kTimelineLaunches][blockIdx.x][field]
#define GGRN_TIMELINE_ON (blockIdx.x < kTimelineCtas)
#endif

namespace ggrn {

// Attempts of one unit claim against other launches' installations.
constexpr uint32_t kClaimTries = 4096;
// Unit shapes: ug consecutive groups of contiguous rows (flat), ug groups
// inside one row (chunk), or rows_per_unit whole rows copied row by row.
constexpr int kUnitFlat = 0;
constexpr int kUnitChunk = 1;
constexpr int kUnitRows = 2;

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// A vector of NW 32-bit words: shared-memory load, evict-first global store.
template <int NW>
struct Words {
  uint32_t w[NW];
};
template <int NW>
__device__ __forceinline__ Words<NW> lds_words(const void* p) {
  Words<NW> r;
  if (NW == 4) {
    uint4 v = *static_cast<const uint4*>(p);
    r.w[0] = v.x, r.w[1 % NW] = v.y, r.w[2 % NW] = v.z, r.w[3 % NW] = v.w;
  } else if (NW == 2) {
    uint2 v = *static_cast<const uint2*>(p);
    r.w[0] = v.x, r.w[1 % NW] = v.y;
  } else {
    r.w[0] = *static_cast<const uint32_t*>(p);
  }
  return r;
}
template <int NW>
__device__ __forceinline__ Words<NW> ldg_words(const void* p) {
  Words<NW> r;
  if (NW == 4) {
    uint4 v = __ldg(static_cast<const uint4*>(p));
    r.w[0] = v.x, r.w[1 % NW] = v.y, r.w[2 % NW] = v.z, r.w[3 % NW] = v.w;
  } else if (NW == 2) {
    uint2 v = __ldg(static_cast<const uint2*>(p));
    r.w[0] = v.x, r.w[1 % NW] = v.y;
  } else {
    r.w[0] = __ldg(static_cast<const uint32_t*>(p));
  }
  return r;
}
template <int NW>
__device__ __forceinline__ void stg_words(void* p, const Words<NW>& v) {
  if (NW == 4) {
    __stcs(static_cast<uint4*>(p), make_uint4(v.w[0], v.w[1 % NW], v.w[2 % NW], v.w[3 % NW]));
  } else if (NW == 2) {
    __stcs(static_cast<uint2*>(p), make_uint2(v.w[0], v.w[1 % NW]));
  } else {
    __stcs(static_cast<unsigned int*>(p), v.w[0]);
  }
}

// Words <-> f32 elements of T (2 per word for 16-bit T, 1 for f32).
template <typename T, int NW>
__device__ __forceinline__ void words_to_f32(const Words<NW>& v, float* f) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < NW; ++i) f[i] = __uint_as_float(v.w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) Elem<T>::unpack2(v.w[i], f[2 * i], f[2 * i + 1]);
  }
}
template <typename T, int NW>
__device__ __forceinline__ Words<NW> f32_to_words(const float* f) {
  Words<NW> v;
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < NW; ++i) v.w[i] = __float_as_uint(f[i]);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) v.w[i] = Elem<T>::pack2(f[2 * i], f[2 * i + 1]);
  }
  return v;
}

// ---------------------------------------------------------------------------
// Unit claims.  The claim word holds epoch << 32 | next: the launch whose
// epoch (a number the host gives each launch) is installed hands out indices
// 0, 1, 2, ... in order, one per atomicAdd.  `v` is what the caller's
// atomicAdd(w, 1) returned.  A word carrying another epoch (the slot's
// previous launch, or a concurrent launch given the same slot) is replaced
// by this epoch with next = 1, the caller taking index 0.  A launch whose
// installation was replaced installs itself again and restarts at 0: units
// may then be processed twice (the same bytes written again) but none is
// skipped, since a CTA stops only on an index >= the count under its own
// launch's latest installation, all lower indices of which went to CTAs of
// that launch.  Returns the index, or -1 (and *ok = false) after
// kClaimTries attempts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t claim_resolve(unsigned long long* w, uint32_t epoch,
                                                 unsigned long long v, bool* ok) {
  const unsigned long long fresh = (static_cast<unsigned long long>(epoch) << 32) | 1ull;
  unsigned long long cur = v + 1;  // the word as the caller's add left it
  for (uint32_t t = 0; t < kClaimTries; ++t) {
    if (static_cast<uint32_t>(v >> 32) == epoch) return static_cast<int64_t>(v & 0xffffffffull);
    const unsigned long long seen = atomicCAS(w, cur, fresh);
    if (seen == cur) return 0;
    if (static_cast<uint32_t>(seen >> 32) == epoch) {
      v = atomicAdd(w, 1ull);  // installed by another CTA: claim normally
      cur = v + 1;
    } else {
      cur = seen;  // still another epoch's word: try to replace what is there now
    }
  }
  *ok = false;
  return -1;
}

// ---------------------------------------------------------------------------
// Pieces of the streaming kernel.  Dynamic shared memory:
// [stages][y slot | gate slot], the weight area, 16 bytes of zeros, then the barriers
// full[NS], empty[NS], wbar, sbar, the unit of each stage (int64 [NS]) and
// its placement (UnitInfo [NS]).
// ---------------------------------------------------------------------------
// A unit as its consumers place it, written by the producer lane beside the
// stage's unit index: the output offset (elements) of its first group (row
// units: of its first row), the index of that group within its row (row
// units: 0), and the unit's group count.
struct UnitInfo {
  int64_t out0;
  int32_t cg0;
  int32_t ngroups;
};

struct StreamCtx {
  unsigned char* ring;
  unsigned char* wsm;    // staged weight (when wbytes != 0)
  long long* unit_of;    // unit in each stage; -1: no more units
  UnitInfo* uinfo;       // placement of each stage's unit
  uint32_t sb;           // bytes of one tensor's slot (128-aligned)
  uint32_t wbytes;       // 0: the weight is read from global memory
  uint32_t full0, empty0, wbar;
  uint32_t sbar;         // every consumer thread done permuting the staged weight
  const unsigned char* zero16;  // 16 bytes of zeros (what slots outside an item read)
  int NS, W;
};

// Barrier set-up (thread 0), then the programmatic-dependent-launch wait:
// nothing global is touched before the previous kernel's writes are visible.
__device__ __forceinline__ StreamCtx stream_setup(const KParams& p, unsigned char* smem) {
  StreamCtx c;
  c.ring = smem;
  c.NS = p.stages;
  c.W = p.consumer_warps;
  c.sb = p.stage_bytes;
  c.wsm = smem + static_cast<size_t>(2) * c.NS * c.sb;
  c.wbytes = p.w_smem_bytes;
  const uint32_t warea = p.w_area_bytes;  // the weight and its slack, 128-byte multiple
  c.zero16 = c.wsm + warea;
  uint64_t* bars = reinterpret_cast<uint64_t*>(c.wsm + warea + 16);
  c.full0 = smem_u32(bars);
  c.empty0 = smem_u32(bars + c.NS);
  c.wbar = smem_u32(bars + 2 * c.NS);
  c.sbar = smem_u32(bars + 2 * c.NS + 1);
  c.unit_of = reinterpret_cast<long long*>(bars + 2 * c.NS + 2);
  c.uinfo = reinterpret_cast<UnitInfo*>(c.unit_of + c.NS);
  if (threadIdx.x == 0) {
    *reinterpret_cast<uint4*>(c.wsm + warea) = make_uint4(0u, 0u, 0u, 0u);
    for (int s = 0; s < c.NS; ++s) {
      mbar_init(c.full0 + 8 * s, 1);
      mbar_init(c.empty0 + 8 * s, c.W);
    }
    mbar_init(c.wbar, 1);
    mbar_init(c.sbar, 32 * c.W);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
#ifdef GGRN_TIMELINE
  const unsigned long long t_entry = timeline_now();
#endif
  pdl_wait();
#ifdef GGRN_TIMELINE
  if (threadIdx.x == 0 && GGRN_TIMELINE_ON) {
    GGRN_TIMELINE_AT(p, 0) = t_entry;
    GGRN_TIMELINE_AT(p, 1) = timeline_now();
    GGRN_TIMELINE_AT(p, 2) = 0;
    GGRN_TIMELINE_AT(p, 3) = 0;
    GGRN_TIMELINE_AT(p, 4) = 0;
  }
  __syncthreads();
#endif
  pdl_launch_dependents();
  return c;
}

// Flat and row units cut a sequence of n groups or rows: head_units units of
// head_size, then units of `mid`, the last one clipped at n.  Returns unit
// u's first element and sets its length.
__device__ __forceinline__ int64_t unit_span(const KParams& p, int64_t u, int64_t mid, int64_t n,
                                             int64_t* len) {
  const bool head = u < p.head_units;
  const int64_t first =
      head ? u * p.head_size : p.head_units * p.head_size + (u - p.head_units) * mid;
  *len = min(head ? static_cast<int64_t>(p.head_size) : mid, n - first);
  return first;
}

// The producer lane: stage the weight, then stream this CTA's units into the
// ring, each stage's unit recorded in unit_of; after the last unit a stage
// with unit -1 (completed by a plain arrive) tells the consumers to stop.
// Finally wait (bounded) until every issued copy has landed.
template <typename T>
__device__ __forceinline__ void stream_produce(const KParams& p, const StreamCtx& c) {
  constexpr int ES = sizeof(T);
  const int64_t gs = p.gs;
  // self-test of the failure path: no copy, no arrival; every consumer wait
  // runs out, records its fault bit and returns
  if (p.no_copies) return;
  if (c.wbytes) {
    mbar_expect_tx(c.wbar, c.wbytes);
    bulk_g2s(smem_u32(c.wsm), p.w, c.wbytes, c.wbar);
  }
  const int NS = c.NS;
  const int64_t G = gridDim.x;
  const bool dyn = p.sched != nullptr;
  int64_t i = 0;
  bool ok = true, claim_ok = true;
  unsigned long long pending = 0;  // the claim issued for the next stage
  int64_t u = blockIdx.x;
  for (;; ++i) {
    const int s = static_cast<int>(i % NS);
    if (i >= NS && !mbar_wait(c.empty0 + 8 * s, static_cast<uint32_t>((i / NS) - 1) & 1u)) {
      ok = false;
      break;
    }
    if (dyn && i >= NS) {
      const int64_t d = claim_resolve(p.sched, p.epoch, pending, &claim_ok);
      u = claim_ok ? NS * G + d : p.units;
    }
    const uint32_t full = c.full0 + 8 * s;
    if (u >= p.units) {
      c.unit_of[s] = -1;
      mbar_arrive(full);
      ++i;
      break;
    }
    // The stage's bytes are declared and its copies issued first (with the
    // claim for the next stage): on an HBM-bound launch the ring runs nearly
    // empty, and the copies wait for nothing else.  Then the unit's index and
    // placement are written and the producer arrives, which completes the
    // phase (and publishes them) once the bytes have landed.
    unsigned char* st = c.ring + static_cast<size_t>(2) * s * c.sb;
    UnitInfo ui;
    if (p.unit_mode == kUnitRows) {
      // R whole rows, one copy per row and tensor, packed in the slot
      int64_t nr;
      const int64_t row0 = unit_span(p, u, p.rows_per_unit, p.rows, &nr);
      const uint32_t rb = static_cast<uint32_t>(p.width * ES);
      mbar_add_tx(full, static_cast<uint32_t>(2 * nr) * rb);
      for (int64_t r = 0; r < nr; ++r) {
        bulk_g2s(smem_u32(st + r * rb), static_cast<const T*>(p.y) + (row0 + r) * p.ys, rb, full);
        bulk_g2s(smem_u32(st + c.sb + r * rb), static_cast<const T*>(p.gate) + (row0 + r) * p.gts,
                 rb, full);
      }
      ui.out0 = row0 * p.os;
      ui.cg0 = 0;
      ui.ngroups = static_cast<int32_t>(nr * p.groups);
    } else {
      int64_t yo, go, ngroups, g0 = 0, row = 0, cg = 0;
      if (p.unit_mode == kUnitFlat) {
        g0 = unit_span(p, u, p.ug, p.total_groups, &ngroups);
        yo = go = g0 * gs;
      } else {
        row = div_by(u, p.units_per_row, p.div_magic);
        cg = (u - row * p.units_per_row) * p.ug;
        const int64_t c0 = cg * gs;
        ngroups = p.ug;
        yo = row * p.ys + c0;
        go = row * p.gts + c0;
      }
      const uint32_t bytes = static_cast<uint32_t>(ngroups * gs * ES);
      mbar_add_tx(full, 2 * bytes);
      bulk_g2s(smem_u32(st), static_cast<const T*>(p.y) + yo, bytes, full);
      bulk_g2s(smem_u32(st + c.sb), static_cast<const T*>(p.gate) + go, bytes, full);
      if (p.unit_mode == kUnitFlat) {
        ui.out0 = g0 * gs;  // out rows of flat units are contiguous
        cg = g0 - div_by(g0, p.groups, p.div_magic2) * p.groups;
      } else {
        ui.out0 = row * p.os + cg * gs;
      }
      ui.cg0 = static_cast<int32_t>(cg);
      ui.ngroups = static_cast<int32_t>(ngroups);
    }
    const int64_t uc = u;
    if (dyn && i + 1 >= NS) {
      pending = atomicAdd(p.sched, 1ull);  // resolved after the next empty wait
    } else {
      u += G;
    }
    c.unit_of[s] = uc;
    c.uinfo[s] = ui;
    mbar_arrive(full);
  }
  if (!ok) atomicOr(p.fault, kFaultProducerWait);
  if (!claim_ok) atomicOr(p.fault, kFaultClaim);
  // Every issued copy lands before this thread leaves: wait for the last
  // phase of each stage used (already complete in the normal course).
  const int64_t n_issued = i;
  for (int s = 0; s < NS && s < n_issued; ++s) {
    const int64_t last = s + ((n_issued - 1 - s) / NS) * NS;
    if (!mbar_wait(c.full0 + 8 * s, static_cast<uint32_t>(last / NS) & 1u))
      atomicOr(p.fault, kFaultDrainWait);
  }
  if (c.wbytes && !mbar_wait(c.wbar, 0)) atomicOr(p.fault, kFaultDrainWait);
}

// floor(n / d) for a group's row offset within a unit: one multiply-high by
// magic = floor(2^32 / d) + 1, exact for every n with n * d < 2^32 (the
// host checks that for every n a unit can give, else passes 0).
__device__ __forceinline__ int div_small(int n, int d, uint32_t magic) {
  if (magic != 0) return static_cast<int>(__umulhi(static_cast<unsigned>(n), magic));
  return d == 1 ? n : n / d;
}

// Output offset (elements) and weight column of group gl of a unit (32-bit
// within the unit: the host streams rows of fewer than 2^30 elements).
__device__ __forceinline__ void group_place(const KParams& p, const UnitInfo& ui, int gl,
                                            int64_t* out_off, int* wcol) {
  const int gs = static_cast<int>(p.gs);
  const int groups = static_cast<int>(p.groups);
  const int cg = ui.cg0 + gl;                          // group index from the unit's first row
  const int r = div_small(cg, groups, p.groups_magic);  // rows past the unit's first row
  *wcol = (cg - r * groups) * gs;  // (unused, and not computed, in ONNX flat and chunk units)
  *out_off = p.unit_mode == kUnitRows ? ui.out0 + r * p.os + *wcol
                                      : ui.out0 + gl * gs;  // flat and chunk: contiguous
}

// The staged f32 weight of MAMBA2 with 16-bit T is read 32 bytes (one
// vector's 8 columns) per lane, lanes 32 bytes apart: as stored, two lanes
// of every 8 would meet on the same banks.  So the staged copy is permuted
// once per CTA: in each 32-byte block whose index has bit 2 set the two
// 16-byte halves trade places, and 8 consecutive blocks then read either
// half from 8 distinct 16-byte bank groups (prefill 960-wide groups: 6078
// -> 6171 GB/s in alternating runs).
__device__ __forceinline__ void swap_weight_halves(unsigned char* wsm, uint32_t wbytes, int tid,
                                                   int nthreads) {
  for (uint32_t b = 4u + 8u * (tid >> 2) + (tid & 3); b < wbytes / 32u; b += 2u * nthreads) {
    uint4* h = reinterpret_cast<uint4*>(wsm + 32u * b);
    const uint4 lo = h[0], hi = h[1];
    h[0] = hi;
    h[1] = lo;
  }
}

// f32 weight of SE columns at wi, as stored (shared memory when staged).
template <int SE>
__device__ __forceinline__ void load_w_cols(const KParams& p, const StreamCtx& c, int64_t wi,
                                            float (&wv)[SE]) {
#pragma unroll
  for (int q = 0; q < SE; q += 4 > SE ? SE : 4) {
    if (SE >= 4) {
      const float4 w4 =
          c.wbytes ? *reinterpret_cast<const float4*>(c.wsm + 4 * (wi + q))
                   : __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.w) + wi + q));
      wv[q] = w4.x, wv[(q + 1) % SE] = w4.y, wv[(q + 2) % SE] = w4.z, wv[(q + 3) % SE] = w4.w;
    } else {
      const float2 w2 =
          c.wbytes ? *reinterpret_cast<const float2*>(c.wsm + 4 * (wi + q))
                   : __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(p.w) + wi + q));
      wv[q] = w2.x, wv[(q + 1) % SE] = w2.y;
    }
  }
}

// ---------------------------------------------------------------------------
// k_stream: TEAM consumers.  SV = bytes per shared-memory vector (16 or 8),
// SE = elements per vector, L lanes per team, VPL vectors per lane, Q groups
// per team item (1, or 2 for groups of an odd number of half vectors), MAXW
// the most consumer warps a launch may have (it sets the register budget:
// 17 warps leave 96 registers a thread, 13 leave 128).
// ---------------------------------------------------------------------------
template <typename T, int MODE, int L, int VPL, int SV, int Q, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32, 1) k_stream(const KParams p) {
  constexpr int ES = sizeof(T);
  constexpr int SE = SV / ES;
  constexpr int NW = SV / 4;
  constexpr int TPW = 32 / L;  // teams (items) per warp
  extern __shared__ __align__(128) unsigned char smem[];

  const StreamCtx c = stream_setup(p, smem);
  const int W = c.W;
  const int NS = c.NS;
  const uint32_t sb = c.sb;
  const uint32_t wbytes = c.wbytes;
  unsigned char* wsm = c.wsm;
  const uint32_t full0 = c.full0, empty0 = c.empty0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t gs = p.gs;
  if (warp == W) {
    if (lane == 0) stream_produce<T>(p, c);
    return;
  }
  if (wbytes && !mbar_wait(c.wbar, 0)) {
    if (lane == 0) atomicOr(p.fault, kFaultConsumerWait);
    return;
  }
  // (teams of 8+ lanes, whose 8-lane phases read consecutive blocks; and
  // paired 4-lane teams, whose phases hold two items 4 apart under the
  // planner's kTeamsApart4 map: their blocks are 100 apart for the 200-wide
  // pairs of 100-wide bf16 groups, and adding 100 flips bit 2)
  constexpr bool kSwz = MODE == kMamba2 && SE == 8 && ((Q == 1 && L >= 8) || (Q == 2 && L == 4));
  if (kSwz && wbytes) {
    // permute the staged weight (all consumer threads), then wait until
    // every consumer thread has finished its share (bounded like every wait)
    swap_weight_halves(wsm, wbytes, threadIdx.x, 32 * W);
    mbar_arrive(c.sbar);
    if (!mbar_wait(c.sbar, 0)) {
      if (lane == 0) atomicOr(p.fault, kFaultConsumerWait);
      return;
    }
  }

  // ---------------- consumers ----------------
  // A team takes an "item" of Q consecutive groups.  Q = 2 pairs groups whose
  // bytes are an odd multiple of half a vector: the pair is whole 16-byte
  // vectors, and the one vector across the boundary (vector vb) splits at its
  // middle, its low half ending the first group.
  const int team = lane / L;
  const int tl = lane & (L - 1);
  // the item this team takes within a warp's pass (TeamMap: keeps the two
  // teams of an 8-lane phase on distinct shared-memory banks)
  int titem = team;
  if constexpr (TPW == 8) {
    if (p.team_map == kTeamsApart4) {
      titem = (team >> 1) + 4 * (team & 1);
    } else if (p.team_map == kTeamsApart2) {
      titem = (team & 4) + ((team >> 1) & 1) + 2 * (team & 1);
    }
  }
  const int nvec = static_cast<int>(Q * gs / SE);
  const int vb = static_cast<int>(gs / SE);
  // Slots that every lane fills, and the slots wholly in an item's first or
  // second group, from the team shapes the planner picks (launch_stream
  // refuses any other): with 4 vectors a lane, L is the power of two at or
  // above nvec / 4, so 2L < nvec <= 4L and a pair's split vector
  // vb = (nvec - 1) / 2 lies in [L, 2L); the 4 x 7 pairs have 17 <= nvec <= 27
  // and 8 <= vb <= 13.  Slot k holds vector k * L + tl.
  constexpr int kFull = VPL == 7 ? 4 : 2;  // k < kFull: v < nvec in every lane
  constexpr int kG0 = VPL == 7 ? 2 : 1;    // k < kG0: v < vb
  constexpr int kG1 = VPL == 7 ? 4 : 2;    // k >= kG1: v > vb
  constexpr bool kBranchFree = MODE == kMamba2;
  const int items_per_pass = W * TPW;
#ifdef GGRN_TIMELINE
  unsigned long long tl_first = 0;  // kept in registers: no global access in the loop
  unsigned long long tl_units = 0;
#endif
  // stage s of the ring and the parity of its current fill
  for (int s = 0, phase = 0;; s = (s + 1 == NS) ? 0 : s + 1, phase ^= (s == 0)) {
    if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>(phase))) {
      if (lane == 0) atomicOr(p.fault, kFaultConsumerWait);
      break;
    }
    const int64_t u = c.unit_of[s];
#ifdef GGRN_TIMELINE
    if (u >= 0) {
      if (tl_units == 0) tl_first = timeline_now();
      ++tl_units;
    }
#endif
    if (u < 0) break;
    // ONNX flat units need only the output offset, which the unit index gives
    // at once; reading the producer's placement instead put a dependent
    // shared-memory load first in every stage (heads 7047 -> 7009 GB/s)
    UnitInfo ui;
    if constexpr (MODE == kOnnx) {
      if (p.unit_mode == kUnitFlat) {
        int64_t ng;
        const int64_t g0 = unit_span(p, u, p.ug, p.total_groups, &ng);
        ui.out0 = g0 * p.gs;
        ui.cg0 = 0;  // (the weight column is not used)
        ui.ngroups = static_cast<int32_t>(ng);
      } else {
        ui = c.uinfo[s];
      }
    } else {
      ui = c.uinfo[s];
    }
    const int nitems = ui.ngroups / Q;
    const unsigned char* sy = smem + static_cast<size_t>(2) * s * sb;
    const unsigned char* sg = sy + sb;
    for (int pass = 0; pass * items_per_pass < nitems; ++pass) {
      const int item = pass * items_per_pass + warp * TPW + titem;
      const bool active = item < nitems;
      // items rise with the pass: a warp with no item left is done with the unit
      if (!__any_sync(0xffffffffu, active)) break;
      // MAMBA2: the loop body is branch-free.  A team past the unit's items
      // computes on the pass's first item (in bounds) and stores nothing; a
      // slot past the item's vectors reads the zero block (y = gate = 0:
      // nothing added to the sums) and stores nothing (prefill +1.5 %, odd
      // span +1.2 %).  ONNX keeps branches around those slots (its 128-wide
      // heads measured 1.5 % slower branch-free).
      const int gl = (active ? item : pass * items_per_pass) * Q;  // first group of the item
      int64_t out_off;  // output origin of that group
      int wcol;         // and its weight column
      group_place(p, ui, gl, &out_off, &wcol);
      const unsigned char* gy = sy + gl * static_cast<int>(gs) * ES;
      const unsigned char* gg = sg + gl * static_cast<int>(gs) * ES;

      Words<NW> yr[VPL], gr[VPL];
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int v = k * L + tl;
        const bool in = k < kFull || v < nvec;
        if (kBranchFree) {
          yr[k] = lds_words<NW>(in ? gy + v * SV : c.zero16);
          gr[k] = lds_words<NW>(in ? gg + v * SV : c.zero16);
        } else if (active && in) {
          yr[k] = lds_words<NW>(gy + v * SV);
          gr[k] = lds_words<NW>(gg + v * SV);
        } else {
#pragma unroll
          for (int q = 0; q < NW; ++q) yr[k].w[q] = 0u, gr[k].w[q] = 0u;
        }
      }
      float a[VPL][SE];
      float s0 = 0.0f, s1 = 0.0f;
      float c0 = 0.0f, c1 = 0.0f;  // Q == 1: even / odd element partial sums
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        float yf[SE];
        words_to_f32<T, NW>(yr[k], yf);
        if (MODE == kMamba2) {
          float gf[SE];
          words_to_f32<T, NW>(gr[k], gf);
          gated_vec<T, SE>(yf, gf, a[k]);
        } else {
#pragma unroll
          for (int e = 0; e < SE; ++e) a[k][e] = yf[e];
        }
        if constexpr (Q == 1) {
          sumsq2<SE>(a[k], c0, c1);
        } else {
          float h0a = 0.0f, h0b = 0.0f, h1a = 0.0f, h1b = 0.0f;
          sumsq2<SE / 2>(a[k], h0a, h0b);
          sumsq2<SE / 2>(a[k] + SE / 2, h1a, h1b);
          const float h0 = h0a + h0b, h1 = h1a + h1b;
          const int v = k * L + tl;
          if (k < kG0) {
            s0 += h0 + h1;
          } else if (k >= kG1) {
            s1 += h0 + h1;
          } else {
            s0 += (v < vb) ? h0 + h1 : (v == vb ? h0 : 0.0f);
            s1 += (v > vb) ? h0 + h1 : (v == vb ? h1 : 0.0f);
          }
        }
      }
      if constexpr (Q == 1) s0 = c0 + c1;
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        if constexpr (Q == 2) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      const float nf0 = normaliser(s0, p.gs_f, p.eps);
      const float nf1 = (Q == 2) ? normaliser(s1, p.gs_f, p.eps) : nf0;

      T* op = static_cast<T*>(p.out) + out_off;
      // The staged, permuted weight (kSwz): slot k's 32-byte block starts
      // k * L * SE columns after the lane's slot-0 block, and its halves are
      // swapped when bit 5 of its first column is set, which is bit 5 of the
      // slot-0 column flipped by the constant bit 5 of k * L * SE (L * SE is a
      // multiple of 32).  wA / wB: the slot-0 block's first / second half as
      // read.  Slots past the last item's vectors read the area's slack.
      const unsigned char* wA = wsm;
      const unsigned char* wB = wsm;
      if (kSwz) {
        const uint32_t wb0 = static_cast<uint32_t>(wcol) + static_cast<uint32_t>(tl * SE);
        const uint32_t x0 = 16u * ((wb0 >> 5) & 1u);
        wA = wsm + 4u * wb0 + x0;
        wB = wsm + 4u * wb0 + (16u - x0);
      }
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int v = k * L + tl;
        const bool in = k < kFull || v < nvec;
        if (!kBranchFree && !(active && in)) continue;
        const int vc = in ? v : 0;  // a slot past the item reads vector 0's weights
        // normaliser of each half of the vector, and whether each half is in
        // the item's first group
        const bool lo0 = Q == 1 || k < kG0 || (k < kG1 && v <= vb);
        const bool hi0 = Q == 1 || k < kG0 || (k < kG1 && v < vb);
        const float nlo = lo0 ? nf0 : nf1;
        const float nhi = hi0 ? nf0 : nf1;
        float r[SE];
        if (MODE == kMamba2) {
          float wv[SE];
          if (kSwz && wbytes) {
            const bool flip = ((k * L * SE) >> 5) & 1;
            const float4 lo = *reinterpret_cast<const float4*>((flip ? wB : wA) + 4 * k * L * SE);
            const float4 hi = *reinterpret_cast<const float4*>((flip ? wA : wB) + 4 * k * L * SE);
            wv[0] = lo.x, wv[1 % SE] = lo.y, wv[2 % SE] = lo.z, wv[3 % SE] = lo.w;
            wv[4 % SE] = hi.x, wv[5 % SE] = hi.y, wv[6 % SE] = hi.z, wv[7 % SE] = hi.w;
          } else {
            load_w_cols<SE>(p, c, wcol + vc * SE, wv);
          }
          mamba2_out<T, SE>(a[k], nlo, nhi, wv, r);
        } else {
          float sc[SE], gf[SE];
          if constexpr (Q == 1) {
            words_to_f32<T, NW>(wbytes ? lds_words<NW>(wsm + vc * SV)
                                       : ldg_words<NW>(static_cast<const T*>(p.w) + vc * SE),
                                sc);
          } else {
            // scale index restarts at each group: each half has its own offset
            const int jlo = in ? v * SE - (lo0 ? 0 : static_cast<int>(gs)) : 0;
            const int jhi = in ? v * SE + SE / 2 - (hi0 ? 0 : static_cast<int>(gs)) : 0;
            const T* wt = static_cast<const T*>(p.w);
            words_to_f32<T, NW / 2>(wbytes ? lds_words<NW / 2>(wsm + jlo * ES)
                                           : ldg_words<NW / 2>(wt + jlo),
                                    sc);
            words_to_f32<T, NW / 2>(wbytes ? lds_words<NW / 2>(wsm + jhi * ES)
                                           : ldg_words<NW / 2>(wt + jhi),
                                    sc + SE / 2);
          }
          words_to_f32<T, NW>(gr[k], gf);
          float sgv[SE];
          silu_vec<T, SE>(gf, sgv);
          onnx_out<SE>(a[k], nlo, nhi, sc, sgv, r);
        }
        const Words<NW> ow = f32_to_words<T, NW>(r);
        if (active && in) stg_words<NW>(op + v * SE, ow);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
#ifdef GGRN_TIMELINE
  if (lane == 0 && GGRN_TIMELINE_ON) {
    atomicMax(&GGRN_TIMELINE_AT(p, 3), timeline_now());
    if (warp == 0) {
      GGRN_TIMELINE_AT(p, 2) = tl_first;
      GGRN_TIMELINE_AT(p, 4) = tl_units;
    }
  }
#endif
}

// Launch one instantiation, opting in to more than 48 KB of dynamic shared
// memory once per device (the flag is per kernel: a template on the kernel
// itself, not on its type, which every instantiation shares).
template <auto kernel>
cudaError_t launch_stream_kernel(const KParams& k, const Plan& p, cudaStream_t s) {
  static unsigned long long opted_in = 0;  // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (p.smem > 48 * 1024 && !(__atomic_load_n(&opted_in, __ATOMIC_ACQUIRE) & bit)) {
    // the device's whole per-block limit less the kernel's static shared
    // memory, so later launches of this kernel with a larger ring need no
    // further call
    int limit = 0;
    e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             limit - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&opted_in, bit, __ATOMIC_RELEASE);
  }
  return launch_kernel(kernel, k, p, s);
}

template <typename T, int MODE, int SV, int Q>
cudaError_t launch_stream_sv(const KParams& k, const Plan& p, cudaStream_t s) {
  switch (p.lanes) {
    case 1: return launch_stream_kernel<k_stream<T, MODE, 1, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    case 2: return launch_stream_kernel<k_stream<T, MODE, 2, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    case 4: return launch_stream_kernel<k_stream<T, MODE, 4, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    case 8: return launch_stream_kernel<k_stream<T, MODE, 8, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    case 16: return launch_stream_kernel<k_stream<T, MODE, 16, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    case 32: return launch_stream_kernel<k_stream<T, MODE, 32, 4, SV, Q, kStreamMaxWarps>>(k, p, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

// The team shapes k_stream's static slot ranges assume (kFull, kG0, kG1):
// 4 vectors a lane with 2L < nvec <= 4L, or 4 lanes x 7 vectors with
// 17 <= nvec <= 27; pairs of groups have an odd vector count.
inline bool stream_shape_ok(const Plan& p) {
  if (p.items_groups == 2 && p.nvec % 2 == 0) return false;
  if (p.vpl == 7) return p.lanes == 4 && p.nvec >= 17 && p.nvec <= 27;
  return p.vpl == 4 && p.nvec > 2 * p.lanes && p.nvec <= 4 * p.lanes;
}

template <typename T, int MODE>
cudaError_t launch_stream(const KParams& k, const Plan& p, cudaStream_t s) {
  if (!stream_shape_ok(p)) return cudaErrorInvalidConfiguration;
  if (p.smem_vec_bytes == 16 && p.items_groups == 2 && p.lanes == 4 && p.vpl == 7)
    return launch_stream_kernel<k_stream<T, MODE, 4, 7, 16, 2, stream_max_warps(MODE, 7)>>(k, p, s);
  if (p.vpl != 4) return cudaErrorInvalidConfiguration;
  if (p.smem_vec_bytes == 16 && p.items_groups == 1) return launch_stream_sv<T, MODE, 16, 1>(k, p, s);
  if (p.smem_vec_bytes == 16 && p.items_groups == 2) return launch_stream_sv<T, MODE, 16, 2>(k, p, s);
  if (p.smem_vec_bytes == 8 && p.items_groups == 1) return launch_stream_sv<T, MODE, 8, 1>(k, p, s);
  return cudaErrorInvalidConfiguration;
}

}  // namespace ggrn
