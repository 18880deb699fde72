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
// Waits are bounded: after kWaitLimit polls a thread records a fault bit in
// the library's device status word and stops; the producer lane then waits
// (again bounded) until every copy it issued has landed, so no copy targets
// the shared memory of a finished CTA.
#pragma once

#include "ggrn_kernels.cuh"

namespace ggrn {

// At most kWaitLimit polls, each suspending for at most ~kWaitHintNs: a wait
// gives up after about a second (a normal wait lasts microseconds).
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kWaitHintNs = 1000;
// Fault bits of the device status word.
constexpr uint32_t kFaultConsumerWait = 1u;
constexpr uint32_t kFaultProducerWait = 2u;
constexpr uint32_t kFaultDrainWait = 4u;
// Unit shapes: ug consecutive groups of contiguous rows (flat), ug groups
// inside one row (chunk), or rows_per_unit whole rows copied row by row.
constexpr int kUnitFlat = 0;
constexpr int kUnitChunk = 1;
constexpr int kUnitRows = 2;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kWaitHintNs)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
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

// Round to T and widen back, element-wise (identity for f32).
template <typename T, int N>
__device__ __forceinline__ void round_to_t(float* f) {
  if constexpr (sizeof(T) != 4) {
#pragma unroll
    for (int e = 0; e < N; e += 2) Elem<T>::round_pair(f[e], f[e + 1]);
  }
}

// ---------------------------------------------------------------------------
// k_stream: TEAM consumers.  SV = bytes per shared-memory vector (16 or 8),
// SE = elements per vector, L lanes per team, VPL vectors per lane, Q groups
// per team item (1, or 2 for groups of an odd number of half vectors).
// Dynamic shared memory: [stages][y chunk | gate chunk] then the barriers.
// ---------------------------------------------------------------------------
template <typename T, int MODE, int L, int VPL, int SV, int Q>
__global__ void __launch_bounds__(17 * 32, 1) k_stream(const KParams p) {
  constexpr int ES = sizeof(T);
  constexpr int SE = SV / ES;
  constexpr int NW = SV / 4;
  constexpr int TPW = 32 / L;  // teams (items) per warp
  extern __shared__ __align__(128) unsigned char smem[];

  const int W = p.consumer_warps;
  const int NS = p.stages;
  const uint32_t sb = p.stage_bytes;  // bytes of one tensor's chunk slot (128-aligned)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The weight (MAMBA2 f32 [width], ONNX scale [C]) is staged once per CTA
  // after the ring when it fits: every unit then reads it from shared memory.
  unsigned char* wsm = smem + static_cast<size_t>(2) * NS * sb;
  const uint32_t wbytes = p.w_smem_bytes;                 // 0: read from global
  const uint32_t warea = (wbytes + 127u) & ~127u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + warea);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + NS);
  const uint32_t wbar = smem_u32(bars + 2 * NS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, W);
    }
    mbar_init(wbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int64_t gs = p.gs;
  if (warp == W) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    if (wbytes) {
      mbar_expect_tx(wbar, wbytes);
      bulk_g2s(smem_u32(wsm), p.w, wbytes, wbar);
    }
    int64_t i = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      const int s = static_cast<int>(i % NS);
      if (i >= NS && !mbar_wait(empty0 + 8 * s, static_cast<uint32_t>((i / NS) - 1) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t full = full0 + 8 * s;
      unsigned char* st = smem + static_cast<size_t>(2) * s * sb;
      if (p.unit_mode == kUnitRows) {
        // R whole rows, one copy per row and tensor, packed in the slot
        const int64_t row0 = u * p.rows_per_unit;
        const int64_t nr = min(static_cast<int64_t>(p.rows_per_unit), p.rows - row0);
        const uint32_t rb = static_cast<uint32_t>(p.width * ES);
        mbar_expect_tx(full, static_cast<uint32_t>(2 * nr) * rb);
        for (int64_t r = 0; r < nr; ++r) {
          bulk_g2s(smem_u32(st + r * rb), static_cast<const T*>(p.y) + (row0 + r) * p.ys, rb, full);
          bulk_g2s(smem_u32(st + sb + r * rb), static_cast<const T*>(p.gate) + (row0 + r) * p.gts,
                   rb, full);
        }
      } else {
        int64_t yo, go, ngroups;
        if (p.unit_mode == kUnitFlat) {
          const int64_t g0 = u * p.ug;
          ngroups = min(static_cast<int64_t>(p.ug), p.total_groups - g0);
          yo = go = g0 * gs;
        } else {
          const int64_t row = div_by(u, p.units_per_row, p.div_magic);
          const int64_t c0 = (u - row * p.units_per_row) * p.ug * gs;
          ngroups = p.ug;
          yo = row * p.ys + c0;
          go = row * p.gts + c0;
        }
        const uint32_t bytes = static_cast<uint32_t>(ngroups * gs * ES);
        mbar_expect_tx(full, 2 * bytes);
        bulk_g2s(smem_u32(st), static_cast<const T*>(p.y) + yo, bytes, full);
        bulk_g2s(smem_u32(st + sb), static_cast<const T*>(p.gate) + go, bytes, full);
      }
    }
    if (!ok) atomicOr(p.fault, kFaultProducerWait);
    // Every issued copy lands before this thread leaves: wait for the last
    // phase of each stage used (already complete in the normal course).
    const int64_t n_issued = i;
    for (int s = 0; s < NS && s < n_issued; ++s) {
      const int64_t last = s + ((n_issued - 1 - s) / NS) * NS;
      if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>(last / NS) & 1u))
        atomicOr(p.fault, kFaultDrainWait);
    }
    if (wbytes && !mbar_wait(wbar, 0)) atomicOr(p.fault, kFaultDrainWait);
    return;
  }
  if (wbytes && !mbar_wait(wbar, 0)) {
    if (lane == 0) atomicOr(p.fault, kFaultConsumerWait);
    return;
  }

  // ---------------- consumers ----------------
  // A team takes an "item" of Q consecutive groups.  Q = 2 pairs groups whose
  // bytes are an odd multiple of half a vector: the pair is whole 16-byte
  // vectors, and the one vector across the boundary (vector vb) splits at its
  // middle, its low half ending the first group.
  const int team = lane / L;
  const int tl = lane & (L - 1);
  const int nvec = static_cast<int>(Q * gs / SE);
  const int vb = static_cast<int>(gs / SE);
  const int items_per_pass = W * TPW;
  int64_t i = 0;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    const int s = static_cast<int>(i % NS);
    if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>(i / NS) & 1u)) {
      if (lane == 0) atomicOr(p.fault, kFaultConsumerWait);
      break;
    }
    // unit -> first group (flattened) and its row/column origin
    int64_t g0 = 0, ngroups, row_u = 0, col_u = 0;
    if (p.unit_mode == kUnitFlat) {
      g0 = u * p.ug;
      ngroups = min(static_cast<int64_t>(p.ug), p.total_groups - g0);
    } else if (p.unit_mode == kUnitChunk) {
      row_u = div_by(u, p.units_per_row, p.div_magic);
      col_u = (u - row_u * p.units_per_row) * p.ug * gs;
      ngroups = p.ug;
    } else {
      row_u = u * p.rows_per_unit;
      ngroups = min(static_cast<int64_t>(p.rows_per_unit), p.rows - row_u) * p.groups;
    }
    const int nitems = static_cast<int>(ngroups / Q);
    const unsigned char* sy = smem + static_cast<size_t>(2) * s * sb;
    const unsigned char* sg = sy + sb;
    for (int pass = 0; pass * items_per_pass < nitems; ++pass) {
      const int item = pass * items_per_pass + warp * TPW + team;
      const bool active = item < nitems;
      const int gl = item * Q;  // first group of the item within the unit
      // output origin and weight column of that group
      int64_t out_off, wcol;
      if (p.unit_mode == kUnitFlat) {
        const int64_t G = g0 + gl;
        out_off = G * gs;  // flat: out rows are contiguous
        const int64_t row = div_by(G, p.groups, p.div_magic2);
        wcol = (G - row * p.groups) * gs;
      } else if (p.unit_mode == kUnitChunk) {
        out_off = row_u * p.os + col_u + gl * gs;
        wcol = col_u + gl * gs;
      } else {
        const int r = gl / static_cast<int>(p.groups);   // row within the unit
        wcol = (gl - r * p.groups) * gs;
        out_off = (row_u + r) * p.os + wcol;
      }
      const unsigned char* gy = sy + static_cast<size_t>(gl) * gs * ES;
      const unsigned char* gg = sg + static_cast<size_t>(gl) * gs * ES;

      Words<NW> yr[VPL], gr[VPL];
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int v = k * L + tl;
        if (active && v < nvec) {
          yr[k] = lds_words<NW>(gy + v * SV);
          gr[k] = lds_words<NW>(gg + v * SV);
        } else {
#pragma unroll
          for (int q = 0; q < NW; ++q) yr[k].w[q] = 0u, gr[k].w[q] = 0u;
        }
      }
      float a[VPL][SE];
      float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        float yf[SE];
        words_to_f32<T, NW>(yr[k], yf);
        if (MODE == kMamba2) {
          float gf[SE];
          words_to_f32<T, NW>(gr[k], gf);
#pragma unroll
          for (int e = 0; e < SE; ++e) a[k][e] = yf[e] * silu<T>(gf[e]);
        } else {
#pragma unroll
          for (int e = 0; e < SE; ++e) a[k][e] = yf[e];
        }
        if constexpr (Q == 1) {
#pragma unroll
          for (int e = 0; e < SE; ++e) s0 = fmaf(a[k][e], a[k][e], s0);
        } else {
          float h0 = 0.0f, h1 = 0.0f;
#pragma unroll
          for (int e = 0; e < SE / 2; ++e) h0 = fmaf(a[k][e], a[k][e], h0);
#pragma unroll
          for (int e = SE / 2; e < SE; ++e) h1 = fmaf(a[k][e], a[k][e], h1);
          const int v = k * L + tl;
          s0 += (v < vb) ? h0 + h1 : (v == vb ? h0 : 0.0f);
          s1 += (v > vb) ? h0 + h1 : (v == vb ? h1 : 0.0f);
        }
      }
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        if constexpr (Q == 2) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      const float nf0 = normaliser(s0, p.gs_f, p.eps);
      const float nf1 = (Q == 2) ? normaliser(s1, p.gs_f, p.eps) : nf0;

      T* op = static_cast<T*>(p.out) + out_off;
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int v = k * L + tl;
        if (active && v < nvec) {
          // normaliser of each half of the vector
          const float nlo = (Q == 1 || v <= vb) ? nf0 : nf1;
          const float nhi = (Q == 1 || v < vb) ? nf0 : nf1;
          float r[SE];
          if (MODE == kMamba2) {
            float wv[SE];
            const int64_t wi = wcol + v * SE;
#pragma unroll
            for (int q = 0; q < SE; q += 4 > SE ? SE : 4) {
              if (SE >= 4) {
                const float4 w4 =
                    wbytes ? *reinterpret_cast<const float4*>(wsm + 4 * (wi + q))
                           : __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.w) + wi + q));
                wv[q] = w4.x, wv[(q + 1) % SE] = w4.y, wv[(q + 2) % SE] = w4.z,
                wv[(q + 3) % SE] = w4.w;
              } else {
                const float2 w2 =
                    wbytes ? *reinterpret_cast<const float2*>(wsm + 4 * (wi + q))
                           : __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(p.w) + wi + q));
                wv[q] = w2.x, wv[(q + 1) % SE] = w2.y;
              }
            }
#pragma unroll
            for (int e = 0; e < SE; ++e) r[e] = a[k][e] * (e < SE / 2 ? nlo : nhi);
            round_to_t<T, SE>(r);
#pragma unroll
            for (int e = 0; e < SE; ++e) r[e] = wv[e] * r[e];
          } else {
            float sc[SE], gf[SE];
            if constexpr (Q == 1) {
              words_to_f32<T, NW>(wbytes ? lds_words<NW>(wsm + v * SV)
                                         : ldg_words<NW>(static_cast<const T*>(p.w) + v * SE),
                                  sc);
            } else {
              // scale index restarts at each group: each half has its own offset
              const int jlo = v * SE - (v <= vb ? 0 : static_cast<int>(gs));
              const int jhi = v * SE + SE / 2 - (v < vb ? 0 : static_cast<int>(gs));
              const T* wt = static_cast<const T*>(p.w);
              words_to_f32<T, NW / 2>(wbytes ? lds_words<NW / 2>(wsm + jlo * ES)
                                             : ldg_words<NW / 2>(wt + jlo),
                                      sc);
              words_to_f32<T, NW / 2>(wbytes ? lds_words<NW / 2>(wsm + jhi * ES)
                                             : ldg_words<NW / 2>(wt + jhi),
                                      sc + SE / 2);
            }
            words_to_f32<T, NW>(gr[k], gf);
#pragma unroll
            for (int e = 0; e < SE; ++e)
              r[e] = ((a[k][e] * (e < SE / 2 ? nlo : nhi)) * sc[e]) * silu<T>(gf[e]);
          }
          stg_words<NW>(op + v * SE, f32_to_words<T, NW>(r));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
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
    // the device's whole per-block limit, so later launches of this kernel
    // with a larger ring need no further call
    int limit = 0;
    e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&opted_in, bit, __ATOMIC_RELEASE);
  }
  return launch_kernel(kernel, k, p, s);
}

template <typename T, int MODE, int SV, int Q>
cudaError_t launch_stream_sv(const KParams& k, const Plan& p, cudaStream_t s) {
  switch (p.lanes) {
    case 1: return launch_stream_kernel<k_stream<T, MODE, 1, 4, SV, Q>>(k, p, s);
    case 2: return launch_stream_kernel<k_stream<T, MODE, 2, 4, SV, Q>>(k, p, s);
    case 4: return launch_stream_kernel<k_stream<T, MODE, 4, 4, SV, Q>>(k, p, s);
    case 8: return launch_stream_kernel<k_stream<T, MODE, 8, 4, SV, Q>>(k, p, s);
    case 16: return launch_stream_kernel<k_stream<T, MODE, 16, 4, SV, Q>>(k, p, s);
    case 32: return launch_stream_kernel<k_stream<T, MODE, 32, 4, SV, Q>>(k, p, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

template <typename T, int MODE>
cudaError_t launch_stream(const KParams& k, const Plan& p, cudaStream_t s) {
  if (p.smem_vec_bytes == 16 && p.items_groups == 2 && p.lanes == 4 && p.vpl == 7)
    return launch_stream_kernel<k_stream<T, MODE, 4, 7, 16, 2>>(k, p, s);
  if (p.vpl != 4) return cudaErrorInvalidConfiguration;
  if (p.smem_vec_bytes == 16 && p.items_groups == 1) return launch_stream_sv<T, MODE, 16, 1>(k, p, s);
  if (p.smem_vec_bytes == 16 && p.items_groups == 2) return launch_stream_sv<T, MODE, 16, 2>(k, p, s);
  if (p.smem_vec_bytes == 8 && p.items_groups == 1) return launch_stream_sv<T, MODE, 8, 1>(k, p, s);
  return cudaErrorInvalidConfiguration;
}

}  // namespace ggrn
