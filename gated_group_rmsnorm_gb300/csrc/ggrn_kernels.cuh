// ggrn_kernels.cuh -- sm_103a kernels of the fused gated group-RMSNorm.
//
// The operation ("gated_group_rmsnorm" Mojo module page, math block; and
// "com.microsoft.GatedRMSNorm" README, Description), per row and per group of
// gs contiguous columns:
//   MAMBA2: gated = y*silu(gate); m2 = sum gated^2; nf = rsqrt(m2/gs + eps);
//           out = cast_T(w[col] * cast_T(gated*nf))
//   ONNX:   m2 = sum x^2; nf as above; out = cast_T(((x*nf)*scale[j])*silu(gate))
//
// The op is a streaming reduction bound by HBM bandwidth: each element of y
// and gate is read once and each output written once (6 bytes per element for
// 16-bit T).  Every family below keeps the whole group on chip between the
// reduction and the epilogue so nothing is re-read from HBM, moves data in
// 16-byte vectors (8 x 16-bit or 4 x f32 per lane per instruction, one
// contiguous 512-byte run per warp instruction when a warp covers a group),
// marks y/gate loads L1::no_allocate and output stores evict-first so the
// small weight stays cached, and reduces in f32 with warp shuffles.
//
// Families:
//   k_team      a team of LANES (1..32, power of two) lanes of one warp per
//               group, VPL vectors per lane; a segmented xor butterfly over the
//               low lane bits reduces each team independently, so 32/LANES
//               groups share a warp with no shared memory and no barrier.
//   k_wide      one CTA per group; warp butterflies, then one shared-memory
//               exchange and one barrier.
//   k_straddle  one warp per row chunk holding whole groups, for group sizes
//               that are not a multiple of the vector: each vector's squares
//               are split at the (at most one) group boundary it crosses, the
//               two partials go to warp-private shared memory, and one lane
//               per group adds its vectors' partials in a fixed order.
//   k_scalar    element loads, LANES lanes per group, two passes over the
//               group (a correctness path for any alignment and size).
//
// All reductions have a fixed order, so results are deterministic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ggrn_internal.h"

namespace ggrn {

// ---------------------------------------------------------------------------
// Element traits: 16-byte vector width, unpack/pack, rounding to T.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int E = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[E]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[E]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ __forceinline__ static void round_pair(float& a, float& b) { (void)a, (void)b; }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
  // f32 outputs carry a relative tolerance of 1e-5 at every magnitude: their
  // silu uses the accurate exponential and the IEEE divide.
  static constexpr bool kExactSilu = true;
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void unpack2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // RNE
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[E]) {
    unpack2(v.x, f[0], f[1]);
    unpack2(v.y, f[2], f[3]);
    unpack2(v.z, f[4], f[5]);
    unpack2(v.w, f[6], f[7]);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[E]) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
  __device__ __forceinline__ static void round_pair(float& a, float& b) { unpack2(pack2(a, b), a, b); }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    unsigned short h = __ldg(static_cast<const unsigned short*>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
  static constexpr bool kExactSilu = false;
};

template <>
struct Elem<__half> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void unpack2(uint32_t u, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);  // RNE
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[E]) {
    unpack2(v.x, f[0], f[1]);
    unpack2(v.y, f[2], f[3]);
    unpack2(v.z, f[4], f[5]);
    unpack2(v.w, f[6], f[7]);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[E]) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
  __device__ __forceinline__ static void round_pair(float& a, float& b) { unpack2(pack2(a, b), a, b); }
  __device__ __forceinline__ static float load1(const void* p, int64_t i) {
    return __half2float(__ldg(static_cast<const __half*>(p) + i));
  }
  __device__ __forceinline__ static void store1(void* p, int64_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  }
  static constexpr bool kExactSilu = false;
};

// ---------------------------------------------------------------------------
// Memory helpers.
// ---------------------------------------------------------------------------
// 16-byte streaming load: read-only path, no L1 allocation (y and gate are
// read exactly once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// 16-byte evict-first store (out is written once and not re-read here).
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  __stcs(static_cast<uint4*>(p), v);
}

// 16-byte cached load of the weight (re-read by every row; stays in L1/L2).
__device__ __forceinline__ uint4 ld_weight(const void* p) {
  return __ldg(static_cast<const uint4*>(p));
}

// Programmatic dependent launch: wait for the previous kernel in the stream
// (its writes visible) before touching global memory; let the next kernel's
// CTAs be scheduled as soon as ours have all started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Math helpers.
// ---------------------------------------------------------------------------
// Approximate base-2 exponential and reciprocal of the PTX ISA (one MUFU
// operation each, subnormal results flushed to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// silu(b) = b * sigmoid(b) = b / (1 + exp(-b)), in f32.
// 16-bit T: exp(-b) = 2^(-b * log2(e)) and the divide as a reciprocal
// times b, two MUFU operations per element.  Numerator and denominator are
// both scaled by 1/16 (exactly), so the reciprocal's argument stays below
// 2^126 for every finite exponential and the quotient is never flushed: the
// result keeps the exact limits of the definition -- b itself once
// exp(-b) < 2^-24, -0 once exp(-b) overflows, NaN for b = -inf.
template <typename T>
__device__ __forceinline__ float silu(float b) {
  if (Elem<T>::kExactSilu) return b / (1.0f + expf(-b));
  const float e = ex2_approx(b * -1.4426950408889634f);
  const float d = fmaf(e, 0.0625f, 0.0625f);
  return (b * 0.0625f) * rcp_approx(d);
}

// ---------------------------------------------------------------------------
// Packed f32 pairs.  sm_100-family SMs execute add/mul/fma on the two f32
// halves of a 64-bit register pair in one instruction (PTX .f32x2), each
// half rounded exactly as the scalar .rn instruction rounds it.  The
// elementwise chain of the vector kernels runs on element pairs (2i, 2i+1),
// halving its FMA-pipe instructions; MUFU operations stay scalar.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
// (d0, d1) = (a0 * b0, a1 * b1)
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)));
  upk2(r, d0, d1);
}
// (d0, d1) = (fma(a0, b0, c0), fma(a1, b1, c1))
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)), "l"(pk2(c0, c1)));
  upk2(r, d0, d1);
}

// silu of two elements: the operations of silu<T>, on pairs.
template <typename T>
__device__ __forceinline__ void silu2(float b0, float b1, float& s0, float& s1) {
  if (Elem<T>::kExactSilu) {
    s0 = silu<T>(b0);
    s1 = silu<T>(b1);
    return;
  }
  constexpr float kNegLog2e = -1.4426950408889634f;
  float t0, t1, d0, d1, q0, q1;
  mul2(t0, t1, b0, b1, kNegLog2e, kNegLog2e);
  fma2(d0, d1, ex2_approx(t0), ex2_approx(t1), 0.0625f, 0.0625f, 0.0625f, 0.0625f);
  mul2(q0, q1, b0, b1, 0.0625f, 0.0625f);
  mul2(s0, s1, q0, q1, rcp_approx(d0), rcp_approx(d1));
}

// a[e] = y[e] * silu(g[e]), e < N (N even).
template <typename T, int N>
__device__ __forceinline__ void gated_vec(const float* y, const float* g, float* a) {
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    float s0, s1;
    silu2<T>(g[e], g[e + 1], s0, s1);
    mul2(a[e], a[e + 1], y[e], y[e + 1], s0, s1);
  }
}
// s[e] = silu(g[e]), e < N (N even).
template <typename T, int N>
__device__ __forceinline__ void silu_vec(const float* g, float* s) {
#pragma unroll
  for (int e = 0; e < N; e += 2) silu2<T>(g[e], g[e + 1], s[e], s[e + 1]);
}
// (c0, c1) += squares of a[e], e < N (N even): even elements into c0, odd
// into c1.
template <int N>
__device__ __forceinline__ void sumsq2(const float* a, float& c0, float& c1) {
#pragma unroll
  for (int e = 0; e < N; e += 2) fma2(c0, c1, a[e], a[e + 1], a[e], a[e + 1], c0, c1);
}

// floor(n / d) for the work-item counters (row = item / items_per_row).  The
// host passes magic = floor(2^64 / d) + 1 when every n is below 2^32: then
// n * magic / 2^64 exceeds n / d by less than 2^-32 <= 1/d, which cannot
// carry past the next integer, so the high word of the product is the exact
// quotient (division by an invariant integer, Granlund and Montgomery 1994).
// magic == 0 selects the plain 64-bit division.
__device__ __forceinline__ int64_t div_by(int64_t n, int64_t d, uint64_t magic) {
  if (d == 1) return n;
  if (magic != 0) return static_cast<int64_t>(__umul64hi(static_cast<uint64_t>(n), magic));
  return n / d;
}

// nf = rsqrt(m2 / gs + eps): the IEEE divide (the definition divides the
// sum by the group size), then the PTX ISA's approximate reciprocal square
// root (rsqrt.approx.f32: one MUFU operation, an error of a few f32 ulps,
// subnormal arguments kept, rsqrt(0) = +inf, rsqrt(+inf) = +0).  Its error is
// far below half an ulp of the 16-bit output; where it moves the rounding of
// gated * nf, the move is one of the flips the tolerance admits, as for the
// order of the sum.  Against the correctly rounded rsqrt it measured +0.5 %
// (prefill) and +1.2 % (odd span): the normaliser sits on every group's
// dependency chain.
__device__ __forceinline__ float normaliser(float m2, float gs_f, float eps) {
  const float v = __fdiv_rn(m2, gs_f) + eps;
  float r;
  asm("rsqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Mamba-2 output values of N elements (N even), before the final rounding:
// r = w * cast_T(gated * nf), with nf = nlo on the first N/2 elements and
// nhi on the rest (the two groups of a vector split at its middle).
template <typename T, int N>
__device__ __forceinline__ void mamba2_out(const float* gated, float nlo, float nhi,
                                           const float* w, float* r) {
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    const float nf = e < N / 2 ? nlo : nhi;
    mul2(r[e], r[e + 1], gated[e], gated[e + 1], nf, nf);
    Elem<T>::round_pair(r[e], r[e + 1]);
    mul2(r[e], r[e + 1], w[e], w[e + 1], r[e], r[e + 1]);
  }
}

// ONNX output values of N elements (N even): r = ((x * nf) * scale) * silu,
// nf split as in mamba2_out.
template <int N>
__device__ __forceinline__ void onnx_out(const float* x, float nlo, float nhi, const float* sc,
                                         const float* sg, float* r) {
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    const float nf = e < N / 2 ? nlo : nhi;
    mul2(r[e], r[e + 1], x[e], x[e + 1], nf, nf);
    mul2(r[e], r[e + 1], r[e], r[e + 1], sc[e], sc[e + 1]);
    mul2(r[e], r[e + 1], r[e], r[e + 1], sg[e], sg[e + 1]);
  }
}

// Mamba-2 epilogue on one vector: out = cast_T(w * cast_T(gated * nf)).
template <typename T>
__device__ __forceinline__ uint4 epilogue_mamba2(const float (&gated)[Elem<T>::E], float nf,
                                                 const float* wv) {
  float t[Elem<T>::E];
  mamba2_out<T, Elem<T>::E>(gated, nf, nf, wv, t);
  return Elem<T>::pack(t);
}

// ONNX epilogue on one vector: out = cast_T(((x * nf) * scale) * silu(gate)).
template <typename T>
__device__ __forceinline__ uint4 epilogue_onnx(const float (&x)[Elem<T>::E],
                                               const float (&sg)[Elem<T>::E], float nf,
                                               const float (&sc)[Elem<T>::E]) {
  float r[Elem<T>::E];
  onnx_out<Elem<T>::E>(x, nf, nf, sc, sg, r);
  return Elem<T>::pack(r);
}

// Weight of one vector: MAMBA2 -> E floats of w at column col (16-byte
// aligned); ONNX -> E values of scale (T) at index j, widened.
template <typename T, int MODE>
__device__ __forceinline__ void load_weight_vec(const void* w, int64_t idx, float (&wv)[Elem<T>::E]) {
  constexpr int E = Elem<T>::E;
  if (MODE == kMamba2) {
    const float* wp = static_cast<const float*>(w) + idx;
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      uint4 u = ld_weight(wp + 4 * q);
      wv[4 * q + 0] = __uint_as_float(u.x);
      wv[4 * q + 1] = __uint_as_float(u.y);
      wv[4 * q + 2] = __uint_as_float(u.z);
      wv[4 * q + 3] = __uint_as_float(u.w);
    }
  } else {
    uint4 u = ld_weight(static_cast<const T*>(w) + idx);
    Elem<T>::unpack(u, wv);
  }
}

// Half a vector (8 bytes) of the ONNX scale (T) at index j, widened.
template <typename T>
__device__ __forceinline__ void load_half_scale(const void* w, int64_t j, float* out) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const T*>(w) + j));
  if constexpr (sizeof(T) == 4) {
    out[0] = __uint_as_float(u.x);
    out[1] = __uint_as_float(u.y);
  } else {
    Elem<T>::unpack2(u.x, out[0], out[1]);
    Elem<T>::unpack2(u.y, out[2], out[3]);
  }
}

// ---------------------------------------------------------------------------
// TEAM: LANES lanes per item, VPL 16-byte vectors per lane per tensor.  An
// item is Q consecutive groups: Q = 1, or Q = 2 for groups whose bytes are an
// odd multiple of 8 (the pair is whole 16-byte vectors; the vector across
// the boundary, vector vb, splits at its middle and two accumulators keep the
// groups apart).  Vector v of an item (0 <= v < nvec) sits in slot
// k = v / LANES of lane v % LANES, so each load instruction of a team covers
// LANES consecutive vectors.  Teams are aligned LANES-lane segments of a
// warp; the xor butterfly with offsets < LANES never crosses a segment.
// ---------------------------------------------------------------------------
// Resident CTAs per SM the register budget targets: ONNX keeps the gate's
// raw words until the epilogue, so its kernels get a larger budget.
constexpr int team_min_blocks(int mode) { return mode == kOnnx ? 3 : 4; }

template <typename T, int MODE, int LANES, int VPL, int Q>
__global__ void __launch_bounds__(256, team_min_blocks(MODE)) k_team(const KParams p) {
  constexpr int E = Elem<T>::E;
  pdl_wait();
  pdl_launch_dependents();

  const int lane = threadIdx.x & (LANES - 1);
  const int teams_per_warp = 32 / LANES;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int team_in_warp = (threadIdx.x & 31) / LANES;
  const int vb = static_cast<int>(p.gs / E);  // Q == 2: the vector split at its middle

  for (int64_t base = warp_id * teams_per_warp; base < p.items;
       base += warps_total * teams_per_warp) {
    const int64_t item = base + team_in_warp;
    const bool active = item < p.items;
    int64_t row = 0, g = 0;
    if (active) {
      row = div_by(item, p.items_per_row, p.div_magic);
      g = (item - row * p.items_per_row) * Q;  // first group of the item
    }
    const int64_t col0 = g * p.gs;
    const T* yp = static_cast<const T*>(p.y) + row * p.ys + col0;
    const T* gp = static_cast<const T*>(p.gate) + row * p.gts + col0;

    uint4 yr[VPL], gr[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * LANES + lane;
      if (active && v < p.nvec) {
        yr[k] = ld_stream(yp + (int64_t)v * E);
        gr[k] = ld_stream(gp + (int64_t)v * E);
      } else {
        yr[k] = make_uint4(0u, 0u, 0u, 0u);
        gr[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    }

    // MAMBA2: a = gated = y * silu(gate).  ONNX: a = x; the gate enters only
    // the epilogue, so its raw bits wait there and silu is evaluated once.
    float a[VPL][E];
    float s0 = 0.0f, s1 = 0.0f;
    float c0 = 0.0f, c1 = 0.0f;  // Q == 1: even / odd element partial sums
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      float yf[E];
      Elem<T>::unpack(yr[k], yf);
      if (MODE == kMamba2) {
        float gf[E];
        Elem<T>::unpack(gr[k], gf);
        gated_vec<T, E>(yf, gf, a[k]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) a[k][e] = yf[e];
      }
      if constexpr (Q == 1) {
        sumsq2<E>(a[k], c0, c1);
      } else {
        float h0a = 0.0f, h0b = 0.0f, h1a = 0.0f, h1b = 0.0f;
        sumsq2<E / 2>(a[k], h0a, h0b);
        sumsq2<E / 2>(a[k] + E / 2, h1a, h1b);
        const float h0 = h0a + h0b, h1 = h1a + h1b;
        const int v = k * LANES + lane;
        s0 += (v < vb) ? h0 + h1 : (v == vb ? h0 : 0.0f);
        s1 += (v > vb) ? h0 + h1 : (v == vb ? h1 : 0.0f);
      }
    }
    if constexpr (Q == 1) s0 = c0 + c1;
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      if constexpr (Q == 2) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    const float nf0 = normaliser(s0, p.gs_f, p.eps);
    const float nf1 = (Q == 2) ? normaliser(s1, p.gs_f, p.eps) : nf0;

    T* op = static_cast<T*>(p.out) + row * p.os + col0;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * LANES + lane;
      if (active && v < p.nvec) {
        // normaliser of each half of the vector
        const float nlo = (Q == 1 || v <= vb) ? nf0 : nf1;
        const float nhi = (Q == 1 || v < vb) ? nf0 : nf1;
        float wv[E];
        uint4 o;
        if (MODE == kMamba2) {
          load_weight_vec<T, MODE>(p.w, col0 + (int64_t)v * E, wv);
          float t[E];
          mamba2_out<T, E>(a[k], nlo, nhi, wv, t);
          o = Elem<T>::pack(t);
        } else {
          if constexpr (Q == 1) {
            load_weight_vec<T, MODE>(p.w, (int64_t)v * E, wv);
          } else {
            // the scale index restarts with each group: one offset per half
            const int jlo = v * E - (v <= vb ? 0 : static_cast<int>(p.gs));
            const int jhi = v * E + E / 2 - (v < vb ? 0 : static_cast<int>(p.gs));
            load_half_scale<T>(p.w, jlo, wv);
            load_half_scale<T>(p.w, jhi, wv + E / 2);
          }
          float gf[E], sg[E], r[E];
          Elem<T>::unpack(gr[k], gf);
          silu_vec<T, E>(gf, sg);
          onnx_out<E>(a[k], nlo, nhi, wv, sg, r);
          o = Elem<T>::pack(r);
        }
        st_stream(op + (int64_t)v * E, o);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// WIDE: one CTA per group, VPL vectors per thread; vector v sits in slot
// v / blockDim of thread v % blockDim.  Warp partials meet in shared memory
// (double-buffered by loop parity, so one barrier per group suffices) and
// every thread adds them in the same order.
// ---------------------------------------------------------------------------
// Resident CTAs per SM the register budget targets (CTAs of at most 256
// threads): MAMBA2 six (40 registers; a 28-byte spill is cheaper than the
// latency fewer CTAs leave exposed: 6.49 -> 6.80 TB/s on 5120-wide groups,
// where seven or eight spill heavily and fall to 4 TB/s); ONNX four.
constexpr int wide_min_blocks(int mode, int maxt) {
  return maxt <= 256 ? (mode == kOnnx ? 4 : 6) : 1;
}

template <typename T, int MODE, int VPL, int MAXT>
__global__ void __launch_bounds__(MAXT, wide_min_blocks(MODE, MAXT)) k_wide(const KParams p) {
  constexpr int E = Elem<T>::E;
  __shared__ float red[2][32];
  pdl_wait();
  pdl_launch_dependents();

  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int nwarps = nthreads >> 5;
  int parity = 0;
  for (int64_t item = blockIdx.x; item < p.items; item += gridDim.x, parity ^= 1) {
    const int64_t row = div_by(item, p.groups, p.div_magic);
    const int64_t g = item - row * p.groups;
    const int64_t col0 = g * p.gs;
    const T* yp = static_cast<const T*>(p.y) + row * p.ys + col0;
    const T* gp = static_cast<const T*>(p.gate) + row * p.gts + col0;

    uint4 yr[VPL], gr[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * nthreads + tid;
      if (v < p.nvec) {
        yr[k] = ld_stream(yp + (int64_t)v * E);
        gr[k] = ld_stream(gp + (int64_t)v * E);
      } else {
        yr[k] = make_uint4(0u, 0u, 0u, 0u);
        gr[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // One vector per thread in CTAs of at most 256 threads (launches of a
    // few groups, e.g. a decode step, where each group's latency is the
    // cost): the weight is fetched with y and gate, not after the reduction,
    // so its round trip overlaps theirs (decode 960-wide: 1.57 -> 1.47 us per
    // call in a 21-call graph).  Not in the 1024-thread kernel: 9 more
    // registers there halve the resident 640-thread CTAs (-23 % at 256 rows
    // of 5120-wide groups).
    constexpr bool kPrefetchW = VPL == 1 && MAXT <= 256;
    float wpre[kPrefetchW ? E : 1];
    if constexpr (kPrefetchW) {
      if (tid < p.nvec)
        load_weight_vec<T, MODE>(p.w, (MODE == kMamba2 ? col0 : 0) + (int64_t)tid * E, wpre);
    }
    // MAMBA2: a = gated.  ONNX: a = x; the gate's raw words wait for the
    // epilogue (fewer live registers than its widened silu).
    float a[VPL][E];
    float c0 = 0.0f, c1 = 0.0f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      float yf[E];
      Elem<T>::unpack(yr[k], yf);
      if (MODE == kMamba2) {
        float gf[E];
        Elem<T>::unpack(gr[k], gf);
        gated_vec<T, E>(yf, gf, a[k]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) a[k][e] = yf[e];
      }
      sumsq2<E>(a[k], c0, c1);
    }
    float ss = c0 + c1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[parity][tid >> 5] = ss;
    __syncthreads();
    float m2 = 0.0f;
    if (MAXT > 256 && nwarps > 8) {
      // many warps (a single wide group, e.g. batch-1 decode of one
      // 7680-wide group): one shared-memory read per lane and a butterfly,
      // instead of a chain of nwarps dependent reads; the xor butterfly adds
      // each pair symmetrically, so every lane ends with the same bits
      m2 = (tid & 31) < nwarps ? red[parity][tid & 31] : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
    } else {
      for (int i = 0; i < nwarps; ++i) m2 += red[parity][i];
    }
    const float nf = normaliser(m2, p.gs_f, p.eps);

    T* op = static_cast<T*>(p.out) + row * p.os + col0;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * nthreads + tid;
      if (v < p.nvec) {
        float wv[E];
        uint4 o;
        if constexpr (kPrefetchW) {
#pragma unroll
          for (int e = 0; e < E; ++e) wv[e] = wpre[e];
        } else {
          load_weight_vec<T, MODE>(p.w, (MODE == kMamba2 ? col0 : 0) + (int64_t)v * E, wv);
        }
        if (MODE == kMamba2) {
          o = epilogue_mamba2<T>(a[k], nf, wv);
        } else {
          float gf[E], sg[E];
          Elem<T>::unpack(gr[k], gf);
          silu_vec<T, E>(gf, sg);
          o = epilogue_onnx<T>(a[k], sg, nf, wv);
        }
        st_stream(op + (int64_t)v * E, o);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// STRADDLE: group size not a multiple of E (and larger than E).  One warp
// per chunk of a row.  Chunks start at multiples of lcm(gs, E) elements, so
// they start 16-byte aligned, hold whole groups, and map vector slots to
// groups identically in every chunk.  A vector touches at most two groups and
// a group boundary falls inside it at a multiple of G = gcd(gs, E): the
// vector's squares are summed in E/G sub-blocks, and the sub-block sums are
// split at the boundary into (lo, hi) partials.  The partials go to
// warp-private shared memory; lane t then adds, in vector order, the
// partials of group t.  Shared memory per warp: part_lo[32*VPL],
// part_hi[32*VPL], nf[chunk_groups]; no block-wide barrier.
// ---------------------------------------------------------------------------
template <typename T, int MODE, int VPL, int G>
__global__ void __launch_bounds__(256, MODE == kOnnx ? 2 : 3) k_straddle(const KParams p) {
  constexpr int E = Elem<T>::E;
  constexpr int NS = E / G;          // sub-blocks per vector
  constexpr int SLOTS = 32 * VPL;
  extern __shared__ float sm[];
  const int lane = threadIdx.x & 31;
  float* part_lo = sm + (threadIdx.x >> 5) * p.warp_smem;
  float* part_hi = part_lo + SLOTS;
  float* nf_s = part_hi + SLOTS;
  pdl_wait();
  pdl_launch_dependents();

  const int gs = static_cast<int>(p.gs);
  // Slot k of this lane holds chunk vector v = 32k + lane: its first element's
  // group (floor(v*E / gs) by multiply-high with the host's magic number,
  // exact for v*E, gs < 2^11) and the offset of the next group boundary.
  int glo[VPL], bnd[VPL];
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const int e0 = (k * 32 + lane) * E;
    glo[k] = static_cast<int>(__umulhi(static_cast<unsigned>(e0), p.gs_magic));
    bnd[k] = (glo[k] + 1) * gs - e0;
  }

  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       item < p.items; item += warps_total) {
    const int64_t row = div_by(item, p.chunks_per_row, p.div_magic);
    const int64_t c0 = (item - row * p.chunks_per_row) * p.chunk_elems;
    const int clen = static_cast<int>(min(p.chunk_elems, p.width - c0));
    const int nv = clen / E;   // the width is a multiple of E: whole vectors only
    const int ng = clen / gs;
    const T* yp = static_cast<const T*>(p.y) + row * p.ys + c0;
    const T* gp = static_cast<const T*>(p.gate) + row * p.gts + c0;

    uint4 yr[VPL], gr[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int e0 = (k * 32 + lane) * E;
      if (e0 < clen) {
        yr[k] = ld_stream(yp + e0);
        gr[k] = ld_stream(gp + e0);
      } else {
        yr[k] = make_uint4(0u, 0u, 0u, 0u);
        gr[k] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float a[VPL][E];
    float sg[MODE == kOnnx ? VPL : 1][E];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * 32 + lane;
      float yf[E], gf[E];
      Elem<T>::unpack(yr[k], yf);
      Elem<T>::unpack(gr[k], gf);
      float sub[NS];
#pragma unroll
      for (int i = 0; i < NS; ++i) sub[i] = 0.0f;
      if (MODE == kMamba2) {
        gated_vec<T, E>(yf, gf, a[k]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) a[k][e] = yf[e];
        silu_vec<T, E>(gf, sg[MODE == kOnnx ? k : 0]);
      }
#pragma unroll
      for (int e = 0; e < E; ++e) sub[e / G] = fmaf(a[k][e], a[k][e], sub[e / G]);
      float lo = 0.0f, hi = 0.0f;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        if (i * G < bnd[k]) lo += sub[i];
        else hi += sub[i];
      }
      if (v < nv) {
        part_lo[v] = lo;
        part_hi[v] = hi;
      }
    }
    __syncwarp();
    for (int t = lane; t < ng; t += 32) {
      const int first = t * gs;
      const int vf = first / E;
      const int vl = (first + gs - 1) / E;
      float m2 = (vf * E >= first) ? part_lo[vf] : part_hi[vf];
      for (int v = vf + 1; v <= vl; ++v) m2 += part_lo[v];
      nf_s[t] = normaliser(m2, p.gs_f, p.eps);
    }
    __syncwarp();

    T* op = static_cast<T*>(p.out) + row * p.os + c0;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * 32 + lane;
      const int e0 = v * E;
      if (v < nv) {
        const float nf_lo = nf_s[glo[k]];
        const float nf_hi = (bnd[k] < E && glo[k] + 1 < ng) ? nf_s[glo[k] + 1] : nf_lo;
        float nfv[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) nfv[i] = (i * G < bnd[k]) ? nf_lo : nf_hi;
        float r[E];
        if (MODE == kMamba2) {
          float wv[E];
          load_weight_vec<T, MODE>(p.w, c0 + e0, wv);
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            mul2(r[e], r[e + 1], a[k][e], a[k][e + 1], nfv[e / G], nfv[(e + 1) / G]);
            Elem<T>::round_pair(r[e], r[e + 1]);
            mul2(r[e], r[e + 1], wv[e], wv[e + 1], r[e], r[e + 1]);
          }
        } else {
          // scale index j of each element: offset from its group's start
          const int jlo = e0 - glo[k] * gs;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int j = (e / G * G < bnd[k]) ? jlo + e : jlo + e - gs;
            r[e] = ((a[k][e] * nfv[e / G]) * Elem<T>::load1(p.w, j)) * sg[MODE == kOnnx ? k : 0][e];
          }
        }
        st_stream(op + e0, Elem<T>::pack(r));
      }
    }
    __syncwarp();  // the next chunk rewrites this warp's partials
  }
}

// ---------------------------------------------------------------------------
// SCALAR: LANES lanes per group, element loads (any alignment, any size),
// two passes over the group: sum of squares, then recompute and store.
// ---------------------------------------------------------------------------
template <typename T, int MODE, int LANES>
__global__ void __launch_bounds__(256) k_scalar(const KParams p) {
  pdl_wait();
  pdl_launch_dependents();

  const int lane = threadIdx.x & (LANES - 1);
  const int teams_per_warp = 32 / LANES;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int team_in_warp = (threadIdx.x & 31) / LANES;

  for (int64_t base = warp_id * teams_per_warp; base < p.items;
       base += warps_total * teams_per_warp) {
    const int64_t item = base + team_in_warp;
    const bool active = item < p.items;
    int64_t row = 0, g = 0;
    if (active) {
      row = div_by(item, p.groups, p.div_magic);
      g = item - row * p.groups;
    }
    const int64_t col0 = g * p.gs;
    const int64_t yo = row * p.ys + col0, go = row * p.gts + col0, oo = row * p.os + col0;
    float ss = 0.0f;
    if (active) {
      for (int64_t j = lane; j < p.gs; j += LANES) {
        const float y = Elem<T>::load1(p.y, yo + j);
        float a = y;
        if (MODE == kMamba2) a = y * silu<T>(Elem<T>::load1(p.gate, go + j));
        ss = fmaf(a, a, ss);
      }
    }
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float nf = normaliser(ss, p.gs_f, p.eps);
    if (active) {
      for (int64_t j = lane; j < p.gs; j += LANES) {
        const float y = Elem<T>::load1(p.y, yo + j);
        const float sgv = silu<T>(Elem<T>::load1(p.gate, go + j));
        float r;
        if (MODE == kMamba2) {
          float t = (y * sgv) * nf;
          float dummy = 0.0f;
          Elem<T>::round_pair(t, dummy);
          r = __ldg(static_cast<const float*>(p.w) + col0 + j) * t;
        } else {
          r = ((y * nf) * Elem<T>::load1(p.w, j)) * sgv;
        }
        Elem<T>::store1(p.out, oo + j, r);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Shared-memory barriers (mbarrier) and bounded waits, used by the cluster
// kernel below and by the streaming family (ggrn_stream.cuh).
// ---------------------------------------------------------------------------
// At most kWaitLimit polls, each suspending for at most ~kWaitHintNs: a wait
// gives up after about a second (a normal wait lasts microseconds).
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kWaitHintNs = 1000;
// Fault bits of the device status word.
constexpr uint32_t kFaultConsumerWait = 1u;
constexpr uint32_t kFaultProducerWait = 2u;
constexpr uint32_t kFaultDrainWait = 4u;
constexpr uint32_t kFaultClaim = 8u;
constexpr uint32_t kFaultClusterWait = 32u;
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
// Raise the bytes the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_add_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
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

// ---------------------------------------------------------------------------
// k_wide_cluster: one cluster of CN CTAs per group (a few wide groups: a
// batch-1 decode step of a norm with one wide group).  CTA `rank` takes
// vectors [rank * per, (rank + 1) * per) of the group, one per thread
// (per = p.cluster_vecs; CTAs x warps per CTA <= 32).  Lane r of each warp
// sends the warp's partial sum of squares to slot rank * warps + warp of CTA
// r with an asynchronous remote store (st.async) that also counts its 4 bytes
// on CTA r's mbarrier; each CTA waits on its own mbarrier for all the
// cluster's slots, then every warp adds the 32 slots with the same butterfly,
// so all CTAs get the same bits.  A CTA's shared memory receives nothing
// after its wait completes, so it may exit then.  The mbarrier is set up
// before a relaxed cluster arrive at entry, which every CTA waits on before
// its first remote store: each target is running and its mbarrier is
// initialised when the stores arrive.  The waits are bounded.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Map a shared-memory address of this CTA to the same location in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t own, uint32_t rank) {
  uint32_t m;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(m) : "r"(own), "r"(rank));
  return m;
}
// Store v at `addr` in another CTA of the cluster, counting 4 bytes on the
// mbarrier `bar` of that CTA (both addresses mapped with map_to_rank).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(
                   addr),
               "f"(v), "r"(bar)
               : "memory");
}

template <typename T, int MODE>
__global__ void __launch_bounds__(512) k_wide_cluster(const KParams p) {
  constexpr int E = Elem<T>::E;
  // slot r * nwarps + w: warp w of CTA r's partial sum (CTAs x warps <= 32)
  __shared__ float partials[32];
  __shared__ __align__(8) unsigned long long full;  // every slot has landed
  const int CN = p.cluster_ctas;  // CTAs per cluster (the launch's cluster size)
  const int tid = threadIdx.x;
  const int nwarps = blockDim.x >> 5;
  const int nslots = CN * nwarps;
  const uint32_t bar = smem_u32(&full);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_expect_tx(bar, static_cast<uint32_t>(nslots) * 4u);  // the one arrival, and the bytes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_arrive_relaxed();  // waited on before the first remote store
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t rank = cluster_ctarank();
  const int64_t item = blockIdx.x / CN;  // the group of this cluster
  const int64_t row = div_by(item, p.groups, p.div_magic);
  const int64_t g = item - row * p.groups;
  const int64_t col0 = g * p.gs;
  const int v = static_cast<int>(rank) * p.cluster_vecs + tid;  // this thread's vector
  const bool has = tid < p.cluster_vecs && v < p.nvec;
  const T* yp = static_cast<const T*>(p.y) + row * p.ys + col0;
  const T* gp = static_cast<const T*>(p.gate) + row * p.gts + col0;
  uint4 yr = make_uint4(0u, 0u, 0u, 0u), gr = make_uint4(0u, 0u, 0u, 0u);
  float wv[E];
  if (has) {
    yr = ld_stream(yp + (int64_t)v * E);
    gr = ld_stream(gp + (int64_t)v * E);
    load_weight_vec<T, MODE>(p.w, (MODE == kMamba2 ? col0 : 0) + (int64_t)v * E, wv);
  }
  float a[E];
  float c0 = 0.0f, c1 = 0.0f;
  {
    float yf[E];
    Elem<T>::unpack(yr, yf);
    if (MODE == kMamba2) {
      float gf[E];
      Elem<T>::unpack(gr, gf);
      gated_vec<T, E>(yf, gf, a);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = yf[e];
    }
    sumsq2<E>(a, c0, c1);
  }
  float ss = c0 + c1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  // every warp sends its partial to its slot in every CTA of the cluster
  // (lane r to CTA r)
  const int warp = tid >> 5, lane = tid & 31;
  cluster_wait();  // every CTA of the cluster is running, its mbarrier set up
  if (lane < CN) {
    const uint32_t r = static_cast<uint32_t>(lane);
    st_async_f32(map_to_rank(smem_u32(&partials[static_cast<int>(rank) * nwarps + warp]), r), ss,
                 map_to_rank(bar, r));
  }
  if (!mbar_wait(bar, 0)) {
    if (tid == 0) atomicOr(p.fault, kFaultClusterWait);
    return;
  }
  // a warp butterfly over the 32 slots (0 past the used ones): the same
  // operations, hence the same bits, in every warp of every CTA
  float m2 = lane < nslots ? partials[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
  const float nf = normaliser(m2, p.gs_f, p.eps);
  if (has) {
    uint4 o;
    if (MODE == kMamba2) {
      o = epilogue_mamba2<T>(a, nf, wv);
    } else {
      float gf[E], sg[E];
      Elem<T>::unpack(gr, gf);
      silu_vec<T, E>(gf, sg);
      o = epilogue_onnx<T>(a, sg, nf, wv);
    }
    st_stream(static_cast<T*>(p.out) + row * p.os + col0 + (int64_t)v * E, o);
  }
}

// ---------------------------------------------------------------------------
// Launch of the kernel a plan names, for one element type.  (The streaming
// family lives in ggrn_stream.cuh.)
// ---------------------------------------------------------------------------
template <typename T, int MODE>
cudaError_t launch_stream(const KParams& k, const Plan& p, cudaStream_t s);

template <typename K>
cudaError_t launch_kernel(K kernel, const KParams& k, const Plan& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(p.block));
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, k);
}

template <typename T, int MODE, int G>
cudaError_t launch_straddle_g(const KParams& k, const Plan& p, cudaStream_t s) {
  switch (p.vpl) {
    case 1: return launch_kernel(k_straddle<T, MODE, 1, G>, k, p, s);
    case 2: return launch_kernel(k_straddle<T, MODE, 2, G>, k, p, s);
    case 4: return launch_kernel(k_straddle<T, MODE, 4, G>, k, p, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

template <typename T, int MODE>
cudaError_t launch_straddle(const KParams& k, const Plan& p, cudaStream_t s) {
  // G = gcd(group size, E) < E
  switch (p.straddle_g) {
    case 1: return launch_straddle_g<T, MODE, 1>(k, p, s);
    case 2: return launch_straddle_g<T, MODE, 2>(k, p, s);
    case 4:
      if (Elem<T>::E > 4) return launch_straddle_g<T, MODE, (Elem<T>::E > 4 ? 4 : 2)>(k, p, s);
      break;
    default: break;
  }
  return cudaErrorInvalidConfiguration;
}

template <typename T, int MODE>
cudaError_t launch_mode(const KParams& k, const Plan& p, cudaStream_t s) {
  switch (p.path) {
    case kTeam:
      if (p.items_groups == 2) {
        switch (p.lanes * 8 + p.vpl) {   // paired items: at least 4 vectors
          case 1 * 8 + 4: return launch_kernel(k_team<T, MODE, 1, 4, 2>, k, p, s);
          case 2 * 8 + 4: return launch_kernel(k_team<T, MODE, 2, 4, 2>, k, p, s);
          case 4 * 8 + 4: return launch_kernel(k_team<T, MODE, 4, 4, 2>, k, p, s);
          case 8 * 8 + 4: return launch_kernel(k_team<T, MODE, 8, 4, 2>, k, p, s);
          case 16 * 8 + 4: return launch_kernel(k_team<T, MODE, 16, 4, 2>, k, p, s);
          case 32 * 8 + 4: return launch_kernel(k_team<T, MODE, 32, 4, 2>, k, p, s);
          default: break;
        }
        break;
      }
      switch (p.lanes * 8 + p.vpl) {   // (lanes, vectors per lane) pairs the host plans
        case 1 * 8 + 1: return launch_kernel(k_team<T, MODE, 1, 1, 1>, k, p, s);
        case 1 * 8 + 2: return launch_kernel(k_team<T, MODE, 1, 2, 1>, k, p, s);
        case 1 * 8 + 4: return launch_kernel(k_team<T, MODE, 1, 4, 1>, k, p, s);
        case 2 * 8 + 4: return launch_kernel(k_team<T, MODE, 2, 4, 1>, k, p, s);
        case 4 * 8 + 4: return launch_kernel(k_team<T, MODE, 4, 4, 1>, k, p, s);
        case 8 * 8 + 4: return launch_kernel(k_team<T, MODE, 8, 4, 1>, k, p, s);
        case 16 * 8 + 4: return launch_kernel(k_team<T, MODE, 16, 4, 1>, k, p, s);
        case 32 * 8 + 4: return launch_kernel(k_team<T, MODE, 32, 4, 1>, k, p, s);
        default: break;
      }
      break;
    case kWide:
      if (p.block <= 256) {
        if (p.vpl == 4) return launch_kernel(k_wide<T, MODE, 4, 256>, k, p, s);
        if (p.vpl == 2) return launch_kernel(k_wide<T, MODE, 2, 256>, k, p, s);
        if (p.vpl == 1) return launch_kernel(k_wide<T, MODE, 1, 256>, k, p, s);
      } else {
        if (p.vpl == 4) return launch_kernel(k_wide<T, MODE, 4, 1024>, k, p, s);
        if (p.vpl == 2) return launch_kernel(k_wide<T, MODE, 2, 1024>, k, p, s);
        if (p.vpl == 1) return launch_kernel(k_wide<T, MODE, 1, 1024>, k, p, s);
      }
      break;
    case kStraddle:
      return launch_straddle<T, MODE>(k, p, s);
    case kScalar:
      if (p.lanes == 1) return launch_kernel(k_scalar<T, MODE, 1>, k, p, s);
      if (p.lanes == 32) return launch_kernel(k_scalar<T, MODE, 32>, k, p, s);
      break;
    case kStream:
      return launch_stream<T, MODE>(k, p, s);
    case kWideCluster: {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
      cfg.blockDim = dim3(static_cast<unsigned>(p.block));
      cfg.stream = s;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = static_cast<unsigned>(p.cluster_ctas);
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      return cudaLaunchKernelEx(&cfg, k_wide_cluster<T, MODE>, k);
    }
    default:
      break;
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace ggrn
