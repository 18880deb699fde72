// ggrn_outproj.cu -- the gated group-RMSNorm fused into the A operand of the
// following out_proj GEMM (bf16, Mamba-2 semantics), on the 5th-generation
// tensor cores of sm_103a.
//
//   Z[m, n] = sum_k A[m, k] * W_out[n, k],
//   A[m, k] = cast_bf16(w[k] * cast_bf16(y*silu(gate) * nf[m, g(k)]))
//
// The norm's output is the out_proj's input ("gated_group_rmsnorm" page, the
// paragraph after the math block: the op returns the model dtype, so the
// out_proj that follows takes it as it is).  Here A is never written to
// memory: producer warps build each A tile in shared memory from y and gate
// while the tensor cores multiply the previous tile.
//
// Two kernels:
//   k_nf      one warp per (row, group): the normaliser nf = rsqrt(m2/gs +
//             eps) of every group (the only cross-column step), rows x
//             groups floats into a caller-owned workspace;
//   k_outproj one CTA per 128 x (2 x BNH) tile of Z, K looped in blocks of 64:
//             warp 0 moves the y, gate and W_out blocks of a stage with
//             tensor-map bulk copies (TMA); warps 2-9 turn y and gate into the
//             A block (the norm's arithmetic, rounded exactly as the norm
//             kernels round) and store it in the tensor cores' 128-byte
//             swizzled K-major layout; one thread of warp 1 issues
//             tcgen05.mma (bf16 x bf16 -> f32, M = 128, N = BNH, K = 16) into
//             two accumulators in tensor memory; after the last block warps
//             2-9 read the accumulators (tcgen05.ld), round to bf16 and store
//             Z.  Two stages of shared memory; every wait is bounded.
//
// Each CTA of a row block rebuilds the same A block.  Sharing it across a
// cluster of CTAs (each building a slice and storing it into every CTA's
// shared memory, the stage released by a multicast commit) was correct but
// slower: 4096 x 3840 x 7680 in 329 us with single CTAs, 599 with pairs, 716
// with clusters of four -- every K block then waits for the slowest CTA of
// the cluster and the remote arrivals, which two stages cannot hide.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/ggrn.h"
#include "ggrn_internal.h"
#include "ggrn_stream.cuh"

namespace ggrn {
namespace outproj {

constexpr int kBM = 128;        // rows of a tile (UMMA M)
constexpr int kBK = 64;         // K of a stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 2;
constexpr int kThreads = 320;   // warp 0 copies, warp 1 MMA, warps 2-9 A blocks / epilogue
constexpr int kProducerThreads = 256;
constexpr uint32_t kABytes = kBM * kBK * 2;             // 16 KB
constexpr uint32_t kBMaxBytes = 2 * 256 * kBK * 2;      // 64 KB (two halves of up to 256 rows)
constexpr uint32_t kYBytes = kBM * kBK * 2;             // 16 KB
constexpr uint32_t kStageBytes = kABytes + kBMaxBytes + 2 * kYBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kHalfCol = 256;                      // TMEM column of the second accumulator
// dynamic shared memory: 1 KB of alignment slack, the stages, then barriers
constexpr uint32_t kSmemBytes = 1024 + kStages * kStageBytes + 256;

// Fault bits (the library's device status word) of this kernel's waits.
constexpr uint32_t kFaultGemmWait = 16u;

struct Params {
  const float* w;      // norm weight, f32 [K]
  const float* nf;     // [M, G]
  void* z;             // bf16 [M, N]
  void* a_out;         // optional bf16 [M, K] (the A operand, for verification)
  unsigned int* fault;
  int64_t M, N, K, gs, G;
  int bnh;             // N of one accumulator (two per tile)
};

// ---------------------------------------------------------------------------
// PTX wrappers (tensor memory, tensor-core MMA, tensor-map copies).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// 16 consecutive f32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of the tensor cores for a K-major operand
// in the 128-byte swizzled layout: rows of 128 bytes (64 bf16 of K), the 16-
// byte chunk c of row r stored at chunk c ^ (r mod 8), 8-row groups 1024
// bytes apart (the stride), the tile 1024-byte aligned.  Fields: start
// address >> 4 (bits 0-13), leading offset >> 4 (16-29; unused by this
// layout, 1), stride offset >> 4 (32-45), descriptor version 1 (46-47),
// layout 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
  return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (uint64_t{1} << 16) |
         (uint64_t{1024 >> 4} << 32) | (uint64_t{1} << 46) | (uint64_t{2} << 61);
}
// Instruction descriptor of tcgen05.mma kind::f16: f32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), both K-major (15, 16 =
// 0), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// k_nf: nf[row, g] = rsqrt(sum_j gated^2 / gs + eps), one warp per group.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_nf(const __nv_bfloat16* y, const __nv_bfloat16* gate,
                                            int64_t ys, int64_t gts, int64_t rows, int64_t G,
                                            int64_t gs, float eps, float* nf) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (item >= rows * G) return;
  const int64_t row = item / G, g = item - row * G;
  const __nv_bfloat16* yp = y + row * ys + g * gs;
  const __nv_bfloat16* gp = gate + row * gts + g * gs;
  float c0 = 0.0f, c1 = 0.0f;
  for (int64_t v = lane; v < gs / 8; v += 32) {
    float yf[8], gf[8], a[8];
    Elem<__nv_bfloat16>::unpack(ld_stream(yp + 8 * v), yf);
    Elem<__nv_bfloat16>::unpack(ld_stream(gp + 8 * v), gf);
    gated_vec<__nv_bfloat16, 8>(yf, gf, a);
    sumsq2<8>(a, c0, c1);
  }
  float s = c0 + c1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) nf[item] = normaliser(s, static_cast<float>(gs), eps);
}

// ---------------------------------------------------------------------------
// k_outproj
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    k_outproj(const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_g,
              const __grid_constant__ CUtensorMap tm_b, const Params p) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned base (the swizzled tiles need it)
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_u - raw_u);
  const uint32_t bar_u = base_u + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  // barriers: full_yg[2] (y and gate landed), full_b[2] (W_out landed),
  // full_a[2] (A built; also: y and gate read), empty_b[2] (the MMAs of the
  // stage done: A and B free), acc_full; then the TMEM address slot and the
  // abort flag
  auto full_yg = [&](int s) { return bar_u + 8u * s; };
  auto full_b = [&](int s) { return bar_u + 8u * (2 + s); };
  auto full_a = [&](int s) { return bar_u + 8u * (4 + s); };
  auto empty_b = [&](int s) { return bar_u + 8u * (6 + s); };
  const uint32_t acc_full = bar_u + 8u * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  auto sA = [&](int s) { return base_u + s * kStageBytes; };
  auto sB = [&](int s) { return base_u + s * kStageBytes + kABytes; };
  auto sY = [&](int s) { return base_u + s * kStageBytes + kABytes + kBMaxBytes; };
  auto sG = [&](int s) { return base_u + s * kStageBytes + kABytes + kBMaxBytes + kYBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bnh = p.bnh;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 2 * bnh;
  const int KB = static_cast<int>(p.K / kBK);
  const uint32_t b_half_bytes = static_cast<uint32_t>(bnh) * kBK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_yg(s), 1);
      mbar_init(full_b(s), 1);
      mbar_init(full_a(s), kProducerThreads);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // nothing global is read before the previous kernel (the nf pass) is done
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---- copies: lane 0 y and gate (refilled once the A block is built
    // from them), lane 1 the two W_out halves (refilled once the stage's
    // MMAs are done) ----
    if (lane < 2) {
      const bool yg = lane == 0;
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kStages;
        const uint32_t prev = static_cast<uint32_t>(kb / kStages - 1) & 1u;
        if (kb >= kStages && !mbar_wait(yg ? full_a(s) : empty_b(s), prev)) {
          *abort_flag = 1;
          atomicOr(p.fault, kFaultGemmWait);
          break;
        }
        if (*abort_flag) break;
        const int k0 = kb * kBK;
        if (yg) {
          mbar_expect_tx(full_yg(s), 2 * kYBytes);
          tma_load_2d(sY(s), &tm_y, k0, static_cast<int>(m0), full_yg(s));
          tma_load_2d(sG(s), &tm_g, k0, static_cast<int>(m0), full_yg(s));
        } else {
          mbar_expect_tx(full_b(s), 2 * b_half_bytes);
          tma_load_2d(sB(s), &tm_b, k0, static_cast<int>(n0), full_b(s));
          tma_load_2d(sB(s) + b_half_bytes, &tm_b, k0, static_cast<int>(n0 + bnh), full_b(s));
        }
        issued = kb + 1;
      }
      // every issued copy lands before the CTA can leave
      for (int kb = issued - kStages < 0 ? 0 : issued - kStages; kb < issued; ++kb)
        if (!mbar_wait(yg ? full_yg(kb % kStages) : full_b(kb % kStages),
                       static_cast<uint32_t>(kb / kStages) & 1u))
          atomicOr(p.fault, kFaultGemmWait);
    }
  } else if (warp == 1) {
    // ---- MMA issue (one thread) ----
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, bnh);
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
        if (*abort_flag || !mbar_wait(full_a(s), ph) || !mbar_wait(full_b(s), ph)) {
          *abort_flag = 1;
          atomicOr(p.fault, kFaultGemmWait);
          break;
        }
        tc_fence_after();
        const uint64_t a_desc = desc_sw128(sA(s));
        const uint64_t b_desc0 = desc_sw128(sB(s));
        const uint64_t b_desc1 = desc_sw128(sB(s) + b_half_bytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // the next 16 columns of K: 32 bytes further in every swizzled row
          const uint64_t adv = static_cast<uint64_t>(kk * 32 >> 4);
          mma_bf16(tmem, a_desc + adv, b_desc0 + adv, idesc, kb > 0 || kk > 0);
          mma_bf16(tmem + kHalfCol, a_desc + adv, b_desc1 + adv, idesc, kb > 0 || kk > 0);
        }
        mma_commit(empty_b(s));  // frees A and B of the stage once these MMAs have read them
      }
      mma_commit(acc_full);  // the accumulators are complete (or abandoned)
      // wait for it here too, so that no MMA still runs when TMEM is freed
      if (!mbar_wait(acc_full, 0)) atomicOr(p.fault, kFaultGemmWait);
    }
  } else {
    // ---- A blocks: warps 2-9 ----
    const int t = threadIdx.x - 64;       // 0..255
    const int rq = t >> 3;                // row within a group of 32 rows
    const int c = t & 7;                  // 16-byte chunk (8 columns) of the 64
    const float* w = p.w;
    // the weight columns and normalisers of the next block are fetched one
    // block ahead (their global-memory latency then overlaps this block)
    float4 w_lo = __ldg(reinterpret_cast<const float4*>(w + 8 * c));
    float4 w_hi = __ldg(reinterpret_cast<const float4*>(w + 8 * c + 4));
    float nfv[kBM / 32];
#pragma unroll
    for (int i = 0; i < kBM / 32; ++i) nfv[i] = __ldg(p.nf + (m0 + rq + 32 * i) * p.G);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
      // y and gate of this block landed; A[s] free (the MMAs of kb - 2 done)
      if (*abort_flag || !mbar_wait(full_yg(s), ph) ||
          (kb >= kStages && !mbar_wait(empty_b(s), ph ^ 1u))) {
        *abort_flag = 1;
        if (lane == 0) atomicOr(p.fault, kFaultGemmWait);
        break;
      }
      const int64_t k0 = static_cast<int64_t>(kb) * kBK;
      const float wv[8] = {w_lo.x, w_lo.y, w_lo.z, w_lo.w, w_hi.x, w_hi.y, w_hi.z, w_hi.w};
      float nfc[kBM / 32];
#pragma unroll
      for (int i = 0; i < kBM / 32; ++i) nfc[i] = nfv[i];
      if (kb + 1 < KB) {
        const int64_t k1 = k0 + kBK;
        const int64_t g1 = k1 / p.gs;  // a K block never crosses a group (gs % 64 == 0)
        w_lo = __ldg(reinterpret_cast<const float4*>(w + k1 + 8 * c));
        w_hi = __ldg(reinterpret_cast<const float4*>(w + k1 + 8 * c + 4));
#pragma unroll
        for (int i = 0; i < kBM / 32; ++i) nfv[i] = __ldg(p.nf + (m0 + rq + 32 * i) * p.G + g1);
      }
#pragma unroll
      for (int i = 0; i < kBM / 32; ++i) {
        const int r = rq + 32 * i;
        const float nf = nfc[i];
        uint4 yv, gv;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(yv.x), "=r"(yv.y), "=r"(yv.z), "=r"(yv.w)
                     : "r"(sY(s) + r * 128 + c * 16));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(gv.x), "=r"(gv.y), "=r"(gv.z), "=r"(gv.w)
                     : "r"(sG(s) + r * 128 + c * 16));
        float yf[8], gf[8], a[8], o[8];
        Elem<__nv_bfloat16>::unpack(yv, yf);
        Elem<__nv_bfloat16>::unpack(gv, gf);
        gated_vec<__nv_bfloat16, 8>(yf, gf, a);
        mamba2_out<__nv_bfloat16, 8>(a, nf, nf, wv, o);
        const uint4 av = Elem<__nv_bfloat16>::pack(o);
        // the 128-byte swizzle: chunk c of row r at chunk c ^ (r mod 8)
        const uint32_t dst = sA(s) + r * 128 + ((c ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(av.x), "r"(av.y),
                     "r"(av.z), "r"(av.w)
                     : "memory");
        if (p.a_out && blockIdx.x == 0)
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.a_out) + (m0 + r) * p.K + k0 +
                                    8 * c) = av;
      }
      fence_async_smem();  // the tensor cores read the block through the async proxy
      mbar_arrive(full_a(s));
    }
    // ---- epilogue: accumulators -> bf16 Z ----
    const bool ok = mbar_wait(acc_full, 0) && !*abort_flag;
    tc_fence_after();
    if (ok) {
      const int q = warp & 3;                 // the lanes (rows) this warp may read
      const int half = (warp - 2) >> 2;       // which accumulator
      const int row = 32 * q + lane;
      __nv_bfloat16* zrow = static_cast<__nv_bfloat16*>(p.z) + (m0 + row) * p.N + n0 +
                            static_cast<int64_t>(half) * bnh;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * kHalfCol;
      for (int c0 = 0; c0 < bnh; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tbase + c0, r);
        uint4 lo, hi;
        lo.x = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[0]), __uint_as_float(r[1]));
        lo.y = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[2]), __uint_as_float(r[3]));
        lo.z = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[4]), __uint_as_float(r[5]));
        lo.w = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[6]), __uint_as_float(r[7]));
        hi.x = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[8]), __uint_as_float(r[9]));
        hi.y = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[10]), __uint_as_float(r[11]));
        hi.z = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[12]), __uint_as_float(r[13]));
        hi.w = Elem<__nv_bfloat16>::pack2(__uint_as_float(r[14]), __uint_as_float(r[15]));
        st_stream(zrow + c0, lo);
        st_stream(zrow + c0 + 8, hi);
      }
    } else if (lane == 0) {
      atomicOr(p.fault, kFaultGemmWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// A 2-D bf16 tensor map: `cols` x `rows` at row stride `stride` elements, box
// of box_cols x box_rows, with or without the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, int64_t stride,
              uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride) * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// N of one accumulator: the largest UMMA N (multiple of 16, at most 256)
// whose pair divides d_model.
int pick_bnh(int64_t n) {
  for (int b = 256; b >= 16; b -= 16)
    if (n % (2 * b) == 0) return b;
  return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap_bytes(const void* a, int64_t na, const void* b, int64_t nb) {
  if (na <= 0 || nb <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

}  // namespace outproj
}  // namespace ggrn

using namespace ggrn;

extern "C" int64_t ggrn_norm_outproj_workspace_bytes(int64_t rows, int64_t width,
                                                     int64_t group_size) {
  if (rows <= 0 || width <= 0 || group_size <= 0 || width % group_size != 0) return 0;
  return (rows * (width / group_size) * 4 + 255) / 256 * 256;
}

extern "C" int ggrn_norm_outproj(const void* y, const void* gate, const void* w,
                                 const void* w_out, void* z, int64_t rows, int64_t width,
                                 int64_t group_size, int64_t y_row_stride,
                                 int64_t gate_row_stride, int64_t d_model, float eps,
                                 void* workspace, int64_t workspace_bytes, void* a_out,
                                 void* cuda_stream) {
  using namespace ggrn::outproj;
  // the norm's own checks on y, gate and w (out is checked as [rows, width]:
  // a_out when given, else a stand-in that cannot overlap anything)
  const Args a = call_args(y, gate, w, a_out ? a_out : const_cast<void*>(w_out), rows, width,
                           group_size, y_row_stride, gate_row_stride, width, eps, kBF16, kMamba2);
  if (rows < 0 || width <= 0 || group_size <= 0 || width % group_size != 0) return GGRN_ERR_SHAPE;
  if (rows == 0) return GGRN_OK;
  if (!w_out || !z || !workspace) return GGRN_ERR_NULL;
  int st = a_out ? validate_call(a) : GGRN_OK;
  if (st != GGRN_OK) return st;
  if (!a_out) {
    // y, gate, w as the norm checks them (with z standing in for out only
    // for its NULL and alignment checks)
    Args b = a;
    b.out = z;
    st = validate_call(b);
    if (st != GGRN_OK && st != GGRN_ERR_OVERLAP) return st;
  }
  if (d_model <= 0) return GGRN_ERR_SHAPE;
  if (rows % kBM != 0 || width % kBK != 0 || group_size % kBK != 0 || pick_bnh(d_model) == 0 ||
      rows > INT32_MAX || width > INT32_MAX || d_model > INT32_MAX)
    return GGRN_ERR_UNSUPPORTED;
  if (!aligned16(y) || !aligned16(gate) || !aligned16(w) || !aligned16(w_out) || !aligned16(z) ||
      (a_out && !aligned16(a_out)) || !aligned16(workspace) ||
      (rows > 1 && ((y_row_stride * 2) % 16 != 0 || (gate_row_stride * 2) % 16 != 0)))
    return GGRN_ERR_ALIGN;
  if (workspace_bytes < ggrn_norm_outproj_workspace_bytes(rows, width, group_size))
    return GGRN_ERR_ARG;
  {
    // z [rows, d_model] and the nf workspace must not overlap any input
    const int64_t ysx = rows > 1 ? y_row_stride : width;
    const int64_t gsx = rows > 1 ? gate_row_stride : width;
    const int64_t zb = rows * d_model * 2, wsb = workspace_bytes;
    const int64_t yb = ((rows - 1) * ysx + width) * 2, gb = ((rows - 1) * gsx + width) * 2;
    const int64_t wb = width * 4, wob = d_model * width * 2;
    struct R { const void* p; int64_t n; };
    const R outs[2] = {{z, zb}, {workspace, wsb}};
    const R ins[4] = {{y, yb}, {gate, gb}, {w, wb}, {w_out, wob}};
    for (const R& o : outs)
      for (const R& i : ins)
        if (ranges_overlap_bytes(o.p, o.n, i.p, i.n)) return GGRN_ERR_OVERLAP;
    if (ranges_overlap_bytes(z, zb, workspace, wsb)) return GGRN_ERR_OVERLAP;
    if (a_out && (ranges_overlap_bytes(a_out, rows * width * 2, z, zb) ||
                  ranges_overlap_bytes(a_out, rows * width * 2, workspace, wsb)))
      return GGRN_ERR_OVERLAP;
  }
  const int64_t ys = rows > 1 ? y_row_stride : width, gts = rows > 1 ? gate_row_stride : width;
  const int bnh = pick_bnh(d_model);
  const int64_t G = width / group_size;
  unsigned int* fault = device_fault_word();
  if (!fault) return GGRN_ERR_CUDA;
  CUtensorMap tm_y, tm_g, tm_b;
  if (!make_map(&tm_y, y, width, rows, ys, kBK, kBM, false) ||
      !make_map(&tm_g, gate, width, rows, gts, kBK, kBM, false) ||
      !make_map(&tm_b, w_out, width, d_model, width, kBK, static_cast<uint32_t>(bnh), true))
    return GGRN_ERR_UNSUPPORTED;
  const cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  float* nf = static_cast<float*>(workspace);

  // the normalisers
  {
    cudaLaunchConfig_t cfg = {};
    const int64_t items = rows * G;
    cfg.gridDim = dim3(static_cast<unsigned>((items * 32 + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_nf, static_cast<const __nv_bfloat16*>(y),
                                       static_cast<const __nv_bfloat16*>(gate), ys, gts, rows, G,
                                       group_size, eps, nf);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return GGRN_ERR_CUDA;
    }
  }
  // the GEMM
  {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
      attr_err = cudaFuncSetAttribute(k_outproj, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemBytes));
    });
    if (attr_err != cudaSuccess) {
      record_cuda_error(attr_err);
      return GGRN_ERR_CUDA;
    }
    Params p;
    p.w = static_cast<const float*>(w);
    p.nf = nf;
    p.z = z;
    p.a_out = a_out;
    p.fault = fault;
    p.M = rows;
    p.N = d_model;
    p.K = width;
    p.gs = group_size;
    p.G = G;
    p.bnh = bnh;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d_model / (2 * bnh)), static_cast<unsigned>(rows / kBM));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_outproj, tm_y, tm_g, tm_b, p);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return GGRN_ERR_CUDA;
    }
  }
  return GGRN_OK;
}
