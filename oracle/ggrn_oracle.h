/*
 * ggrn_oracle.h -- plain single-threaded CPU oracle of the fused gated
 * group-RMSNorm.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this library: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, helper or
 * constant with the CUDA library; the enum values below are restated here on
 * purpose because both sides implement the same argument contract.
 *
 * What it computes (one row n, one group g of group_size contiguous columns,
 * col = g * group_size + j):
 *
 *   mode MAMBA2  -- "gated_group_rmsnorm" Mojo module page, math block:
 *       gated = f32(y) * silu(f32(gate))                         (f32)
 *       m2    = sum_j gated^2                                    (f32, over the group)
 *       nf    = rsqrt(m2 / group_size + eps)
 *       out   = cast_T( f32(w[col]) * f32(cast_T(gated * nf)) )  w is f32, length width
 *
 *   mode ONNX    -- "com.microsoft.GatedRMSNorm" README, Description:
 *       Y = X * rsqrt(mean(X^2) + eps) * scale * SiLU(gate)
 *       with the mean over each contiguous group of C = group_size elements,
 *       scale of type T and length C (shared by every group of every row),
 *       every intermediate in f32 and only the store narrowed.
 *
 * Precision follows the pages: f32 arithmetic, f32 accumulation, and RNE
 * casts to T.  Summation is sequential in j.  rsqrt is taken correctly
 * rounded (through double) since the Mojo page only says it matches a
 * framework rms_norm.  A second entry point evaluates the same definition in
 * double precision, keeping only the roundings to T (the brute-force twin).
 */
#ifndef GGRN_ORACLE_H
#define GGRN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (same numbering as the product's C ABI). */
enum {
  GGRN_ORACLE_OK = 0,
  GGRN_ORACLE_ERR_NULL = 1,   /* a required pointer is NULL (only when rows > 0) */
  GGRN_ORACLE_ERR_SHAPE = 2,  /* rows < 0, width <= 0, group_size <= 0,
                                 width % group_size != 0, or a row stride < width */
  GGRN_ORACLE_ERR_DTYPE = 4   /* unknown dtype/mode, or ONNX with bf16 */
};

/* Element type T of y, gate and out (and of scale in ONNX mode). */
enum { GGRN_ORACLE_F32 = 0, GGRN_ORACLE_F16 = 1, GGRN_ORACLE_BF16 = 2 };

/* Semantics. */
enum { GGRN_ORACLE_MODE_MAMBA2 = 0, GGRN_ORACLE_MODE_ONNX = 1 };

/*
 * Forward pass over host buffers, f32 arithmetic as the pages state it.
 *   y, gate : T, [rows, width], row strides y_row_stride / gate_row_stride
 *             (elements), unit inner stride.
 *   w       : MAMBA2 -> float[width] indexed by col;
 *             ONNX   -> T[group_size] indexed by j.
 *   out     : T, [rows, width], row stride out_row_stride (elements).
 *   t_out   : optional (may be NULL).  MAMBA2 only: receives the intermediate
 *             cast_T(gated * nf), contiguous [rows, width] of T.
 * rows == 0 is a no-op returning OK.
 */
int ggrn_oracle_forward(const void* y, const void* gate, const void* w, void* out,
                        int64_t rows, int64_t width, int64_t group_size,
                        int64_t y_row_stride, int64_t gate_row_stride,
                        int64_t out_row_stride, float eps, int dtype, int mode);

int ggrn_oracle_forward_ex(const void* y, const void* gate, const void* w, void* out,
                           void* t_out, int64_t rows, int64_t width,
                           int64_t group_size, int64_t y_row_stride,
                           int64_t gate_row_stride, int64_t out_row_stride,
                           float eps, int dtype, int mode);

/* As ggrn_oracle_forward_ex, and pre_out (optional, contiguous [rows, width]
 * f32) receives each element's value just before its rounding to T: MAMBA2
 * the product gated * nf that the intermediate cast rounds, ONNX the product
 * that the store rounds.  The comparison rules of the tests use it to tell
 * whether a one-ulp difference of the intermediate (a "flip" caused by a
 * different summation order) can explain a difference of the output. */
int ggrn_oracle_forward_pre(const void* y, const void* gate, const void* w, void* out,
                            void* t_out, float* pre_out, int64_t rows, int64_t width,
                            int64_t group_size, int64_t y_row_stride,
                            int64_t gate_row_stride, int64_t out_row_stride,
                            float eps, int dtype, int mode);

/* Same definition evaluated in double; only the casts to T round
 * (directly from double, RNE).  For tiny inputs. */
int ggrn_oracle_forward_f64(const void* y, const void* gate, const void* w, void* out,
                            int64_t rows, int64_t width, int64_t group_size,
                            int64_t y_row_stride, int64_t gate_row_stride,
                            int64_t out_row_stride, float eps, int dtype, int mode);

/* The oracle's own T <-> f32 codecs (RNE, quiet NaN kept, overflow -> inf,
 * fp16 subnormals), exposed so tests can pin them to a library conversion. */
void ggrn_oracle_encode(const float* in, void* out, int64_t n, int dtype);
void ggrn_oracle_decode(const void* in, float* out, int64_t n, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* GGRN_ORACLE_H */
