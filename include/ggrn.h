/*
 * ggrn.h -- C ABI of the GB300 (sm_103a) fused gated group-RMSNorm library.
 *
 * The operation.  For every row n and every contiguous group g of
 * group_size columns (col = g * group_size + j, 0 <= j < group_size):
 *
 *   GGRN_MODE_MAMBA2 -- "gated_group_rmsnorm" Mojo module page, math block
 *   (norm_before_gate=False branch of the Mamba-2 mixer norm):
 *       gated = f32(y[n,col]) * silu(f32(gate[n,col]))
 *       m2    = sum_j gated^2                     (f32, over the group)
 *       nf    = rsqrt(m2 / group_size + eps)
 *       out[n,col] = cast_T( f32(w[col]) * f32(cast_T(gated * nf)) )
 *     w: float32, length width, indexed by col.  T in {f32, f16, bf16}.
 *
 *   GGRN_MODE_ONNX -- "com.microsoft.GatedRMSNorm" README, Description and
 *   Type constraints:
 *       Y = X * rsqrt(mean(X^2) + eps) * scale * SiLU(gate)
 *     mean over each contiguous group of C = group_size elements, scale of
 *     type T and length C shared by all groups and rows, every intermediate
 *     f32, only the store narrows.  T in {f32, f16} (bf16 is rejected).
 *     Leading axes of X are folded into rows (rows = numel / width).
 *
 * Memory.  Every pointer is a DEVICE pointer owned by the caller.  y, gate
 * and out are [rows, width] matrices of T with unit inner stride and the
 * given row strides in ELEMENTS (a strided view split from a fused in-proj
 * output is read in place).  The library allocates no device memory (its
 * own state is a few module-scope device words per device: the status word
 * below and the unit-claim words of the STREAM family's schedule), does not
 * synchronise, and enqueues all work on `cuda_stream` (a cudaStream_t;
 * NULL = the legacy default stream), so calls may be captured in a CUDA
 * graph (a captured STREAM launch uses the static schedule, which replays
 * unchanged).  out must not overlap y or gate.
 *
 * Errors.  Argument errors are detected on the host before anything is
 * enqueued and returned synchronously (nothing is launched).  A launch
 * failure returns GGRN_ERR_CUDA.  Faults inside a kernel surface, as usual
 * for CUDA, at the next synchronising call of the caller.
 *
 * Numerics.  f32 arithmetic and accumulation as the pages state; the group
 * sum is a tree (warp butterflies), not the sequential order, so a 16-bit
 * result may differ from a sequential-order evaluation by one ulp (two in
 * MAMBA2 when the intermediate cast flips).  Results are deterministic:
 * identical inputs give identical bits on every call.
 */
#ifndef GGRN_H
#define GGRN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GGRN_OK = 0,
  GGRN_ERR_NULL = 1,        /* a required pointer is NULL (checked only when rows > 0) */
  GGRN_ERR_SHAPE = 2,       /* rows < 0, width <= 0, group_size <= 0, width % group_size != 0,
                               a row stride < width (rows > 1), or a size that overflows int64 */
  GGRN_ERR_ALIGN = 3,       /* a forced vector path was given pointers/strides it cannot load
                               with 16-byte vectors (automatic selection never returns this:
                               it falls back to the scalar path) */
  GGRN_ERR_DTYPE = 4,       /* unknown dtype or mode, or MODE_ONNX with BF16 */
  GGRN_ERR_OVERLAP = 5,     /* the address range of out intersects that of y or gate */
  GGRN_ERR_CUDA = 6,        /* a CUDA runtime call (launch, query) failed */
  GGRN_ERR_UNSUPPORTED = 7, /* a forced path does not cover this shape */
  GGRN_ERR_ARG = 8,         /* an invalid path id, a NULL out-parameter, or a bad call list */
  GGRN_ERR_LIMIT = 9        /* ggrn_forward_noalloc: more streamed units than
                               GGRN_NOALLOC_MAX_UNITS */
} ggrn_status;

typedef enum { GGRN_F32 = 0, GGRN_F16 = 1, GGRN_BF16 = 2 } ggrn_dtype; /* T of y, gate, out */

typedef enum { GGRN_MODE_MAMBA2 = 0, GGRN_MODE_ONNX = 1 } ggrn_mode;

/* Kernel families.  AUTO lets the library choose (the normal case). */
typedef enum {
  GGRN_PATH_AUTO = 0,
  GGRN_PATH_TEAM = 1,     /* a team of 1..32 lanes of one warp per group, group held in
                             registers, segmented butterfly; several groups per warp when
                             the team is narrower than a warp (narrow and medium groups) */
  GGRN_PATH_WIDE = 2,     /* one CTA per group, group held in registers across the CTA,
                             warp partials combined through shared memory (wide groups) */
  GGRN_PATH_STRADDLE = 3, /* one warp per row chunk; 16-byte vectors that straddle group
                             boundaries; per-vector partial sums combined per group through
                             shared memory (group_size not a multiple of the vector) */
  GGRN_PATH_SCALAR = 4,   /* element loads, any alignment and any group size; the group is
                             read twice (a correctness path for layouts the vector paths
                             cannot load) */
  GGRN_PATH_STREAM = 5,   /* persistent CTAs; a producer lane streams row chunks into a
                             shared-memory ring with bulk (TMA) copies, consumer warps
                             reduce from shared memory (group bytes a multiple of 8,
                             4..128 shared-memory vectors per group, enough rows) */
  GGRN_PATH_WIDE_CLUSTER = 6 /* a cluster of 2..8 CTAs per group, one 16-byte vector per
                                thread; the CTAs' partial sums of squares are combined
                                through distributed shared memory (a few wide groups, e.g.
                                a batch-1 step of a norm with one wide group; group a
                                multiple of the vector, at most 1024 vectors) */
} ggrn_path;

/*
 * ggrn_forward -- enqueue the fused gated group-RMSNorm on `cuda_stream`.
 *   y, gate   : const T*, [rows, width], row strides y_row_stride,
 *               gate_row_stride (elements, >= width when rows > 1).
 *   w         : MAMBA2: const float* [width];  ONNX: const T* [group_size].
 *   out       : T*, [rows, width], row stride out_row_stride (elements).
 *   rows      : >= 0; rows == 0 returns GGRN_OK and launches nothing.
 *   width     : > 0, a multiple of group_size.
 *   group_size: > 0 (any value; no relation to the warp or vector width).
 *   eps       : added to the mean of squares (no default; pass it).
 *   dtype     : ggrn_dtype of y, gate, out (and scale in ONNX mode).
 *   mode      : ggrn_mode.
 * Returns a ggrn_status.
 */
int ggrn_forward(const void* y, const void* gate, const void* w, void* out, int64_t rows,
                 int64_t width, int64_t group_size, int64_t y_row_stride,
                 int64_t gate_row_stride, int64_t out_row_stride, float eps, int dtype,
                 int mode, void* cuda_stream);

/*
 * ggrn_forward_path -- ggrn_forward with the kernel family forced (tests and
 * tuning).  Same arguments plus `path` (ggrn_path).  Returns
 * GGRN_ERR_UNSUPPORTED when the family cannot compute this shape and
 * GGRN_ERR_ALIGN when it cannot load these pointers/strides.
 */
int ggrn_forward_path(const void* y, const void* gate, const void* w, void* out, int64_t rows,
                      int64_t width, int64_t group_size, int64_t y_row_stride,
                      int64_t gate_row_stride, int64_t out_row_stride, float eps, int dtype,
                      int mode, int path, void* cuda_stream);

/*
 * ggrn_forward_inproj -- ggrn_forward reading y and gate straight from the
 * packed output of a fused input projection ("gated_group_rmsnorm" page,
 * Parallelization: a y/gate view split from the fused in-proj is read as
 * it lies, with no host-side copy).
 *   inproj            : const T*, rows of inproj_row_stride elements; y is
 *                       columns [y_col, y_col + width) of every row and gate
 *                       columns [gate_col, gate_col + width); other columns
 *                       are never read.
 *   inproj_row_stride : elements between rows (>= y_col + width and
 *                       >= gate_col + width, also when rows == 1).
 *   y_col, gate_col   : >= 0, in elements (any value: an offset that breaks
 *                       16-byte alignment selects a narrower-load family).
 *   w, out, out_row_stride, rows, width, group_size, eps, dtype, mode,
 *   cuda_stream       : as in ggrn_forward.
 * Returns the ggrn_forward statuses; GGRN_ERR_SHAPE also when a column range
 * leaves the row.  out must not overlap the y or gate columns.
 */
int ggrn_forward_inproj(const void* inproj, int64_t inproj_row_stride, int64_t y_col,
                        int64_t gate_col, const void* w, void* out, int64_t out_row_stride,
                        int64_t rows, int64_t width, int64_t group_size, float eps, int dtype,
                        int mode, void* cuda_stream);

/*
 * ggrn_forward_host -- the operation on HOST-resident y, gate and out.
 * Two routes, chosen per call:
 *   - y_host, gate_host and out_host all mapped into the current device's
 *     address space at their own addresses (page-locked memory from
 *     cudaHostAlloc/cudaMallocHost, or registered with cudaHostRegister, on
 *     a system with unified addressing): one kernel on `cuda_stream` reads y
 *     and gate and writes out in place over the host link (plain loads and
 *     stores; no copies, the workspace unused and allowed to be NULL);
 *   - otherwise rows are cut into chunks that cycle through three slots of
 *     `workspace`; on three streams of the library (created on the first
 *     call on a device), the host-to-device copies of one chunk, the kernel
 *     of the previous one and the device-to-host copy of the one before run
 *     at the same time.
 * Either way ordered after the work already on `cuda_stream`; work enqueued
 * on `cuda_stream` afterwards runs after the last output row has arrived in
 * `out_host`.
 *   y_host, gate_host : const T*, host [rows, width] matrices with the given
 *                       row strides (elements).  Pageable memory gives
 *                       correct results with the copies serialised.
 *   out_host          : T*, host, row stride out_row_stride.
 *   w                 : DEVICE pointer, as in ggrn_forward.
 *   workspace         : DEVICE memory owned by the caller, 16-byte aligned,
 *                       workspace_bytes long (copy route only);
 *                       ggrn_host_workspace_bytes() gives the size that
 *                       allows full-size chunks; less shortens the chunks (at
 *                       least one row per slot: 9 x (width x sizeof(T)
 *                       rounded up to 256) bytes).
 *   other arguments   : as in ggrn_forward.
 * Returns the ggrn_forward statuses (argument checks on the host matrices,
 * before anything is enqueued); on the copy route also GGRN_ERR_NULL for a
 * NULL workspace, GGRN_ERR_ALIGN for a misaligned one, GGRN_ERR_ARG for one
 * too small.  Calls from several host threads on one device are serialised
 * while they enqueue; the workspace of a call must not be used by other work
 * until `cuda_stream` has passed the call.
 */
int ggrn_forward_host(const void* y_host, const void* gate_host, const void* w, void* out_host,
                      int64_t rows, int64_t width, int64_t group_size, int64_t y_row_stride,
                      int64_t gate_row_stride, int64_t out_row_stride, float eps, int dtype,
                      int mode, void* workspace, int64_t workspace_bytes, void* cuda_stream);

/*
 * ggrn_forward_inproj_host -- ggrn_forward_host on y and gate given as two
 * column ranges of one packed HOST matrix, the output of a fused input
 * projection ("gated_group_rmsnorm" page, Parallelization: the y/gate views
 * split from the fused in-proj).
 *   inproj_host       : const T*, host, rows of inproj_row_stride elements;
 *                       y is columns [y_col, y_col + width), gate columns
 *                       [gate_col, gate_col + width).  The caller declares
 *                       the whole of every row up to the end of the later
 *                       range part of this one matrix: the copy route may
 *                       then move y and gate of a chunk as one contiguous
 *                       copy (columns between the ranges included, and never
 *                       used), which ggrn_forward_host never does for two
 *                       separately given matrices.
 *   inproj_row_stride, y_col, gate_col : as in ggrn_forward_inproj.
 *   other arguments   : as in ggrn_forward_host.
 * Returns the ggrn_forward_host statuses; GGRN_ERR_SHAPE also when a column
 * range leaves the row.
 */
int ggrn_forward_inproj_host(const void* inproj_host, int64_t inproj_row_stride, int64_t y_col,
                             int64_t gate_col, const void* w, void* out_host,
                             int64_t out_row_stride, int64_t rows, int64_t width,
                             int64_t group_size, float eps, int dtype, int mode, void* workspace,
                             int64_t workspace_bytes, void* cuda_stream);

/*
 * ggrn_norm_outproj -- the Mamba-2 gated group-RMSNorm fused into the A
 * operand of the out_proj GEMM that follows it ("gated_group_rmsnorm" page,
 * the paragraph after the math block: the norm returns the model dtype and
 * the out_proj consumes it as it is):
 *     A[m, k] = the norm's output (MAMBA2 semantics, bf16),
 *     z[m, n] = cast_bf16( sum_k f32(A[m, k]) * f32(w_out[n, k]) )   (f32 sums)
 * A is built tile by tile in shared memory and fed to the tensor cores; it is
 * written to memory only when `a_out` is given.  Two kernels on `cuda_stream`:
 * the per-group normalisers into `workspace`, then the GEMM.
 *   y, gate       : const bf16*, DEVICE, [rows, width], row strides
 *                   y_row_stride / gate_row_stride (elements, multiples of 8).
 *   w             : const float*, DEVICE, [width] (the norm weight).
 *   w_out         : const bf16*, DEVICE, [d_model, width] row-major (the
 *                   out_proj weight as a Linear layer stores it).
 *   z             : bf16*, DEVICE, [rows, d_model] contiguous.
 *   workspace     : DEVICE, caller-owned, at least
 *                   ggrn_norm_outproj_workspace_bytes(rows, width, group_size)
 *                   bytes, 16-byte aligned (rows x groups floats).
 *   a_out         : optional bf16*, DEVICE, [rows, width] contiguous: the
 *                   normalised A as the GEMM used it (verification); NULL to
 *                   skip.
 * Shapes the kernel covers: rows a multiple of 128, width and group_size
 * multiples of 64, d_model a multiple of 32 (split into tiles of 2 x N with
 * N the largest multiple of 16 up to 256 that divides it); all pointers
 * 16-byte aligned.  Returns GGRN_OK; GGRN_ERR_SHAPE / NULL / ALIGN / OVERLAP
 * as ggrn_forward for y, gate and w, and for z, w_out, workspace and a_out;
 * GGRN_ERR_ARG for a workspace too small; GGRN_ERR_UNSUPPORTED for shapes
 * outside the above; GGRN_ERR_CUDA when a launch fails.  Allocates nothing;
 * the device status word (ggrn_fault_status) gets bit 16 if a bounded wait
 * of the GEMM ran out.
 */
int ggrn_norm_outproj(const void* y, const void* gate, const void* w, const void* w_out, void* z,
                      int64_t rows, int64_t width, int64_t group_size, int64_t y_row_stride,
                      int64_t gate_row_stride, int64_t d_model, float eps, void* workspace,
                      int64_t workspace_bytes, void* a_out, void* cuda_stream);

/* Workspace bytes ggrn_norm_outproj needs (0 for invalid shapes). */
int64_t ggrn_norm_outproj_workspace_bytes(int64_t rows, int64_t width, int64_t group_size);

/* Device workspace in bytes for which ggrn_forward_host uses full-size
 * chunks (about 32 MB of y and gate per chunk, three slots); 0 for rows <= 0
 * or width <= 0. */
int64_t ggrn_host_workspace_bytes(int64_t rows, int64_t width, int dtype);

/* What a call would launch (host only: launches nothing, dereferences no pointer). */
typedef struct {
  int32_t path;            /* ggrn_path chosen */
  int32_t team_lanes;      /* TEAM: lanes per group; WIDE/STRADDLE: threads per CTA */
  int32_t vec_per_lane;    /* 16-byte vectors (TEAM/WIDE/STRADDLE) each lane holds per tensor */
  int32_t elems_per_vec;   /* elements per 16-byte vector (16 / sizeof(T)); 1 on SCALAR */
  int64_t grid_blocks;     /* CTAs launched */
  int32_t block_threads;   /* threads per CTA */
  int32_t smem_bytes;      /* dynamic shared memory per CTA */
  int64_t items;           /* work items: groups (TEAM/WIDE/SCALAR) or row chunks (STRADDLE) */
} ggrn_plan_info;

/*
 * ggrn_plan -- fill `info` with the launch that ggrn_forward_path(..., path)
 * would make for these arguments (path = GGRN_PATH_AUTO for ggrn_forward).
 * Pointers are only inspected for alignment.  Validation is the same as in
 * ggrn_forward, except that rows == 0 still yields a plan (with 0 blocks) and
 * out may be NULL (an output not allocated yet; NULL counts as 16-byte
 * aligned).
 * The SM count used for grid sizing is the one of the current device when
 * a GPU is present, else 152.
 */
int ggrn_plan(const void* y, const void* gate, const void* w, const void* out, int64_t rows,
              int64_t width, int64_t group_size, int64_t y_row_stride,
              int64_t gate_row_stride, int64_t out_row_stride, int dtype, int mode,
              int path, ggrn_plan_info* info);

/* One call of a decode chain (the arguments of ggrn_forward without the stream). */
typedef struct {
  const void* y;
  const void* gate;
  const void* w;
  void* out;
  int64_t rows, width, group_size;
  int64_t y_row_stride, gate_row_stride, out_row_stride;
  float eps;
  int32_t dtype, mode;
} ggrn_call;

/*
 * Decode graphs -- batch-1 decode is launch-bound (one call per layer per
 * token; the work is a few thousand elements), so a chain of calls is
 * captured once into a CUDA graph and replayed with one launch.
 *
 * ggrn_graph_create: validates every call (as ggrn_forward does), captures
 *   the n calls in order on a private stream, and instantiates the graph.
 *   Buffers are baked into the graph: the caller keeps them alive and
 *   refills them in place between replays.  *graph receives an opaque
 *   handle.  Host memory is allocated for the handle and the graph; no
 *   device memory is allocated by this library.  A chain of one call is not
 *   captured: the handle keeps the call, and each launch issues it as
 *   ggrn_forward would (a graph of one small kernel costs more to launch
 *   than the kernel itself).
 * ggrn_graph_launch: one cudaGraphLaunch of the chain on `cuda_stream` (one
 *   call: that call's launch on `cuda_stream`).
 * ggrn_graph_destroy: frees the handle (NULL is a no-op).  The caller must
 *   make sure no launch of it is still running on the GPU.
 */
int ggrn_graph_create(const ggrn_call* calls, int32_t n, void** graph);
int ggrn_graph_launch(void* graph, void* cuda_stream);
int ggrn_graph_destroy(void* graph);

/* Static description of a status code (never NULL). */
const char* ggrn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ggrn_version(void);

/*
 * ggrn_fault_status -- the device status word of the current device.  The
 * STREAM kernels bound every wait on a shared-memory barrier; a wait that
 * runs out stops the kernel and sets a bit here: 1 = a consumer waited for
 * data, 2 = the producer waited for a free stage, 4 = the producer waited for
 * its copies to land, 8 = a unit claim of the dynamic schedule gave up;
 * 32 = a WIDE_CLUSTER CTA waited for its cluster's partial sums (16: see
 * ggrn_norm_outproj).
 * Nonzero means the outputs of some call are incomplete.  Synchronises the device, writes the word to *flags and, when
 * `clear` is nonzero, resets it.  Returns GGRN_OK, GGRN_ERR_ARG (flags NULL)
 * or GGRN_ERR_CUDA.
 */
int ggrn_fault_status(uint32_t* flags, int clear);

/* Name of the CUDA error behind this thread's last GGRN_ERR_CUDA from a
 * launch ("cudaSuccess" if none); a static string, never NULL. */
const char* ggrn_last_cuda_error(void);

/*
 * ggrn_selftest_wait_timeout -- exercise the STREAM family's failure path.
 * Launches the streaming kernel (MAMBA2, contiguous rows) on the given
 * buffers with its producer issuing nothing: each consumer's bounded wait
 * runs out (about a second), sets bit 1 of the status word and ends; no
 * buffer is read or written and the CUDA context stays usable.  Arguments as
 * in ggrn_forward (row strides = width, eps fixed); the buffers only have to
 * be valid for the shape.  Read the result with ggrn_fault_status.
 */
int ggrn_selftest_wait_timeout(const void* y, const void* gate, const void* w, void* out,
                               int64_t rows, int64_t width, int64_t group_size, int dtype,
                               void* cuda_stream);

/*
 * ggrn_forward_noalloc -- an addition of this library; the pages have no
 * counterpart.
 *
 * For callers that cannot allocate device memory: code that runs while a
 * framework's caching allocator owns the device (a raw cudaMalloc would fall
 * outside its budget and accounting, or fail once the cache holds the free
 * memory), real-time loops that must never block in the driver's allocator,
 * and embedders whose device memory all comes from a pool they do not
 * control.  This entry point runs the STREAM family with its dynamic unit
 * schedule and keeps the schedule's claim counter in a fixed array built
 * into the library: GGRN_NOALLOC_SCRATCH_BYTES per device, present on every
 * GPU that loads the library until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.  (ggrn_forward
 * allocates nothing either; this entry point differs in always taking the
 * STREAM family and in keeping its schedule state in an array of its own
 * that each call clears.)
 *
 * Arguments, layouts, ownership and numerics are those of ggrn_forward.
 * Every call shares the array and clears the counter on `cuda_stream`
 * before its kernel: calls of this entry point that overlap on the GPU
 * (other streams, other threads) race on it and may leave outputs
 * incomplete, so order them (one stream, or events).  The first call on a
 * device looks up the array's device address (once per device, with that
 * device current); make that first call before any stream capture.
 *
 * Returns the ggrn_forward statuses, GGRN_ERR_UNSUPPORTED when the STREAM
 * family cannot compute the shape (group bytes not a multiple of 8, or
 * outside 4..128 shared-memory vectors per group), GGRN_ERR_ALIGN when the
 * pointers or row strides are not 16-byte aligned, and GGRN_ERR_LIMIT when
 * the call would stream more than GGRN_NOALLOC_MAX_UNITS units.
 */
#define GGRN_NOALLOC_SCRATCH_BYTES 256
#define GGRN_NOALLOC_MAX_UNITS (1LL << 30)
int ggrn_forward_noalloc(const void* y, const void* gate, const void* w, void* out,
                         int64_t rows, int64_t width, int64_t group_size, int64_t y_row_stride,
                         int64_t gate_row_stride, int64_t out_row_stride, float eps, int dtype,
                         int mode, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GGRN_H */
