// ggrn_internal.h -- host-side plan and launch interface shared by the C ABI
// (ggrn_api.cu) and the per-dtype kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ggrn {

enum Mode : int { kMamba2 = 0, kOnnx = 1 };
enum Dtype : int { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum Path : int {
  kAuto = 0, kTeam = 1, kWide = 2, kStraddle = 3, kScalar = 4, kStream = 5, kWideCluster = 6
};
// STREAM with 8 teams per warp: how the teams of a warp's pass take its 8
// consecutive items (see plan_stream)
enum TeamMap : int { kTeamsInOrder = 0, kTeamsApart2 = 1, kTeamsApart4 = 2 };

// Validated arguments of one call.
struct Args {
  const void* y;
  const void* gate;
  const void* w;
  void* out;
  int64_t rows, width, gs;
  int64_t ys, gts, os;  // row strides, elements
  float eps;
  int dtype, mode;
};

// A launch decision.
struct Plan {
  int path = kAuto;
  int lanes = 0;        // TEAM/STREAM: lanes per group (1..32)
  int vpl = 0;          // vectors per lane per tensor
  int elems_per_vec = 1;
  int block = 0;        // threads per CTA
  int smem = 0;         // dynamic shared memory bytes
  int64_t grid = 0;     // CTAs
  int64_t grid_static = 0;  // STREAM: CTAs of the static schedule (graph capture)
  int64_t items = 0;    // groups, row chunks (STRADDLE) or units (STREAM)
  int64_t groups = 0;   // groups per row
  int64_t items_per_row = 0;  // TEAM: items (groups or pairs of groups) per row
  int nvec = 0;         // TEAM/WIDE: vectors per group; STRADDLE: vectors per chunk (max)
  // STRADDLE
  int64_t chunk_elems = 0;     // elements per chunk (a multiple of lcm(gs, E))
  int64_t chunks_per_row = 0;
  int chunk_groups = 0;        // groups per full chunk
  int straddle_g = 0;          // gcd(gs, E)
  uint32_t gs_magic = 0;       // floor(2^32 / gs) + 1: exact floor(x / gs) for x, gs < 2^11
  int warp_smem = 0;           // floats of shared memory per warp
  uint64_t div_magic = 0;      // floor(2^64 / items_per_row) + 1, or 0 (see div_by)
  // STREAM
  int smem_vec_bytes = 0;      // 16 or 8
  int items_groups = 1;        // groups per team item (2: pairs of odd-half-vector groups)
  int consumer_warps = 0;
  int stages = 0;
  uint32_t stage_bytes = 0;    // one tensor's chunk slot, 128-byte aligned
  uint32_t w_smem_bytes = 0;   // weight staged in shared memory (0: read from global)
  uint32_t w_area_bytes = 0;   // its shared-memory area (128-byte multiple, past-the-end slack)
  int ug = 0;                  // groups per unit
  int64_t units_per_row = 0;   // chunk units per row
  int64_t total_groups = 0;
  int unit_mode = 0;           // 0 flat (contiguous rows), 1 chunk of a row, 2 whole rows
  int rows_per_unit = 0;       // unit_mode 2
  int64_t head_units = 0;      // unit_mode 0 and 2: short units first (see KParams)
  int head_size = 0;
  int team_map = kTeamsInOrder;
  uint64_t div_magic2 = 0;     // magic for floor(group / groups_per_row)
  uint32_t groups_magic = 0;   // STREAM row units: floor(2^32 / groups) + 1, or 0 (see div_small)
  int ctas_per_sm = 0;
  // WIDE_CLUSTER: CTAs per group (the cluster) and vectors per CTA
  int cluster_ctas = 0;
  int cluster_vecs = 0;
};

// Most consumer warps of a streaming launch (the kernels' launch bounds).
// Each SM sub-partition holds a quarter of the register file, so a CTA of
// 17 warps (5 on one sub-partition) leaves 96 registers a thread, one of
// 16 or fewer leaves 128.  The 4-lane x 7-vector paired kernel is bound at
// 15 consumer warps (+ the producer: 16), where 128 registers hold it
// without spills in both modes (ONNX also keeps the gate's words).
constexpr int kStreamMaxWarps = 16;
constexpr int kStreamMaxWarps4x7 = 15;
constexpr int stream_max_warps(int mode, int vpl) {
  (void)mode;
  return vpl == 7 ? kStreamMaxWarps4x7 : kStreamMaxWarps;
}

// Kernel parameters (passed by value).
struct KParams {
  const void* y;
  const void* gate;
  const void* w;
  void* out;
  unsigned int* fault;     // device status word (bits of ggrn_fault_status)
  int64_t items;
  int64_t groups;          // groups per row
  int64_t items_per_row;   // TEAM: items per row
  int64_t width;
  int64_t gs;
  int64_t ys, gts, os;
  int64_t chunk_elems;
  int64_t chunks_per_row;
  int64_t units;
  int64_t units_per_row;
  int64_t total_groups;
  uint64_t div_magic;
  uint64_t div_magic2;
  uint32_t groups_magic;
  int nvec;
  int chunk_groups;
  int warp_smem;
  uint32_t gs_magic;
  int consumer_warps;
  int stages;
  uint32_t stage_bytes;
  uint32_t w_smem_bytes;
  uint32_t w_area_bytes;
  int ug;
  int unit_mode;
  int rows_per_unit;
  // STREAM flat and row units: head_units units of head_size first, then
  // units of the normal size (sizes in groups for flat units, rows for row
  // units)
  int64_t head_units;
  int head_size;
  int team_map;            // STREAM: TeamMap
  int64_t rows;
  int no_copies;              // STREAM self-test: the producer issues nothing
  unsigned long long* sched;  // STREAM: unit-claim word, or NULL (static schedule)
  uint32_t epoch;             // STREAM: this launch's claim epoch (nonzero)
  int cluster_ctas;            // WIDE_CLUSTER: CTAs per group
  int cluster_vecs;            // WIDE_CLUSTER: vectors per CTA
  float eps;
  float gs_f;
};

KParams make_params(const Args& a, const Plan& p);

// The ggrn_forward path for other translation units of the library: the
// arguments of one call (a single row has no row stride), their checks, and
// validation + automatic selection + launch on a stream.
Args call_args(const void* y, const void* gate, const void* w, void* out, int64_t rows,
               int64_t width, int64_t gs, int64_t ys, int64_t gts, int64_t os, float eps,
               int dtype, int mode);
int validate_call(const Args& a);
int forward_call(const Args& a, cudaStream_t s);
// One plain-load family planned for validated arguments (kTeam, kWide with
// `vpl` vectors per thread, kStraddle, kScalar): GGRN_OK, or the status that
// refuses it; and the launch of a plan on a stream.
int plan_family(const Args& a, int path, int vpl, Plan* p);
int launch_plan(const Args& a, const Plan& p, cudaStream_t s);
// Remember the CUDA error behind a GGRN_ERR_CUDA (ggrn_last_cuda_error).
void record_cuda_error(cudaError_t e);
// The current device's status word (bits of ggrn_fault_status), or NULL.
unsigned int* device_fault_word();

// Launchers, one per element type (defined in ggrn_kernels_<T>.cu).  They
// enqueue the kernel the plan names with programmatic dependent launch
// allowed, and return the CUDA error of the launch.
cudaError_t launch_f32(const KParams& k, const Plan& p, int mode, cudaStream_t s);
cudaError_t launch_f16(const KParams& k, const Plan& p, int mode, cudaStream_t s);
cudaError_t launch_bf16(const KParams& k, const Plan& p, int mode, cudaStream_t s);

}  // namespace ggrn
