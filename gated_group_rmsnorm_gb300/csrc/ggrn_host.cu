// ggrn_host.cu -- ggrn_forward_host: the operation on host-resident y, gate
// and out, with the host<->device copies overlapped with the kernels.
//
// Rows are cut into chunks that cycle through kSlots slots of a caller-owned
// device workspace (y, gate and out of one chunk per slot).  Three streams of
// the library run, for consecutive chunks at the same time, the host-to-
// device copies of chunk i, the kernel of chunk i-1 and the device-to-host
// copy of chunk i-2; events order each chunk's three steps and keep a slot
// from being refilled before its output has left.  With pinned host memory
// the two copy directions share the link at once, so a call takes about the
// time of its bytes at the combined host-device rate instead of the sum of
// both directions' times.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/ggrn.h"
#include "ggrn_internal.h"

namespace ggrn {
namespace {

constexpr int kSlots = 3;
// y + gate bytes per chunk aimed at.  Each copy carries a fixed cost, so
// larger chunks pay less of it, while fewer chunks overlap less at the ends:
// a sweep of 2-128 MB over the four prefill workloads measured 32 MB best or
// within 1 % of best on each (8 MB: 9-16 % slower; some larger sizes dipped
// on one workload or another).  Three slots measured as good as four or six.
constexpr int64_t kChunkTargetBytes = int64_t{32} << 20;
constexpr int64_t kAlign = 256;

int64_t align_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int es_of(int dtype) { return dtype == kF32 ? 4 : 2; }

int64_t target_chunk_rows(int64_t rows, int64_t width, int es) {
  const int64_t r = std::max<int64_t>(1, kChunkTargetBytes / (2 * width * es));
  return std::min(rows, r);
}

// Row counts of the chunks, at most `t` each.  When there are enough rows,
// the first kRampLevels chunks grow geometrically to `t` (t/2^R, ..., t/2)
// and the last ones mirror them, so the copies of the two directions overlap
// sooner and longer (+1-2 % end to end against equal chunks at R = 2; deeper
// ramps pay more per-copy fixed cost than they save: prefill 247.4 GB/s at
// R = 2, 243 at R = 3-4, 240.7 at R = 5); the middle rows split evenly.
constexpr int kRampLevels = 2;
int64_t chunk_rows_at(int64_t rows, int64_t t, int64_t c, int64_t* n_chunks) {
  const int R = kRampLevels;
  int64_t ramp[8], sum = 0;
  for (int i = 0; i < R; ++i) {
    ramp[i] = std::max<int64_t>(1, t >> (R - i));
    sum += ramp[i];
  }
  if (rows <= 2 * sum + t) {  // equal chunks
    *n_chunks = (rows + t - 1) / t;
    return std::min(t, rows - c * t);
  }
  const int64_t mid = rows - 2 * sum;
  const int64_t k = (mid + t - 1) / t;  // middle chunks
  const int64_t m = (mid + k - 1) / k;
  *n_chunks = k + 2 * R;
  if (c < R) return ramp[c];
  if (c >= k + R) return ramp[k + 2 * R - 1 - c];
  return std::min(m, mid - (c - R) * m);
}

// Host memory the current device addresses in place: pinned and mapped into
// the device's address space at the same address (page-locked memory from
// cudaHostAlloc/cudaMallocHost under unified addressing).  Kernels then read
// and write it over the host link directly; anything else (pageable memory,
// or a mapping at another address) goes through the copy pipeline.
bool device_maps_in_place(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory may report an error on some runtimes
    return false;
  }
  return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

// Kernels that read y and gate and write out in host memory mapped into the
// device's address space (pinned host memory reached over the host link):
// plain loads and stores only, never STREAM's bulk copies, and the family
// that measured fastest over the link.  Pinned host buffers, GB/s (WIDE /
// TEAM / STRADDLE): prefill 960-wide groups 284 / 278 / -; 5120-wide groups
// 289 / - / -; 128-wide fp16 heads 304 / 267 / -; the odd span's 100-wide
// groups read in place from the packed buffer - / 223 / 284.  WIDE with one
// vector per thread (more requests in flight per group) did better still:
// prefill 296 (4 vectors: 282), 5120-wide 302 (289), heads 303 (303).
int forward_in_place(const Args& a, cudaStream_t s) {
  const int64_t nvec = a.gs / (16 / es_of(a.dtype));
  int vpl = 1;
  while (vpl < 4 && (nvec + vpl - 1) / vpl > 1024) vpl *= 2;
  Plan p;
  int st = GGRN_ERR_UNSUPPORTED;
  for (const int path : {kWide, kStraddle, kTeam, kScalar}) {
    st = plan_family(a, path, vpl, &p);
    if (st == GGRN_OK) break;
  }
  if (st != GGRN_OK) return st;
  return launch_plan(a, p, s);
}

// Both ends of a [rows, width] matrix of es-byte elements at row stride
// `stride` elements (a matrix that runs past its page-locked allocation
// takes the copy route).
bool matrix_maps_in_place(const void* p, int64_t rows, int64_t width, int64_t stride, int es) {
  const char* first = static_cast<const char*>(p);
  const char* last = first + ((rows - 1) * stride + width) * es - 1;
  return device_maps_in_place(first) && device_maps_in_place(last);
}

// Streams and events of one device, created once (the first call there) and
// shared by all calls on that device; `mu` keeps one call's enqueue
// sequence whole when several host threads call at once.
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kSlots] = {}, done[kSlots] = {}, freed[kSlots] = {};
};

HostPipe* pipe_for_device(int dev) {
  static HostPipe pipes[64];
  return (dev >= 0 && dev < 64) ? &pipes[dev] : nullptr;
}

cudaError_t pipe_init(HostPipe* hp) {
  if (hp->ready) return cudaSuccess;
  cudaError_t e;
  for (cudaStream_t* st : {&hp->h2d, &hp->comp, &hp->d2h})
    if ((e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking)) != cudaSuccess) return e;
  cudaEvent_t* evs[] = {&hp->start, &hp->end};
  for (cudaEvent_t* ev : evs)
    if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  for (int i = 0; i < kSlots; ++i)
    for (cudaEvent_t* ev : {&hp->in[i], &hp->done[i], &hp->freed[i]})
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  hp->ready = true;
  return cudaSuccess;
}

// Copy `n` rows of `width` elements between a strided host matrix and a
// contiguous device block (one 1-D copy when the host rows are contiguous;
// strided rows go as one 2-D copy, which measured as fast most of the time
// but at half speed in some runs, hence the joint copy below).
cudaError_t copy_rows(void* dst, int64_t dst_pitch, const void* src, int64_t src_pitch,
                      int64_t row_bytes, int64_t n, cudaMemcpyKind kind, cudaStream_t s) {
  if (dst_pitch == row_bytes && src_pitch == row_bytes)
    return cudaMemcpyAsync(dst, src, static_cast<size_t>(n * row_bytes), kind, s);
  return cudaMemcpy2DAsync(dst, static_cast<size_t>(dst_pitch), src, static_cast<size_t>(src_pitch),
                           static_cast<size_t>(row_bytes), static_cast<size_t>(n), kind, s);
}

}  // namespace
}  // namespace ggrn

using namespace ggrn;

extern "C" int64_t ggrn_host_workspace_bytes(int64_t rows, int64_t width, int dtype) {
  if (rows <= 0 || width <= 0) return 0;
  const int es = es_of(dtype);
  return kSlots * 3 * align_up(target_chunk_rows(rows, width, es) * width * es);
}

namespace ggrn {
namespace {

// The host entry points' common body.  `packed`: the caller declared y and
// gate to be two column ranges of one packed host matrix (the fused in-proj
// layout), so the bytes between and around the two ranges of each row, up
// to the end of the later range, belong to that matrix and may be copied.
int forward_host_impl(const Args& a, bool packed, void* workspace, int64_t workspace_bytes,
                      cudaStream_t caller) {
  const void* y_host = a.y;
  const void* gate_host = a.gate;
  const void* w = a.w;
  void* out_host = a.out;
  const int64_t rows = a.rows, width = a.width, group_size = a.gs;
  const float eps = a.eps;
  const int dtype = a.dtype, mode = a.mode;
  int st = validate_call(a);
  if (st != GGRN_OK || rows == 0) return st;
  // Pinned, mapped host buffers: one kernel on the caller's stream reads y
  // and gate and writes out in place over the host link, which measured
  // faster than staging through the workspace with copies (prefill 284
  // against 247 GB/s end to end; the copies' pipeline peaks near 282 GB/s
  // with both directions busy).  The workspace is then unused (may be NULL).
  const int es = es_of(dtype);
  if (matrix_maps_in_place(y_host, rows, width, a.ys, es) &&
      matrix_maps_in_place(gate_host, rows, width, a.gts, es) &&
      matrix_maps_in_place(out_host, rows, width, a.os, es))
    return forward_in_place(a, caller);
  if (!workspace) return GGRN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return GGRN_ERR_ALIGN;
  const int64_t row_bytes = width * es;
  // rows per chunk: the target, as far as kSlots x (y, gate, out) slots of
  // 256-byte-aligned parts fit
  int64_t chunk = std::min(target_chunk_rows(rows, width, es),
                           workspace_bytes / (kSlots * 3 * row_bytes));
  while (chunk > 0 && kSlots * 3 * align_up(chunk * row_bytes) > workspace_bytes) --chunk;
  if (chunk < 1) return GGRN_ERR_ARG;
  const int64_t part = align_up(chunk * row_bytes);  // one tensor of one slot
  // y and gate declared as two column ranges of one packed host matrix (a
  // fused in-proj output) that cover at least 90 % of its rows: one
  // contiguous copy per chunk, from the first used byte of its first row to
  // the last used byte of its last row, into the slot's y and gate parts
  // together; the kernel then reads the two ranges in place.  Two separate
  // matrices are never copied that way: the bytes between them need not be
  // anyone's memory.
  const char* yb = static_cast<const char*>(y_host);
  const char* gb = static_cast<const char*>(gate_host);
  const int64_t pitch = a.ys * es;
  const char* lo = std::min(yb, gb);
  const int64_t span = (std::max(yb, gb) - lo) + row_bytes;  // used bytes of a row
  bool joint = packed && rows > 1 && a.ys == a.gts && span <= pitch &&
               10 * 2 * row_bytes >= 9 * pitch;
  if (joint) {
    chunk = std::min(chunk, (2 * part - span) / pitch + 1);  // (n - 1) * pitch + span <= 2 * part
    joint = chunk >= 1;
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  HostPipe* hp = e == cudaSuccess ? pipe_for_device(dev) : nullptr;
  if (!hp) {
    record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return GGRN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(hp->mu);
  if ((e = pipe_init(hp)) != cudaSuccess) {
    record_cuda_error(e);
    return GGRN_ERR_CUDA;
  }
  // everything enqueued so far on the caller's stream comes first
  e = cudaEventRecord(hp->start, caller);
  for (cudaStream_t s : {hp->h2d, hp->comp, hp->d2h})
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->start, 0);
  const char* yh = static_cast<const char*>(y_host);
  const char* gh = static_cast<const char*>(gate_host);
  char* oh = static_cast<char*>(out_host);
  char* ws = static_cast<char*>(workspace);
  const int64_t ysb = a.ys * es, gsb = a.gts * es, osb = a.os * es;
  int64_t n_chunks = 1;
  chunk_rows_at(rows, chunk, 0, &n_chunks);
  for (int64_t c = 0, r0 = 0, n = 0; c < n_chunks && e == cudaSuccess && st == GGRN_OK;
       ++c, r0 += n) {
    n = chunk_rows_at(rows, chunk, c, &n_chunks);
    const int slot = static_cast<int>(c % kSlots);
    char* dy = ws + slot * 3 * part;
    char* dg = dy + part;
    char* dout = dg + part;
    // host -> device, once the slot's previous output has left
    e = cudaStreamWaitEvent(hp->h2d, hp->freed[slot], 0);
    const void *ky = dy, *kg = dg;  // the kernel's y and gate
    int64_t kstride = width;
    if (joint) {
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(dy, lo + r0 * pitch, static_cast<size_t>((n - 1) * pitch + span),
                            cudaMemcpyHostToDevice, hp->h2d);
      ky = dy + (yb - lo);
      kg = dy + (gb - lo);
      kstride = a.ys;
    } else {
      if (e == cudaSuccess)
        e = copy_rows(dy, row_bytes, yh + r0 * ysb, ysb, row_bytes, n, cudaMemcpyHostToDevice,
                      hp->h2d);
      if (e == cudaSuccess)
        e = copy_rows(dg, row_bytes, gh + r0 * gsb, gsb, row_bytes, n, cudaMemcpyHostToDevice,
                      hp->h2d);
    }
    if (e == cudaSuccess) e = cudaEventRecord(hp->in[slot], hp->h2d);
    // the kernel on the chunk
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->in[slot], 0);
    if (e == cudaSuccess) {
      st = forward_call(call_args(ky, kg, w, dout, n, width, group_size, kstride, kstride, width,
                                  eps, dtype, mode),
                        hp->comp);
      if (st == GGRN_OK) e = cudaEventRecord(hp->done[slot], hp->comp);
    }
    // device -> host
    if (e == cudaSuccess && st == GGRN_OK) e = cudaStreamWaitEvent(hp->d2h, hp->done[slot], 0);
    if (e == cudaSuccess && st == GGRN_OK)
      e = copy_rows(oh + r0 * osb, osb, dout, row_bytes, row_bytes, n, cudaMemcpyDeviceToHost,
                    hp->d2h);
    if (e == cudaSuccess && st == GGRN_OK) e = cudaEventRecord(hp->freed[slot], hp->d2h);
  }
  // the caller's stream continues after the last output has arrived (the
  // last copy follows every kernel and every input copy of the call)
  if (e == cudaSuccess && st == GGRN_OK) e = cudaEventRecord(hp->end, hp->d2h);
  if (e == cudaSuccess && st == GGRN_OK) e = cudaStreamWaitEvent(caller, hp->end, 0);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return GGRN_ERR_CUDA;
  }
  return st;
}

}  // namespace
}  // namespace ggrn

extern "C" int ggrn_forward_host(const void* y_host, const void* gate_host, const void* w,
                                 void* out_host, int64_t rows, int64_t width,
                                 int64_t group_size, int64_t y_row_stride,
                                 int64_t gate_row_stride, int64_t out_row_stride, float eps,
                                 int dtype, int mode, void* workspace, int64_t workspace_bytes,
                                 void* cuda_stream) {
  // The host matrices get the checks of ggrn_forward (shapes, dtype, NULL,
  // element alignment, out overlapping y or gate).
  const Args a = call_args(y_host, gate_host, w, out_host, rows, width, group_size, y_row_stride,
                           gate_row_stride, out_row_stride, eps, dtype, mode);
  return forward_host_impl(a, /*packed=*/false, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int ggrn_forward_inproj_host(const void* inproj_host, int64_t inproj_row_stride,
                                        int64_t y_col, int64_t gate_col, const void* w,
                                        void* out_host, int64_t out_row_stride, int64_t rows,
                                        int64_t width, int64_t group_size, float eps, int dtype,
                                        int mode, void* workspace, int64_t workspace_bytes,
                                        void* cuda_stream) {
  if (rows < 0 || width <= 0) return GGRN_ERR_SHAPE;
  if (rows == 0) return GGRN_OK;
  if (!inproj_host) return GGRN_ERR_NULL;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return GGRN_ERR_DTYPE;
  if (y_col < 0 || gate_col < 0 || y_col > inproj_row_stride - width ||
      gate_col > inproj_row_stride - width)
    return GGRN_ERR_SHAPE;
  const int es = es_of(dtype);
  const char* base = static_cast<const char*>(inproj_host);
  const Args a = call_args(base + y_col * es, base + gate_col * es, w, out_host, rows, width,
                           group_size, inproj_row_stride, inproj_row_stride, out_row_stride, eps,
                           dtype, mode);
  return forward_host_impl(a, /*packed=*/true, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(cuda_stream));
}
