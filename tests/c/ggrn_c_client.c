/*
 * A plain C client of the library's C ABI (include/ggrn.h), with no Python
 * in the process: the tests build it with the host C compiler and run it.
 *
 *   ggrn_c_client validate
 *       argument checks that return before anything is enqueued (no GPU
 *       needed): prints "name status" lines.
 *   ggrn_c_client run IN OUT ROWS WIDTH GS DTYPE MODE EPS
 *       IN holds y, gate (ROWS x WIDTH elements of T each) and the weight
 *       (WIDTH f32 in MAMBA2 mode, GS elements of T in ONNX mode), raw and
 *       back to back.  Runs ggrn_forward on device copies and
 *       ggrn_forward_host on pinned host copies, checks the device status
 *       word, and writes the ggrn_forward output to OUT and the
 *       ggrn_forward_host output to OUT.host.
 *   ggrn_c_client packed IN OUT ROWS WIDTH GS DTYPE MODE EPS PACKED_WIDTH GATE_COL
 *       IN holds one packed matrix (ROWS x PACKED_WIDTH elements of T; y is
 *       its columns [0, WIDTH), gate its columns [GATE_COL, GATE_COL +
 *       WIDTH)) and the weight.  Runs ggrn_forward on the two strided views
 *       (row stride PACKED_WIDTH), ggrn_forward_inproj on the packed matrix
 *       and ggrn_forward_host on a pinned host copy of it; writes OUT,
 *       OUT.inproj and OUT.host (contiguous ROWS x WIDTH outputs).
 *
 * The client only moves bytes: inputs come from the tests' seeded generator
 * and the outputs are checked against the oracle by the tests.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ggrn.h"

#define CUDA_OK(call)                                                          \
  do {                                                                         \
    cudaError_t e_ = (call);                                                   \
    if (e_ != cudaSuccess) {                                                   \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));              \
      return 2;                                                                \
    }                                                                          \
  } while (0)

static int validate(void) {
  /* fake, aligned, far-apart addresses: the checks never dereference them */
  const void* y = (const void*)(uintptr_t)0x100000;
  const void* g = (const void*)(uintptr_t)0x200000;
  const void* w = (const void*)(uintptr_t)0x300000;
  void* o = (void*)(uintptr_t)0x400000;
  printf("version %d\n", ggrn_version());
  printf("null_y %d\n", ggrn_forward(NULL, g, w, o, 4, 16, 8, 16, 16, 16, 1e-5f, GGRN_BF16,
                                     GGRN_MODE_MAMBA2, NULL));
  printf("shape %d\n", ggrn_forward(y, g, w, o, 4, 16, 3, 16, 16, 16, 1e-5f, GGRN_BF16,
                                    GGRN_MODE_MAMBA2, NULL));
  printf("dtype %d\n", ggrn_forward(y, g, w, o, 4, 16, 8, 16, 16, 16, 1e-5f, GGRN_BF16,
                                    GGRN_MODE_ONNX, NULL));
  printf("overlap %d\n", ggrn_forward(y, g, w, (void*)(uintptr_t)0x100008, 4, 16, 8, 16, 16, 16,
                                      1e-5f, GGRN_BF16, GGRN_MODE_MAMBA2, NULL));
  printf("rows0 %d\n", ggrn_forward(NULL, NULL, NULL, NULL, 0, 16, 8, 16, 16, 16, 1e-5f,
                                    GGRN_BF16, GGRN_MODE_MAMBA2, NULL));
  printf("host_null_ws %d\n", ggrn_forward_host(y, g, w, o, 4, 16, 8, 16, 16, 16, 1e-5f,
                                                GGRN_BF16, GGRN_MODE_MAMBA2, NULL, 0, NULL));
  printf("status_string_1 %s\n", ggrn_status_string(1));
  return 0;
}

static int run(int argc, char** argv) {
  if (argc != 10) {
    fprintf(stderr, "usage: run IN OUT ROWS WIDTH GS DTYPE MODE EPS\n");
    return 1;
  }
  const char* in_path = argv[2];
  const char* out_path = argv[3];
  const int64_t rows = atoll(argv[4]), width = atoll(argv[5]), gs = atoll(argv[6]);
  const int dtype = atoi(argv[7]), mode = atoi(argv[8]);
  const float eps = (float)atof(argv[9]);
  const size_t es = dtype == GGRN_F32 ? 4 : 2;
  const size_t tbytes = (size_t)rows * (size_t)width * es;
  const size_t wbytes = mode == GGRN_MODE_MAMBA2 ? (size_t)width * 4 : (size_t)gs * es;

  unsigned char *hy, *hg, *hw, *ho_dev, *ho_host;
  CUDA_OK(cudaMallocHost((void**)&hy, tbytes));
  CUDA_OK(cudaMallocHost((void**)&hg, tbytes));
  CUDA_OK(cudaMallocHost((void**)&ho_host, tbytes));
  hw = (unsigned char*)malloc(wbytes);
  ho_dev = (unsigned char*)malloc(tbytes);
  if (!hw || !ho_dev) return 2;
  FILE* f = fopen(in_path, "rb");
  if (!f) return 2;
  if (fread(hy, 1, tbytes, f) != tbytes || fread(hg, 1, tbytes, f) != tbytes ||
      fread(hw, 1, wbytes, f) != wbytes) {
    fprintf(stderr, "short input file\n");
    return 2;
  }
  fclose(f);

  void *dy, *dg, *dw, *dout, *ws;
  CUDA_OK(cudaMalloc(&dy, tbytes));
  CUDA_OK(cudaMalloc(&dg, tbytes));
  CUDA_OK(cudaMalloc(&dw, wbytes));
  CUDA_OK(cudaMalloc(&dout, tbytes));
  CUDA_OK(cudaMemcpy(dy, hy, tbytes, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dg, hg, tbytes, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dw, hw, wbytes, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemset(dout, 0, tbytes));

  uint32_t flags = 0;
  ggrn_fault_status(&flags, 1);
  int st = ggrn_forward(dy, dg, dw, dout, rows, width, gs, width, width, width, eps, dtype, mode,
                        NULL);
  printf("forward %d\n", st);
  if (st != GGRN_OK) return 3;
  CUDA_OK(cudaDeviceSynchronize());
  CUDA_OK(cudaMemcpy(ho_dev, dout, tbytes, cudaMemcpyDeviceToHost));

  const int64_t wsb = ggrn_host_workspace_bytes(rows, width, dtype);
  CUDA_OK(cudaMalloc(&ws, (size_t)wsb));
  memset(ho_host, 0, tbytes);
  st = ggrn_forward_host(hy, hg, dw, ho_host, rows, width, gs, width, width, width, eps, dtype,
                         mode, ws, wsb, NULL);
  printf("forward_host %d\n", st);
  if (st != GGRN_OK) return 3;
  CUDA_OK(cudaDeviceSynchronize());
  ggrn_fault_status(&flags, 0);
  printf("fault %u\n", flags);

  f = fopen(out_path, "wb");
  if (!f || fwrite(ho_dev, 1, tbytes, f) != tbytes) return 2;
  fclose(f);
  char host_path[4096];
  snprintf(host_path, sizeof(host_path), "%s.host", out_path);
  f = fopen(host_path, "wb");
  if (!f || fwrite(ho_host, 1, tbytes, f) != tbytes) return 2;
  fclose(f);
  cudaFree(dy);
  cudaFree(dg);
  cudaFree(dw);
  cudaFree(dout);
  cudaFree(ws);
  cudaFreeHost(hy);
  cudaFreeHost(hg);
  cudaFreeHost(ho_host);
  free(hw);
  free(ho_dev);
  return 0;
}

static int write_file(const char* path, const char* suffix, const void* data, size_t n) {
  char name[4096];
  snprintf(name, sizeof(name), "%s%s", path, suffix);
  FILE* f = fopen(name, "wb");
  if (!f) return 2;
  const size_t w = fwrite(data, 1, n, f);
  fclose(f);
  return w == n ? 0 : 2;
}

static int packed(int argc, char** argv) {
  if (argc != 12) {
    fprintf(stderr, "usage: packed IN OUT ROWS WIDTH GS DTYPE MODE EPS PACKED_WIDTH GATE_COL\n");
    return 1;
  }
  const char* in_path = argv[2];
  const char* out_path = argv[3];
  const int64_t rows = atoll(argv[4]), width = atoll(argv[5]), gs = atoll(argv[6]);
  const int dtype = atoi(argv[7]), mode = atoi(argv[8]);
  const float eps = (float)atof(argv[9]);
  const int64_t pw = atoll(argv[10]), gcol = atoll(argv[11]);
  const size_t es = dtype == GGRN_F32 ? 4 : 2;
  const size_t pbytes = (size_t)rows * (size_t)pw * es;
  const size_t obytes = (size_t)rows * (size_t)width * es;
  const size_t wbytes = mode == GGRN_MODE_MAMBA2 ? (size_t)width * 4 : (size_t)gs * es;

  unsigned char *hp, *hw, *ho, *ho_host;
  CUDA_OK(cudaMallocHost((void**)&hp, pbytes));
  CUDA_OK(cudaMallocHost((void**)&ho_host, obytes));
  hw = (unsigned char*)malloc(wbytes);
  ho = (unsigned char*)malloc(obytes);
  if (!hw || !ho) return 2;
  FILE* f = fopen(in_path, "rb");
  if (!f) return 2;
  if (fread(hp, 1, pbytes, f) != pbytes || fread(hw, 1, wbytes, f) != wbytes) {
    fprintf(stderr, "short input file\n");
    return 2;
  }
  fclose(f);

  void *dp, *dw, *dout;
  CUDA_OK(cudaMalloc(&dp, pbytes));
  CUDA_OK(cudaMalloc(&dw, wbytes));
  CUDA_OK(cudaMalloc(&dout, obytes));
  CUDA_OK(cudaMemcpy(dp, hp, pbytes, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dw, hw, wbytes, cudaMemcpyHostToDevice));
  const unsigned char* dy = (const unsigned char*)dp;
  const unsigned char* dg = dy + (size_t)gcol * es;

  uint32_t flags = 0;
  ggrn_fault_status(&flags, 1);
  int rc = 0;
  CUDA_OK(cudaMemset(dout, 0, obytes));
  int st = ggrn_forward(dy, dg, dw, dout, rows, width, gs, pw, pw, width, eps, dtype, mode, NULL);
  printf("forward %d\n", st);
  if (st != GGRN_OK) return 3;
  CUDA_OK(cudaDeviceSynchronize());
  CUDA_OK(cudaMemcpy(ho, dout, obytes, cudaMemcpyDeviceToHost));
  rc |= write_file(out_path, "", ho, obytes);

  CUDA_OK(cudaMemset(dout, 0, obytes));
  st = ggrn_forward_inproj(dp, pw, 0, gcol, dw, dout, width, rows, width, gs, eps, dtype, mode,
                           NULL);
  printf("forward_inproj %d\n", st);
  if (st != GGRN_OK) return 3;
  CUDA_OK(cudaDeviceSynchronize());
  CUDA_OK(cudaMemcpy(ho, dout, obytes, cudaMemcpyDeviceToHost));
  rc |= write_file(out_path, ".inproj", ho, obytes);

  memset(ho_host, 0, obytes);
  st = ggrn_forward_host(hp, hp + (size_t)gcol * es, dw, ho_host, rows, width, gs, pw, pw, width,
                         eps, dtype, mode, NULL, 0, NULL);
  printf("forward_host %d\n", st);
  if (st != GGRN_OK) return 3;
  CUDA_OK(cudaDeviceSynchronize());
  rc |= write_file(out_path, ".host", ho_host, obytes);
  ggrn_fault_status(&flags, 0);
  printf("fault %u\n", flags);

  cudaFree(dp);
  cudaFree(dw);
  cudaFree(dout);
  cudaFreeHost(hp);
  cudaFreeHost(ho_host);
  free(hw);
  free(ho);
  return rc;
}

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "validate") == 0) return validate();
  if (argc >= 2 && strcmp(argv[1], "run") == 0) return run(argc, argv);
  if (argc >= 2 && strcmp(argv[1], "packed") == 0) return packed(argc, argv);
  fprintf(stderr, "usage: %s validate | run IN OUT ROWS WIDTH GS DTYPE MODE EPS | packed ...\n",
          argv[0]);
  return 1;
}
