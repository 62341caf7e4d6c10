/*
 * A plain C caller of libaq.so through include/aq.h, with host buffers:
 * the end-to-end leg of the decode GEMV as a C program would run it.
 *
 *   c_abi_e2e n k m iters W.bin x.bin y.bin
 *
 * W.bin holds the bf16 weight [n, k] and x.bin the m activation rows [m, k],
 * both as little-endian uint16 bit patterns.  The program quantises the
 * weight once (aq_quantize_nvfp4), then times `iters` calls of
 *   host -> device copy of x, aq_gemv_nvfp4 (AQ_PATH_AUTO),
 *   device -> host copy of y
 * on one stream between two CUDA events, from pinned host memory.  It writes
 * the last call's y [m, n] to y.bin and prints one JSON line.  Every failing
 * call ends the program with exit status 1 and the library's message.
 * Only the CUDA runtime's allocation, copy, event and stream calls are used
 * besides the library's own entry points.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "aq.h"

static void fail_cuda(cudaError_t e, const char *what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "c_abi_e2e: %s: %s\n", what, cudaGetErrorString(e));
    exit(1);
  }
}

static void fail_aq(aq_status s, const char *what) {
  if (s != AQ_OK) {
    fprintf(stderr, "c_abi_e2e: %s: status %d: %s\n", what, (int)s, aq_last_error());
    exit(1);
  }
}

/* Reads exactly `bytes` bytes of `path` into `dst`. */
static void read_file(const char *path, void *dst, size_t bytes) {
  FILE *f = fopen(path, "rb");
  if (!f) {
    fprintf(stderr, "c_abi_e2e: cannot open %s\n", path);
    exit(1);
  }
  const size_t got = fread(dst, 1, bytes, f);
  fclose(f);
  if (got != bytes) {
    fprintf(stderr, "c_abi_e2e: %s holds %zu bytes, %zu expected\n", path, got, bytes);
    exit(1);
  }
}

int main(int argc, char **argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: c_abi_e2e n k m iters W.bin x.bin y.bin\n");
    return 2;
  }
  const int32_t n = (int32_t)atoi(argv[1]), k = (int32_t)atoi(argv[2]);
  const int32_t m = (int32_t)atoi(argv[3]);
  const int iters = atoi(argv[4]);
  if (n <= 0 || k <= 0 || m <= 0 || m > AQ_MAX_M || iters <= 0) {
    fprintf(stderr, "c_abi_e2e: bad sizes\n");
    return 2;
  }
  const size_t w_bytes = (size_t)n * k * 2, x_bytes = (size_t)m * k * 2;
  const size_t y_bytes = (size_t)m * n * 2;
  const size_t packed_bytes = aq_packed_bytes(n, k), scale_bytes = aq_scale_bytes(n, k);
  const size_t qws_bytes = aq_quantize_workspace_bytes();
  const size_t gws_bytes = aq_gemv_workspace_bytes(n, k, m);
  if (packed_bytes == 0 || scale_bytes == 0 || gws_bytes == 0) {
    fprintf(stderr, "c_abi_e2e: shape [%d, %d] outside the library's limits\n", n, k);
    return 2;
  }

  /* pinned host buffers */
  uint16_t *h_w, *h_x, *h_y;
  fail_cuda(cudaMallocHost((void **)&h_w, w_bytes), "cudaMallocHost W");
  fail_cuda(cudaMallocHost((void **)&h_x, x_bytes), "cudaMallocHost x");
  fail_cuda(cudaMallocHost((void **)&h_y, y_bytes), "cudaMallocHost y");
  read_file(argv[5], h_w, w_bytes);
  read_file(argv[6], h_x, x_bytes);

  /* device buffers, owned here; the library allocates nothing */
  uint16_t *d_w, *d_x, *d_y;
  uint8_t *d_packed, *d_scales;
  float *d_gdec;
  void *d_qws, *d_gws;
  fail_cuda(cudaMalloc((void **)&d_w, w_bytes), "cudaMalloc W");
  fail_cuda(cudaMalloc((void **)&d_x, x_bytes), "cudaMalloc x");
  fail_cuda(cudaMalloc((void **)&d_y, y_bytes), "cudaMalloc y");
  fail_cuda(cudaMalloc((void **)&d_packed, packed_bytes), "cudaMalloc packed");
  fail_cuda(cudaMalloc((void **)&d_scales, scale_bytes), "cudaMalloc scales");
  fail_cuda(cudaMalloc((void **)&d_gdec, sizeof(float)), "cudaMalloc g_dec");
  fail_cuda(cudaMalloc(&d_qws, qws_bytes), "cudaMalloc quantise workspace");
  fail_cuda(cudaMalloc(&d_gws, gws_bytes), "cudaMalloc GEMV workspace");
  /* both workspaces are zero-filled once after allocation */
  fail_cuda(cudaMemset(d_qws, 0, qws_bytes), "cudaMemset quantise workspace");
  fail_cuda(cudaMemset(d_gws, 0, gws_bytes), "cudaMemset GEMV workspace");

  cudaStream_t st;
  fail_cuda(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking), "cudaStreamCreate");
  const aq_stream_t ast = (aq_stream_t)st;

  /* load time: the weight once to the device, quantised there */
  aq_nvfp4_weight w;
  w.n = n;
  w.k = k;
  w.packed = d_packed;
  w.scales = d_scales;
  w.global_scale = d_gdec;
  fail_cuda(cudaMemcpyAsync(d_w, h_w, w_bytes, cudaMemcpyHostToDevice, st), "copy W");
  fail_aq(aq_quantize_nvfp4(d_w, n, k, &w, d_qws, qws_bytes, ast), "aq_quantize_nvfp4");
  fail_cuda(cudaStreamSynchronize(st), "quantise");
  fail_aq(aq_poll_device_status(ast), "device status after quantisation");

  /* per call: x in, the GEMV, y out -- all on the one stream */
  cudaEvent_t e0, e1;
  fail_cuda(cudaEventCreate(&e0), "cudaEventCreate");
  fail_cuda(cudaEventCreate(&e1), "cudaEventCreate");
  for (int i = -3; i < iters; ++i) { /* three untimed warm-up calls */
    if (i == 0) fail_cuda(cudaEventRecord(e0, st), "cudaEventRecord");
    fail_cuda(cudaMemcpyAsync(d_x, h_x, x_bytes, cudaMemcpyHostToDevice, st), "copy x");
    fail_aq(aq_gemv_nvfp4(&w, d_x, m, d_y, AQ_PATH_AUTO, d_gws, gws_bytes, ast),
            "aq_gemv_nvfp4");
    fail_cuda(cudaMemcpyAsync(h_y, d_y, y_bytes, cudaMemcpyDeviceToHost, st), "copy y");
  }
  fail_cuda(cudaEventRecord(e1, st), "cudaEventRecord");
  fail_cuda(cudaEventSynchronize(e1), "cudaEventSynchronize");
  fail_aq(aq_poll_device_status(ast), "device status after the GEMV calls");
  float ms = 0.0f;
  fail_cuda(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime");

  FILE *f = fopen(argv[7], "wb");
  if (!f || fwrite(h_y, 1, y_bytes, f) != y_bytes) {
    fprintf(stderr, "c_abi_e2e: cannot write %s\n", argv[7]);
    return 1;
  }
  fclose(f);

  const double us = 1e3 * (double)ms / iters;
  const double weight_bytes = (double)packed_bytes + (double)scale_bytes;
  printf("{\"n\": %d, \"k\": %d, \"m\": %d, \"iters\": %d, \"us_per_call\": %.3f, "
         "\"weight_GBps\": %.1f, \"h2d_bytes_per_call\": %zu, \"d2h_bytes_per_call\": %zu}\n",
         n, k, m, iters, us, weight_bytes / us / 1e3, x_bytes, y_bytes);

  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaStreamDestroy(st);
  cudaFree(d_w);
  cudaFree(d_x);
  cudaFree(d_y);
  cudaFree(d_packed);
  cudaFree(d_scales);
  cudaFree(d_gdec);
  cudaFree(d_qws);
  cudaFree(d_gws);
  cudaFreeHost(h_w);
  cudaFreeHost(h_x);
  cudaFreeHost(h_y);
  return 0;
}
