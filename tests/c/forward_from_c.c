/*
 * forward_from_c.c -- the library driven from plain C through include/moe_ffn.h
 * alone (no Python, no PyTorch): device memory from the CUDA runtime, one
 * bf16 forward pass, its status, and the output written back to a file.
 *
 *   forward_from_c <dir> <T> <E> <D> <H> <k> <pipeline 0 fused | 1 split> [host chunk]
 *
 * With a host chunk (0 automatic, or tokens per chunk) the call is
 * moe_ffn_forward_host: x, ids, weights and out stay in page-locked host
 * memory and the library copies them chunk by chunk.
 *
 * <dir> holds x.bin (bf16 [T, D]), w1.bin (bf16 [E, 2H, D]), w2.bin (bf16
 * [E, D, H]), ids.bin (int32 [T, k]) and w.bin (float32 [T, k]); the program
 * writes out.bin (bf16 [T, D]).  Exit status 0 on success.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe_ffn.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes ? bytes : 1);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 8 && argc != 9) {
    fprintf(stderr, "usage: %s dir T E D H k pipeline [host_chunk]\n", argv[0]);
    return 2;
  }
  const int host = argc == 9;
  const int chunk = host ? atoi(argv[8]) : 0;
  const char* dir = argv[1];
  const int T = atoi(argv[2]), E = atoi(argv[3]), D = atoi(argv[4]), H = atoi(argv[5]), k = atoi(argv[6]);
  const int pipeline = atoi(argv[7]);
  const size_t bx = (size_t)T * D * 2, bw1 = (size_t)E * 2 * H * D * 2, bw2 = (size_t)E * D * H * 2;
  const size_t bids = (size_t)T * k * 4, bw = (size_t)T * k * 4;
  void* hx = read_file(dir, "x.bin", bx);
  void* hw1 = read_file(dir, "w1.bin", bw1);
  void* hw2 = read_file(dir, "w2.bin", bw2);
  void* hids = read_file(dir, "ids.bin", bids);
  void* hw = read_file(dir, "w.bin", bw);
  if (!hx || !hw1 || !hw2 || !hids || !hw) {
    fprintf(stderr, "cannot read the inputs\n");
    return 1;
  }
  void* w1 = to_device(hw1, bw1);
  void* w2 = to_device(hw2, bw2);
  const size_t ws_bytes = host ? moe_ffn_host_workspace_size(T, chunk, E, D, H, k, MOE_BF16, pipeline)
                               : moe_ffn_workspace_size(T, E, D, H, k, MOE_BF16, pipeline);
  void* ws = NULL;
  if (!w1 || !w2 || ws_bytes == 0 || cudaMalloc(&ws, ws_bytes) != cudaSuccess) {
    fprintf(stderr, "device setup failed\n");
    return 1;
  }
  cudaStream_t stream;
  if (cudaStreamCreate(&stream) != cudaSuccess) return 1;
  moe_status_t st = moe_ffn_workspace_init(ws, ws_bytes, stream);
  void* hout = NULL;
  if (host) {
    /* page-locked host buffers: the copies of one chunk overlap the others' computation */
    void *px = NULL, *pids = NULL, *pw = NULL;
    if (cudaHostAlloc(&px, bx, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&pids, bids, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&pw, bw, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&hout, bx, cudaHostAllocDefault) != cudaSuccess) {
      fprintf(stderr, "host allocation failed\n");
      return 1;
    }
    memcpy(px, hx, bx);
    memcpy(pids, hids, bids);
    memcpy(pw, hw, bw);
    if (st == MOE_OK)
      st = moe_ffn_forward_host(px, NULL, w1, NULL, w2, NULL, (const int32_t*)pids, (const float*)pw, hout, T, E, D,
                                H, k, MOE_BF16, pipeline, chunk, ws, ws_bytes, stream);
    if (st == MOE_OK && cudaStreamSynchronize(stream) != cudaSuccess) st = MOE_ERR_CUDA;
    if (st == MOE_OK) st = moe_ffn_sync_status(ws, stream);
  } else {
    void* x = to_device(hx, bx);
    void* ids = to_device(hids, bids);
    void* w = to_device(hw, bw);
    void* out = NULL;
    if (!x || !ids || !w || cudaMalloc(&out, bx) != cudaSuccess) {
      fprintf(stderr, "device setup failed\n");
      return 1;
    }
    if (st == MOE_OK)
      st = moe_ffn_forward(x, NULL, w1, NULL, w2, NULL, (const int32_t*)ids, (const float*)w, out, T, E, D, H, k,
                           MOE_BF16, pipeline, ws, ws_bytes, stream);
    if (st == MOE_OK) st = moe_ffn_sync_status(ws, stream);
    hout = malloc(bx);
    if (st == MOE_OK && (!hout || cudaMemcpy(hout, out, bx, cudaMemcpyDeviceToHost) != cudaSuccess)) return 1;
  }
  if (st != MOE_OK) {
    fprintf(stderr, "moe_ffn: %s\n", moe_ffn_status_string(st));
    return 1;
  }
  char path[4096];
  snprintf(path, sizeof path, "%s/out.bin", dir);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(hout, 1, bx, f) != bx) return 1;
  fclose(f);
  printf("ok: %s pipeline%s, %zu workspace bytes\n", pipeline ? "split" : "fused", host ? ", host buffers" : "",
         ws_bytes);
  return 0;
}
