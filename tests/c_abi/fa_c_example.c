/*
 * libfattn from plain C: no Python, no torch.  Reads bf16 Q, K, V, dO
 * ([B, H, N, D], contiguous, in that order) from a file, runs the forward
 * and the deterministic backward through the C ABI on device buffers it
 * allocates itself, and writes O, LSE, dQ, dK, dV to a second file for the
 * test to compare with the oracle.
 *
 *   fa_c_example <inputs> <outputs> B H N D causal
 *
 * Exit status 0 on success; otherwise the failing call is printed.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "fattn.h"

#define CUDA_OK(x)                                                            \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      return 1;                                                               \
    }                                                                         \
  } while (0)

#define FA_OK_(x)                                                             \
  do {                                                                        \
    fa_status s_ = (x);                                                       \
    if (s_ != FA_OK) {                                                        \
      fprintf(stderr, "%s: %s\n", #x, fa_status_string(s_));                  \
      return 1;                                                               \
    }                                                                         \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s inputs outputs B H N D causal\n", argv[0]);
    return 2;
  }
  const int B = atoi(argv[3]), H = atoi(argv[4]), N = atoi(argv[5]), D = atoi(argv[6]);
  const int causal = atoi(argv[7]);
  const size_t n = (size_t)B * H * N * D, rows = (size_t)B * H * N;
  const size_t bytes16 = n * 2;

  unsigned char* host = (unsigned char*)malloc(4 * bytes16);
  FILE* f = fopen(argv[1], "rb");
  if (!host || !f || fread(host, 1, 4 * bytes16, f) != 4 * bytes16) {
    fprintf(stderr, "cannot read %s\n", argv[1]);
    return 1;
  }
  fclose(f);

  void *q, *k, *v, *dO, *o, *dq, *dk, *dv, *ws;
  float* lse;
  CUDA_OK(cudaMalloc(&q, bytes16));
  CUDA_OK(cudaMalloc(&k, bytes16));
  CUDA_OK(cudaMalloc(&v, bytes16));
  CUDA_OK(cudaMalloc(&dO, bytes16));
  CUDA_OK(cudaMalloc(&o, bytes16));
  CUDA_OK(cudaMalloc(&dq, bytes16));
  CUDA_OK(cudaMalloc(&dk, bytes16));
  CUDA_OK(cudaMalloc(&dv, bytes16));
  CUDA_OK(cudaMalloc((void**)&lse, rows * 4));
  const size_t ws_bytes = fa_bwd_workspace_size(B, H, N, D, 1);
  if (ws_bytes == 0) {
    fprintf(stderr, "fa_bwd_workspace_size rejected the sizes\n");
    return 1;
  }
  CUDA_OK(cudaMalloc(&ws, ws_bytes));  /* cudaMalloc aligns to 256 bytes */
  CUDA_OK(cudaMemcpy(q, host, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(k, host + bytes16, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(v, host + 2 * bytes16, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dO, host + 3 * bytes16, bytes16, cudaMemcpyHostToDevice));

  cudaStream_t stream;
  CUDA_OK(cudaStreamCreate(&stream));
  const float scale = 1.0f / sqrtf((float)D);
  FA_OK_(fa_fwd(q, k, v, o, lse, B, H, N, D, scale, causal, FA_BF16, stream));
  FA_OK_(fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, D, scale, causal, FA_BF16, 1, ws,
                ws_bytes, stream));
  CUDA_OK(cudaStreamSynchronize(stream));
  int code = FA_OK;
  FA_OK_(fa_device_error(stream, &code));
  if (code != FA_OK) {
    fprintf(stderr, "a kernel reported %s\n", fa_status_string((fa_status)code));
    return 1;
  }

  unsigned char* out = (unsigned char*)malloc(4 * bytes16 + rows * 4);
  if (!out) return 1;
  CUDA_OK(cudaMemcpy(out, o, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out + bytes16, lse, rows * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out + bytes16 + rows * 4, dq, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out + 2 * bytes16 + rows * 4, dk, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out + 3 * bytes16 + rows * 4, dv, bytes16, cudaMemcpyDeviceToHost));
  f = fopen(argv[2], "wb");
  if (!f || fwrite(out, 1, 4 * bytes16 + rows * 4, f) != 4 * bytes16 + rows * 4) {
    fprintf(stderr, "cannot write %s\n", argv[2]);
    return 1;
  }
  fclose(f);
  printf("abi %d: forward and deterministic backward done\n", fa_abi_version());
  return 0;
}
