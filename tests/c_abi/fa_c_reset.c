/*
 * libfattn across a cudaDeviceReset, from plain C.  The library caches per
 * device what it sets up once (the device addresses of its error word and of
 * the no-allocation entry point's scratch array, the kernels' shared-memory
 * attribute); a reset replaces the device's context, and those must be set
 * up again in the new one.  The program runs the forward and fa_bwd_noalloc
 * on seeded buffers, resets the device, allocates and runs the same again,
 * and checks that both runs give bit-identical outputs and report no device
 * error.
 *
 *   fa_c_reset B H N D causal
 *
 * Exit status 0 when both runs agree; otherwise the failing step is printed.
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

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

/* bf16 bits of a small pseudo-random value in about [-2, 2) */
static unsigned short draw(unsigned* state) {
  *state = *state * 1664525u + 1013904223u;
  const float x = ((float)(*state >> 8) / 16777216.0f) * 4.0f - 2.0f;
  unsigned bits;
  memcpy(&bits, &x, sizeof bits);
  return (unsigned short)(bits >> 16);
}

/* One forward + no-allocation backward; outputs (O, LSE, dQ, dK, dV) to out. */
static int run(const unsigned short* in, unsigned char* out, int B, int H, int N, int D,
               int causal) {
  const size_t n = (size_t)B * H * N * D, rows = (size_t)B * H * N, bytes16 = n * 2;
  void *q, *k, *v, *dO, *o, *dq, *dk, *dv;
  float* lse;
  CUDA_OK(cudaMalloc(&q, bytes16));
  CUDA_OK(cudaMalloc(&k, bytes16));
  CUDA_OK(cudaMalloc(&v, bytes16));
  CUDA_OK(cudaMalloc(&dO, bytes16));
  CUDA_OK(cudaMalloc(&o, bytes16));
  CUDA_OK(cudaMalloc(&dq, bytes16));
  CUDA_OK(cudaMalloc(&dk, bytes16));
  CUDA_OK(cudaMalloc(&dv, bytes16));
  CUDA_OK(cudaMalloc((void**)&lse, rows * sizeof(float)));
  CUDA_OK(cudaMemcpy(q, in, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(k, in + n, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(v, in + 2 * n, bytes16, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dO, in + 3 * n, bytes16, cudaMemcpyHostToDevice));
  const float scale = 1.0f / (float)D;
  FA_OK_(fa_fwd(q, k, v, o, lse, B, H, N, D, scale, causal, FA_BF16, 0));
  FA_OK_(fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, D, scale, causal, FA_BF16, 0));
  CUDA_OK(cudaDeviceSynchronize());
  int dev_err = -1;
  FA_OK_(fa_device_error(0, &dev_err));
  if (dev_err != FA_OK) {
    fprintf(stderr, "device error %d\n", dev_err);
    return 1;
  }
  CUDA_OK(cudaMemcpy(out, o, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out + bytes16, lse, rows * sizeof(float), cudaMemcpyDeviceToHost));
  unsigned char* g = out + bytes16 + rows * sizeof(float);
  CUDA_OK(cudaMemcpy(g, dq, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(g + bytes16, dk, bytes16, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(g + 2 * bytes16, dv, bytes16, cudaMemcpyDeviceToHost));
  cudaFree(q);
  cudaFree(k);
  cudaFree(v);
  cudaFree(dO);
  cudaFree(o);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(lse);
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s B H N D causal\n", argv[0]);
    return 2;
  }
  const int B = atoi(argv[1]), H = atoi(argv[2]), N = atoi(argv[3]), D = atoi(argv[4]);
  const int causal = atoi(argv[5]);
  const size_t n = (size_t)B * H * N * D, rows = (size_t)B * H * N;
  const size_t out_bytes = 4 * n * 2 + rows * sizeof(float);
  unsigned short* in = (unsigned short*)malloc(4 * n * sizeof(unsigned short));
  unsigned char* a = (unsigned char*)malloc(out_bytes);
  unsigned char* b = (unsigned char*)malloc(out_bytes);
  if (!in || !a || !b) return 1;
  unsigned state = 12345u;
  for (size_t i = 0; i < 4 * n; ++i) in[i] = draw(&state);
  if (run(in, a, B, H, N, D, causal)) return 1;
  CUDA_OK(cudaDeviceReset());
  if (run(in, b, B, H, N, D, causal)) return 1;
  if (memcmp(a, b, out_bytes) != 0) {
    fprintf(stderr, "outputs differ after the reset\n");
    return 1;
  }
  printf("identical across a device reset\n");
  free(in);
  free(a);
  free(b);
  return 0;
}
