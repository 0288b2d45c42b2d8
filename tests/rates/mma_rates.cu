// mma_rates.cu -- cycles per tcgen05.mma product of the shapes the tile
// kernels issue, measured on every SM at once.
//
// One CTA per SM (128 threads, a large shared-memory request keeps a second
// CTA off the SM).  Warp 0 allocates TMEM; warp 1 runs the issue loop with
// all lanes and one elected lane issuing, as the kernels do, and times a run
// of kProducts back-to-back bf16 products accumulating into one TMEM
// accumulator, from the first issue until the commit that covers the last
// one has arrived.  Operands are zero-filled 128-byte-swizzled tiles in
// shared memory (the rate does not depend on the values).  Prints one JSON
// line: the median over CTAs of the cycles per product for each shape.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_runtime.h>

#include "sm103_primitives.cuh"

using namespace fa;

constexpr int kThreads = 128, kProducts = 512;

struct alignas(1024) Tiles {
  uint8_t a[256 * 128];  // up to 256 rows x 128 bytes (64 bf16)
  uint8_t b[256 * 128];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

// kShape: 0 = M128 N128 K16, A and B in shared memory
//         1 = M128 N64  K16, both in shared memory
//         2 = M128 N256 K16, both in shared memory
//         3 = M128 N128 K16, A in TMEM (packed bf16 pairs), B in shared memory
template <int kShape>
__global__ void __launch_bounds__(kThreads, 1) mma_rate_kernel(unsigned long long* cycles,
                                                              uint32_t* err) {
  extern __shared__ uint8_t raw[];
  Tiles& t = *reinterpret_cast<Tiles*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 256 * 128 / 16; i += kThreads) {
    reinterpret_cast<uint4*>(t.a)[i] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(t.b)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    mbar_init(&t.done, 1);
    t.abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&t.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = t.tmem_base;
  if (warp == 1) {
    const bool leader = elect_one_sync();
    constexpr uint32_t N = kShape == 1 ? 64 : (kShape == 2 ? 256 : 128);
    constexpr uint32_t id = idesc_f16(128, N, 1, 0, 0);  // bf16, both K-major
    const uint64_t da = smem_desc_sw128(smem_u32(t.a), 16, 1024);
    const uint64_t db = smem_desc_sw128(smem_u32(t.b), 16, 1024);
    // accumulator in columns [256, 256 + N) (N = 256: [0, 256)); A from TMEM
    // (shape 3) in columns [0, 64)
    const uint32_t d_col = kShape == 2 ? 0u : 256u;
    const unsigned long long t0 = clock64();
    for (int i = 0; i < kProducts; ++i) {
      const uint32_t kk = static_cast<uint32_t>(i & 3);  // 16-element steps within the 64-wide block
      if (leader) {
        if constexpr (kShape == 3)
          tc_mma_ts(tbase + d_col, tbase + kk * 8, desc_add(db, kk * 32), id, i > 0 ? 1u : 0u);
        else
          tc_mma_ss(tbase + d_col, desc_add(da, kk * 32), desc_add(db, kk * 32), id, i > 0 ? 1u : 0u);
      }
    }
    if (leader) tc_commit(&t.done);
    const bool ok = mbar_wait(&t.done, 0, err, &t.abort_flag, 1000000000ull);
    const unsigned long long t1 = clock64();
    if (leader && ok) cycles[blockIdx.x] = t1 - t0;
    if (leader && !ok) cycles[blockIdx.x] = 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int kShape>
static double measure(int sms, uint32_t* err) {
  unsigned long long* cyc = nullptr;
  if (cudaMalloc(&cyc, sizeof(unsigned long long) * sms) != cudaSuccess) return -1.0;
  const int smem = 200 * 1024;
  if (cudaFuncSetAttribute(mma_rate_kernel<kShape>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1.0;
  for (int rep = 0; rep < 2; ++rep) mma_rate_kernel<kShape><<<sms, kThreads, smem>>>(cyc, err);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return -1.0;
  std::vector<unsigned long long> h(sms);
  cudaMemcpy(h.data(), cyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
  cudaFree(cyc);
  std::sort(h.begin(), h.end());
  if (h[0] == 0) return -1.0;  // a wait ran out
  return static_cast<double>(h[sms / 2]) / kProducts;
}

int main() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 2;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint32_t* err = nullptr;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return 2;
  cudaMemset(err, 0, sizeof(uint32_t));
  const double c0 = measure<0>(sms, err), c1 = measure<1>(sms, err), c2 = measure<2>(sms, err),
               c3 = measure<3>(sms, err);
  uint32_t e = 0;
  cudaMemcpy(&e, err, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (c0 < 0 || c1 < 0 || c2 < 0 || c3 < 0 || e != 0) return 3;
  printf("{\"sms\": %d, \"m128n128k16_ss\": %.1f, \"m128n64k16_ss\": %.1f, "
         "\"m128n256k16_ss\": %.1f, \"m128n128k16_ts\": %.1f}\n",
         sms, c0, c1, c2, c3);
  return 0;
}
