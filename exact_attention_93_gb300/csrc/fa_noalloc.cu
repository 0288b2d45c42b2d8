// fa_noalloc.cu -- a backward entry point that allocates no device memory.
//
// fa_bwd needs a caller-provided workspace.  Some callers cannot provide
// one: a plug-in invoked from another framework's execution step that is
// handed only its input and output tensors and no allocator, or a
// latency-bound caller for which cudaMalloc (which can synchronise the whole
// device) is not acceptable mid-step.  fa_bwd_noalloc serves them: it runs
// the deterministic two-pass backward, whose only scratch is the padded
// log2-LSE and Di rows, out of one fixed array in device memory that is part
// of the loaded library.
//
// The array's name is only a host-side stand-in for the device object, so
// host code never passes it to a kernel: the device address is resolved with
// cudaGetSymbolAddress once per device (on the first call made while that
// device is current) and that address is what the kernels receive.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fattn.h"
#include "fa_internal.h"
#include "host_tmap.hpp"

namespace fa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (set up on the
// first call per device, and again on the first call after the device's
// context was replaced, e.g. by cudaDeviceReset); nullptr if it cannot be
// resolved.
unsigned char* scratch_ptr() {
  static unsigned char* ptrs[kMaxDevices] = {};
  static unsigned long long ctxs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev] || ctxs[dev] != ctx) {
    unsigned char* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch) != cudaSuccess)
      return nullptr;
    ptrs[dev] = p;
    ctxs[dev] = ctx;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Contiguous [B, H, N, D] operand.
bool tile_map(CUtensorMap* m, const void* base, int B, int H, int N, int D, int dtype,
              int box_rows = kTile) {
  return operand_map(m, base, dtype == FA_BF16, B, H, N, D, static_cast<long long>(H) * N * D,
                     static_cast<long long>(N) * D, D, box_rows);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int D, float scale, int causal,
                                    fa_dtype dtype, void* stream) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffLL || static_cast<double>(BH) * N * D >= 1099511627776.0)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  // Scratch: lse2 and di, one fp32 per query row padded to whole tiles.
  const size_t rows = static_cast<size_t>(BH) * ((N + kTile - 1) / kTile * kTile);
  const size_t di_off = round256(rows * 4);
  if (di_off + round256(rows * 4) > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_UNSUPPORTED;

  unsigned char* scratch = scratch_ptr();
  uint32_t* err = device_error_word();
  if (!scratch || !err) return FA_ERR_CUDA;

  BwdLaunch a{};
  if (!tile_map(&a.map_q, q, B, H, N, D, dtype) || !tile_map(&a.map_k, k, B, H, N, D, dtype) ||
      !tile_map(&a.map_v, v, B, H, N, D, dtype) || !tile_map(&a.map_do, dO, B, H, N, D, dtype) ||
      !tile_map(&a.map_dq, dq, B, H, N, D, dtype) || !tile_map(&a.map_dk, dk, B, H, N, D, dtype) ||
      !tile_map(&a.map_dv, dv, B, H, N, D, dtype) ||
      !tile_map(&a.map_q64, q, B, H, N, D, dtype, 64) ||
      !tile_map(&a.map_do64, dO, B, H, N, D, dtype, 64) ||
      !tile_map(&a.map_k64, k, B, H, N, D, dtype, 64) ||
      !tile_map(&a.map_v64, v, B, H, N, D, dtype, 64))
    return FA_ERR_CUDA;
  float* lse2 = reinterpret_cast<float*>(scratch);
  float* di = reinterpret_cast<float*>(scratch + di_off);
  a.lse = lse2;
  a.di = di;
  a.dq_accum = nullptr;  // two-pass dQ: nothing in the scratch has to start at zero
  a.N = N;
  a.BH = static_cast<int>(BH);
  a.D = D;
  a.H = H;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.band = Band{-1, causal ? 0 : -1, nullptr, 0, nullptr, 0};
  a.bf16 = dtype == FA_BF16 ? 1 : 0;
  a.err = err;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // The preprocess rewrites every scratch entry the later kernels read
  // (padding rows included), so the previous call's contents never leak in.
  const RowStrides rows_c{static_cast<long long>(H) * N * D, static_cast<long long>(N) * D, D};
  if (launch_bwd_preprocess(o, rows_c, dO, rows_c, lse, lse2, di, nullptr, N, H, BH, D, a.bf16,
                            cs) != cudaSuccess)
    return FA_ERR_CUDA;
  if (launch_bwd_dkdv(a, cs) != cudaSuccess) return FA_ERR_CUDA;
  return launch_bwd_dq(a, cs) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
