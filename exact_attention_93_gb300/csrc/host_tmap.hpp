// host_tmap.hpp -- builds TMA tensor maps (CUtensorMap) on the host.
//
// The driver's cuTensorMapEncodeTiled is fetched through the runtime's
// entry-point query, so the library does not link against libcuda and still
// loads on a machine without a GPU driver.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [batch][head][rows][inner] tensor of elem_bytes-byte elements with
// arbitrary element strides for rows, heads and batches (inner contiguous).
// Boxes are box_inner x box_rows x 1 x 1; out-of-range rows (and inner
// elements) read as zero and are not written.  Returns false when the driver
// rejects the map (alignment, sizes).
inline bool make_tmap_4d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t inner, uint64_t rows, uint64_t heads, uint64_t batches,
                         uint64_t row_stride, uint64_t head_stride, uint64_t batch_stride,
                         uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                         uint64_t elem_bytes = 2) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {inner, rows, heads, batches};
  cuuint64_t strides[3] = {row_stride * elem_bytes, head_stride * elem_bytes,
                           batch_stride * elem_bytes};
  cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The map every tile kernel uses for a [B, H, N, D] operand: 64-column blocks
// (128 bytes, 128-byte swizzle) of box_rows rows.
inline bool operand_map(CUtensorMap* map, const void* base, bool bf16, int B, int H, int N, int D,
                        long long batch_stride, long long head_stride, long long seq_stride,
                        int box_rows) {
  return make_tmap_4d(map, base,
                      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      static_cast<uint64_t>(D), static_cast<uint64_t>(N),
                      static_cast<uint64_t>(H), static_cast<uint64_t>(B),
                      static_cast<uint64_t>(seq_stride), static_cast<uint64_t>(head_stride),
                      static_cast<uint64_t>(batch_stride), 64, static_cast<uint32_t>(box_rows),
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// An 8-bit [B, H, N, D] operand, one whole row per box row: D = 128 with
// 128-byte swizzle, D = 64 with 64-byte swizzle.
inline bool operand_map_u8(CUtensorMap* map, const void* base, int B, int H, int N, int D,
                           long long batch_stride, long long head_stride, long long seq_stride,
                           int box_rows) {
  return make_tmap_4d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(D),
                      static_cast<uint64_t>(N), static_cast<uint64_t>(H),
                      static_cast<uint64_t>(B), static_cast<uint64_t>(seq_stride),
                      static_cast<uint64_t>(head_stride), static_cast<uint64_t>(batch_stride),
                      static_cast<uint32_t>(D), static_cast<uint32_t>(box_rows),
                      D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, 1);
}

}  // namespace fa
