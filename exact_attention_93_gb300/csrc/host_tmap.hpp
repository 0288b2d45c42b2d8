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

// A [slices][rows][inner] tensor of 2- or 4-byte elements, rows `row_stride`
// elements apart, slices `slice_stride` elements apart.  Boxes are
// box_inner x box_rows x 1; out-of-range rows read as zero.
// Returns false when the driver rejects the map (alignment, sizes).
inline bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         int elem_bytes, uint64_t inner, uint64_t rows, uint64_t slices,
                         uint64_t row_stride, uint64_t slice_stride, uint32_t box_inner,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, rows, slices};
  cuuint64_t strides[2] = {row_stride * elem_bytes, slice_stride * elem_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
