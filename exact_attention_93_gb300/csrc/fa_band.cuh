// fa_band.cuh -- which keys a query sees, tile by tile.
//
// The visible keys of query i form one band, i - left <= j <= i + right, a
// negative bound being absent: the sliding window of flash_attn_func's
// window_size (claire-chang.com FlashAttention introduction), with the
// causal mask as right = 0 ("FlashAttention from scratch" walkthrough,
// sec. 5.3: query i sees keys j <= i).  Keys past N are never visible.
#pragma once

#include "fa_internal.h"

namespace fa {

__host__ __device__ __forceinline__ bool band_visible(int i, int j, int left, int right) {
  return (left < 0 || j >= i - left) && (right < 0 || j <= i + right);
}

// Whether some pair of query rows [q0, q0 + nq) and keys [k0, k0 + nk) lies
// outside the band (the tile needs an element mask).
__host__ __device__ __forceinline__ bool band_cuts(int q0, int nq, int k0, int nk, int left,
                                                   int right) {
  return (left >= 0 && k0 < q0 + nq - 1 - left) || (right >= 0 && k0 + nk - 1 > q0 + right);
}

// Key tiles [lo, hi] (tiles of tk keys) that query rows [q0, q0 + nq) see,
// among n_kt tiles.  Never empty for rows below N: each query sees itself.
__host__ __device__ __forceinline__ void band_key_tiles(int q0, int nq, int tk, int n_kt,
                                                        int left, int right, int& lo, int& hi) {
  lo = left < 0 ? 0 : max(0, q0 - left) / tk;
  hi = right < 0 ? n_kt - 1 : min(n_kt - 1, (q0 + nq - 1 + right) / tk);
}

// Query tiles [lo, hi] (tiles of tq rows) that see some key in
// [k0, k0 + nk), among n_qt tiles.
__host__ __device__ __forceinline__ void band_query_tiles(int k0, int nk, int tq, int n_qt,
                                                          int left, int right, int& lo, int& hi) {
  lo = right < 0 ? 0 : max(0, k0 - right) / tq;
  hi = left < 0 ? n_qt - 1 : min(n_qt - 1, (k0 + nk - 1 + left) / tq);
}

// ALiBi slope of slice bh, times log2(e) and negated: the bias in log2
// units is alibi_nslope2(...) * |i - j|.
__device__ __forceinline__ float alibi_nslope2(const Band& b, int bh, int H) {
  return -1.4426950408889634f * b.alibi[(bh / H) * b.alibi_bstride + bh % H];
}

}  // namespace fa
