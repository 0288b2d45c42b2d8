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

// Whether the block mask keeps the pair (query tile qt, key tile kt) of
// slice bh; n_kt key tiles per mask row.
__device__ __forceinline__ bool block_kept(const Band& b, int bh, int H, int n_kt, int qt,
                                           int kt) {
  return b.block_mask[(bh % H) * b.bm_head_stride + static_cast<long long>(qt) * n_kt + kt] != 0;
}

// A set of tile indices 0 .. n - 1 held as a bitmask in shared memory.
struct TileSet {
  const uint32_t* w;
  int n;
  __device__ __forceinline__ bool has(int x) const { return (w[x >> 5] >> (x & 31)) & 1u; }
  // The first member >= x, or n when there is none.
  __device__ __forceinline__ int next(int x) const {
    if (x >= n) return n;
    int i = x >> 5;
    uint32_t bits = w[i] & (0xffffffffu << (x & 31));
    const int nw = (n + 31) >> 5;
    while (bits == 0) {
      if (++i >= nw) return n;
      bits = w[i];
    }
    return min(n, (i << 5) + __ffs(bits) - 1);
  }
  __device__ __forceinline__ int count() const {
    int c = 0;
    for (int i = 0; i < (n + 31) >> 5; ++i) c += __popc(w[i]);
    return c;
  }
};

// The tiles a kernel walks, in increasing order: the range [lo, hi]
// (dense) or the members of `set` (block-sparse); `end` ends every walk.
template <bool kSparse>
struct TileWalk {
  int lo, hi, end;
  TileSet set;
  __device__ __forceinline__ int first() const {
    return kSparse ? set.next(0) : (lo <= hi ? lo : end);
  }
  __device__ __forceinline__ int next(int x) const {
    return kSparse ? set.next(x + 1) : (x + 1 <= hi ? x + 1 : end);
  }
  __device__ __forceinline__ int count() const {
    return kSparse ? set.count() : max(0, hi - lo + 1);
  }
};

// words[0 .. ceil(n / 32)) = { x < n : pred(x) }, built by every thread of
// the block; a __syncthreads() must follow before the set is read.
template <class Pred>
__device__ __forceinline__ void fill_tile_set(uint32_t* words, int n, Pred pred) {
  const int nw = (n + 31) >> 5;
  for (int i = threadIdx.x; i < nw; i += blockDim.x) {
    uint32_t bits = 0;
    for (int b = 0; b < 32; ++b) {
      const int x = (i << 5) + b;
      if (x < n && pred(x)) bits |= 1u << b;
    }
    words[i] = bits;
  }
}

}  // namespace fa
