// fa_internal.h -- launch interface between the C ABI (fa_api.cu) and the
// kernel translation units.  Host-side only; no device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace fa {

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute belongs to the function as loaded
// on each device, so a process that drives several GPUs sets it on each.
// `done` is the calling launcher's own bitmask of devices already set
// (devices past 63 are set on every call).
template <typename K>
cudaError_t ensure_dynamic_smem(K kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Streaming multiprocessors of the current device (cached per device).
inline cudaError_t sm_count(int* out) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && (*out = cached[dev].load(std::memory_order_relaxed)) > 0)
    return cudaSuccess;
  e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cached[dev].store(*out, std::memory_order_relaxed);
  return e;
}

constexpr int kTile = 128;  // rows of a Q tile and of a K/V tile

// Tensor maps are 4-D {D, N, H, B} over the caller's strides (D contiguous);
// kernels address (batch, head) slice bh as head bh % H, batch bh / H.
// Visible keys: query i sees key j when i - win_left <= j <= i + win_right,
// a negative bound being absent; the causal mask is win_right = 0.  ALiBi:
// the score of (i, j) gets -slope * |i - j| added, slope =
// alibi[(bh / H) * alibi_bstride + bh % H] (alibi == nullptr: no bias).
// Block-sparse: query tile qt multiplies key tile kt (tiles of kTile rows)
// only when block_mask[(bh % H) * bm_head_stride + qt * n_kt + kt] != 0
// (block_mask == nullptr: every tile pair).
struct Band {
  int win_left, win_right;
  const float* alibi;
  int alibi_bstride;
  const uint8_t* block_mask;
  long long bm_head_stride;
};

// Largest number of tiles along N a block-sparse call may have (the tile
// sets live in shared memory as bitmasks).
constexpr int kMaxSparseTiles = 16384;

// 16-bit operands: every map has box 64 x 128 x 1 x 1, 128-byte swizzle.
// 8-bit (e4m3) operands (fp8 != 0, D = 128, O in bf16): map_q and map_k
// have box 128 x 128 bytes; map_v covers V^T, a [B][H][D][Npad16] byte
// tensor with inner extent N, box 128 keys x D rows.
struct FwdLaunch {
  CUtensorMap map_q, map_k, map_v, map_o;
  float* lse;                               // [BH][N]
  int N, BH, D, H;
  float scale_log2;                         // scale * log2(e)
  Band band;
  int bf16;
  int fp8;
  // 8-bit only: per-(batch, head) dequantisation factors, [BH] each, or
  // nullptr for 1
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  int tile_major;  // grid order (tile_major_order)
  uint32_t* err;
};

struct BwdLaunch {
  CUtensorMap map_q, map_k, map_v, map_do;  // box 64 x 128 x 1 x 1
  CUtensorMap map_dq, map_dk, map_dv;       // outputs, same geometry
  CUtensorMap map_q64, map_do64;            // Q and dO again, box 64 x 64 x 1 x 1
  CUtensorMap map_k64, map_v64;             // K and V again, box 64 x 64 x 1 x 1
  // D = 64, atomic mode: dq_accum as fp32 {D, N, H, B}, box 64 x 64 x 1 x 1,
  // no swizzle (the target of the dQ bulk reductions)
  CUtensorMap map_dqacc;
  const float* lse;                         // [BH][Npad] LSE * log2(e), +inf padding
  const float* di;                          // [BH][Npad] rowsum(dO * O), 0 padding
  float* dq_accum;                          // [BH][N][D] or nullptr
  int N, BH, D, H;
  float scale, scale_log2;
  Band band;
  int bf16;
  int tile_major;  // grid order (tile_major_order)
  uint32_t* err;
};

// Grid order of the attention kernels.  Head-major (all tiles of one head,
// then the next) keeps the operands that a head's CTAs share in L2 while
// they run.  When the tiles' lengths differ (a causal band: keys bounded on
// the right only) and the operands every CTA streams fit in L2 together
// (`streamed_bytes`), tile-major order (tile 0 of every head, then tile 1,
// ...) is taken instead: with the longest tiles first, the short tiles fill
// the tail rather than leave one head's longest tile to start last.
inline int tile_major_order(const Band& band, long long streamed_bytes) {
  return band.win_left < 0 && band.win_right >= 0 && streamed_bytes <= (64ll << 20);
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s);
// Element strides of one [B, H, N, D] operand (D contiguous).
struct RowStrides {
  long long batch, head, seq;
};

// V [B, H, N, D] bytes (element strides sv, D = 128) -> vt [BH][D][ld]
// bytes, ld >= N a multiple of 16; columns N .. ld-1 are left as they are.
cudaError_t launch_transpose_v8(const void* v, RowStrides sv, void* vt, int N, long long ld, int H,
                                long long BH, int D, cudaStream_t s);

cudaError_t launch_bwd_preprocess(const void* o, RowStrides so, const void* dO, RowStrides sdo,
                                  const float* lse, float* lse2, float* di, float* dq_accum, int N,
                                  int H, long long BH, int D, int bf16, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdLaunch& a, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t s);
cudaError_t launch_dq_convert(const float* acc, void* dq, RowStrides sdq, int N, int H,
                              long long BH, int D, float scale, int bf16, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s);

// Device address of the error word bounded waits write (current device), or
// nullptr if it cannot be resolved.
uint32_t* device_error_word();

}  // namespace fa
