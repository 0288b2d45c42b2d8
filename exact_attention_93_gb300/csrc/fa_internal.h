// fa_internal.h -- launch interface between the C ABI (fa_api.cu) and the
// kernel translation units.  Host-side only; no device code here.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

namespace fa {

// A process-unique ID of the calling thread's current CUDA context (0 if
// there is none or the driver entry points are unavailable), fetched through
// the runtime's entry-point query so that the library does not link against
// libcuda.  What the library caches per device (device addresses of its
// globals, function attributes) is tagged with it: a cudaDeviceReset
// destroys the context those belong to, and the next call then sets them up
// again.  (The ID, unlike the context's handle, is never reused.)
inline unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The contexts (IDs, one per device) in which a kernel's attribute was set.
struct AttrCache {
  std::mutex mu;
  unsigned long long ctx[64] = {};
};

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device and context: the attribute belongs to the function
// as loaded in each context, so a process that drives several GPUs sets it
// on each, and again after a cudaDeviceReset.  `cache` is the calling
// launcher's own record (devices past 63 are set on every call).
template <typename K>
cudaError_t ensure_dynamic_smem(K kern, int bytes, AttrCache& cache) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < 64;
  const unsigned long long ctx = current_context_id();
  if (tracked && ctx != 0) {
    std::lock_guard<std::mutex> lock(cache.mu);
    if (cache.ctx[dev] == ctx) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked && ctx != 0) {
    std::lock_guard<std::mutex> lock(cache.mu);
    cache.ctx[dev] = ctx;
  }
  return e;
}

// Launches kern with programmatic stream serialization: its CTAs may start
// while the preceding kernel in the stream runs its last ones, instead of
// after it.  A kernel launched this way starts with pdl_wait() or
// pdl_wait_and_release() (sm103_primitives.cuh), which return once that
// kernel has completed and its writes are visible, before it touches global
// memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
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
