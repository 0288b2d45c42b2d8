// fa_api.cu -- the C ABI of libfattn (declared in include/fattn.h): argument
// checks, TMA descriptor set-up, workspace layout and kernel launches.  No
// attention arithmetic lives here.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fattn.h"
#include "fa_internal.h"
#include "host_tmap.hpp"

namespace fa {
namespace {

__device__ uint32_t g_error_word;  // written by bounded waits that run out

constexpr int kMaxDevices = 64;

uint32_t* error_word_ptr() {
  // resolved once per device and context (a cudaDeviceReset makes a new one)
  static uint32_t* ptrs[kMaxDevices] = {};
  static unsigned long long ctxs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev] || ctxs[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
    ctxs[dev] = ctx;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct Shape {
  int B, H, N, D;
  long long BH() const { return static_cast<long long>(B) * H; }
  int Npad() const { return (N + kTile - 1) / kTile * kTile; }
};

// Sizes only; pointers are checked by each entry point.
fa_status check_shape(const Shape& s, int dtype) {
  if (s.B < 1 || s.H < 1 || s.N < 1) return FA_ERR_INVALID_ARG;
  if (s.D != 64 && s.D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
  if (s.BH() > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (static_cast<double>(s.BH()) * s.N * s.D >= 1099511627776.0) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status check_scale(float scale) { return std::isfinite(scale) ? FA_OK : FA_ERR_INVALID_ARG; }

struct WsLayout {
  size_t lse2 = 0, di = 0, dq = 0, total = 0;
};

WsLayout ws_layout(const Shape& s, int deterministic) {
  WsLayout w;
  const size_t rows = static_cast<size_t>(s.BH()) * s.Npad();
  w.lse2 = 0;
  w.di = round256(rows * 4);
  w.dq = w.di + round256(rows * 4);
  w.total = w.dq + (deterministic ? 0 : round256(static_cast<size_t>(s.BH()) * s.N * s.D * 4));
  return w;
}

fa_status check_ws(const Shape& s, int deterministic, const void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FA_ERR_INVALID_ARG;
  if (bytes < ws_layout(s, deterministic).total) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Element strides of every operand of one call (D contiguous).
struct Layout {
  RowStrides q, k, v, o, dO, dq, dk, dv;
};

Layout contiguous_layout(const Shape& s) {
  const RowStrides c{static_cast<long long>(s.H) * s.N * s.D, static_cast<long long>(s.N) * s.D,
                     static_cast<long long>(s.D)};
  return Layout{c, c, c, c, c, c, c, c};
}

Layout from_abi(const fa_layout& l) {
  auto r = [](const fa_strides& x) { return RowStrides{x.batch, x.head, x.seq}; };
  return Layout{r(l.q), r(l.k), r(l.v), r(l.o), r(l.dO), r(l.dq), r(l.dk), r(l.dv)};
}

// TMA wants 16-byte multiples; every element of the operand must lie below
// 2^40 bytes from its base.
fa_status check_strides(const Shape& s, const RowStrides& r) {
  const long long st[3] = {r.batch, r.head, r.seq};
  for (long long x : st)
    if (x < 0 || (x & 7) != 0) return FA_ERR_INVALID_ARG;
  const double last = static_cast<double>(s.B - 1) * r.batch + static_cast<double>(s.H - 1) * r.head +
                      static_cast<double>(s.N - 1) * r.seq + s.D;
  return last * 2.0 < 1099511627776.0 ? FA_OK : FA_ERR_INVALID_ARG;
}

// The band of visible keys: the window of `opt` (absent when opt is null)
// intersected with the causal mask (right bound 0), and the ALiBi slopes.
fa_status make_band(const fa_options* opt, int causal, const Shape& sh, Band* b) {
  *b = Band{-1, -1, nullptr, 0, nullptr, 0};
  if (opt) {
    if (opt->window_left < -1 || opt->window_right < -1) return FA_ERR_INVALID_ARG;
    if (opt->alibi_slopes && (reinterpret_cast<uintptr_t>(opt->alibi_slopes) & 3u) != 0)
      return FA_ERR_INVALID_ARG;
    b->win_left = opt->window_left;
    b->win_right = opt->window_right;
    b->alibi = opt->alibi_slopes;
    b->alibi_bstride = opt->alibi_per_batch ? sh.H : 0;
    if (opt->block_mask) {
      const long long nt = (sh.N + kTile - 1) / kTile;
      if (nt > kMaxSparseTiles) return FA_ERR_UNSUPPORTED;
      b->block_mask = opt->block_mask;
      b->bm_head_stride = opt->block_mask_per_head ? nt * nt : 0;
    }
  }
  if (causal) b->win_right = 0;  // j <= i, and j <= i + right for any right >= 0
  return FA_OK;
}

bool tile_map(CUtensorMap* m, const void* base, const Shape& s, int dtype, const RowStrides& r,
              int box_rows = kTile) {
  return operand_map(m, base, dtype == FA_BF16, s.B, s.H, s.N, s.D, r.batch, r.head, r.seq,
                     box_rows);
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

constexpr float kLog2e = 1.4426950408889634f;

// Everything the dK/dV and dQ kernels share.
fa_status make_bwd_launch(BwdLaunch* a, const void* q, const void* k, const void* v,
                          const void* dO, void* dq, void* dk, void* dv, const Shape& s,
                          const Layout& L, float scale, const Band& band, int dtype,
                          int deterministic, void* ws) {
  *a = BwdLaunch{};
  if (!tile_map(&a->map_q, q, s, dtype, L.q) || !tile_map(&a->map_k, k, s, dtype, L.k) ||
      !tile_map(&a->map_v, v, s, dtype, L.v) || !tile_map(&a->map_do, dO, s, dtype, L.dO) ||
      !tile_map(&a->map_q64, q, s, dtype, L.q, 64) ||
      !tile_map(&a->map_do64, dO, s, dtype, L.dO, 64) ||
      !tile_map(&a->map_k64, k, s, dtype, L.k, 64) || !tile_map(&a->map_v64, v, s, dtype, L.v, 64))
    return FA_ERR_CUDA;
  if (dq && !tile_map(&a->map_dq, dq, s, dtype, L.dq)) return FA_ERR_CUDA;
  if (dk && !tile_map(&a->map_dk, dk, s, dtype, L.dk)) return FA_ERR_CUDA;
  if (dv && !tile_map(&a->map_dv, dv, s, dtype, L.dv)) return FA_ERR_CUDA;
  const WsLayout w = ws_layout(s, deterministic);
  auto* base = static_cast<uint8_t*>(ws);
  a->lse = reinterpret_cast<const float*>(base + w.lse2);
  a->di = reinterpret_cast<const float*>(base + w.di);
  a->dq_accum = deterministic ? nullptr : reinterpret_cast<float*>(base + w.dq);
  if (a->dq_accum && s.D == 64 &&
      !make_tmap_4d(&a->map_dqacc, a->dq_accum, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    static_cast<uint64_t>(s.D), static_cast<uint64_t>(s.N),
                    static_cast<uint64_t>(s.H), static_cast<uint64_t>(s.B),
                    static_cast<uint64_t>(s.D), static_cast<uint64_t>(s.N) * s.D,
                    static_cast<uint64_t>(s.H) * s.N * s.D, static_cast<uint32_t>(s.D), 64,
                    CU_TENSOR_MAP_SWIZZLE_NONE, 4))
    return FA_ERR_CUDA;
  a->N = s.N;
  a->BH = static_cast<int>(s.BH());
  a->D = s.D;
  a->H = s.H;
  a->scale = scale;
  a->scale_log2 = scale * kLog2e;
  a->band = band;
  a->bf16 = dtype == FA_BF16 ? 1 : 0;
  a->err = error_word_ptr();
  return a->err ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

// The error word for the current device, for entry points in other files.
uint32_t* device_error_word() { return error_word_ptr(); }

}  // namespace fa

using namespace fa;

extern "C" {

int fa_abi_version(void) { return 5; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                   const Shape& s, const Layout& L, float scale, int causal,
                   const fa_options* opt, int dtype, void* stream) {
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  Band band;
  if ((st = make_band(opt, causal, s, &band)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  for (const RowStrides* r : {&L.q, &L.k, &L.v, &L.o})
    if ((st = check_strides(s, *r)) != FA_OK) return st;
  FwdLaunch a{};
  if (!tile_map(&a.map_q, q, s, dtype, L.q) || !tile_map(&a.map_k, k, s, dtype, L.k) ||
      !tile_map(&a.map_v, v, s, dtype, L.v) || !tile_map(&a.map_o, o, s, dtype, L.o))
    return FA_ERR_CUDA;
  a.lse = lse;
  a.N = s.N;
  a.BH = static_cast<int>(s.BH());
  a.D = s.D;
  a.H = s.H;
  a.scale_log2 = scale * kLog2e;
  a.band = band;
  a.bf16 = dtype == FA_BF16 ? 1 : 0;
  a.err = error_word_ptr();
  if (!a.err) return FA_ERR_CUDA;
  return from_cuda(launch_fwd(a, static_cast<cudaStream_t>(stream)));
}

// 8-bit operands: strides in bytes, multiples of 16.
fa_status check_strides_u8(const Shape& s, const RowStrides& r) {
  const long long st[3] = {r.batch, r.head, r.seq};
  for (long long x : st)
    if (x < 0 || (x & 15) != 0) return FA_ERR_INVALID_ARG;
  const double last = static_cast<double>(s.B - 1) * r.batch + static_cast<double>(s.H - 1) * r.head +
                      static_cast<double>(s.N - 1) * r.seq + s.D;
  return last < 1099511627776.0 ? FA_OK : FA_ERR_INVALID_ARG;
}

// Row pitch of the V^T scratch: N rounded up to 16 bytes.
long long vt_pitch(const Shape& s) { return (static_cast<long long>(s.N) + 15) / 16 * 16; }

size_t fwd8_ws_bytes(const Shape& s) {
  return round256(static_cast<size_t>(s.BH()) * s.D * static_cast<size_t>(vt_pitch(s)));
}

bool aligned4_or_null(const float* p) { return !p || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

fa_status fwd8_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                    const Shape& s, const Layout& L, const fa_options* opt,
                    const float* descale_q, const float* descale_k, const float* descale_v,
                    float scale, int causal, void* ws, size_t ws_bytes, void* stream) {
  fa_status st = check_shape(s, FA_BF16);  // D in {64, 128}
  if (st != FA_OK) return st;
  Band band;
  if ((st = make_band(opt, causal, s, &band)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!aligned4_or_null(descale_q) || !aligned4_or_null(descale_k) ||
      !aligned4_or_null(descale_v))
    return FA_ERR_INVALID_ARG;
  for (const RowStrides* r : {&L.q, &L.k, &L.v})
    if ((st = check_strides_u8(s, *r)) != FA_OK) return st;
  if ((st = check_strides(s, L.o)) != FA_OK) return st;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < fwd8_ws_bytes(s))
    return FA_ERR_INVALID_ARG;
  const long long ld = vt_pitch(s);
  FwdLaunch a{};
  if (!operand_map_u8(&a.map_q, q, s.B, s.H, s.N, s.D, L.q.batch, L.q.head, L.q.seq, kTile) ||
      !operand_map_u8(&a.map_k, k, s.B, s.H, s.N, s.D, L.k.batch, L.k.head, L.k.seq, kTile) ||
      !make_tmap_4d(&a.map_v, ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(s.N),
                    static_cast<uint64_t>(s.D), static_cast<uint64_t>(s.H),
                    static_cast<uint64_t>(s.B), static_cast<uint64_t>(ld),
                    static_cast<uint64_t>(ld) * s.D, static_cast<uint64_t>(ld) * s.D * s.H, 128,
                    static_cast<uint32_t>(s.D), CU_TENSOR_MAP_SWIZZLE_128B, 1) ||
      !tile_map(&a.map_o, o, s, FA_BF16, L.o))
    return FA_ERR_CUDA;
  a.lse = lse;
  a.N = s.N;
  a.BH = static_cast<int>(s.BH());
  a.D = s.D;
  a.H = s.H;
  a.scale_log2 = scale * kLog2e;
  a.band = band;
  a.bf16 = 1;
  a.fp8 = 1;
  a.descale_q = descale_q;
  a.descale_k = descale_k;
  a.descale_v = descale_v;
  a.err = error_word_ptr();
  if (!a.err) return FA_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_transpose_v8(v, L.v, ws, s.N, ld, s.H, s.BH(), s.D, cs);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return from_cuda(launch_fwd(a, cs));
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, const Shape& s, const Layout& L,
                   float scale, int causal, const fa_options* opt, int dtype, int deterministic,
                   void* workspace, size_t workspace_bytes, void* stream) {
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  Band band;
  if ((st = make_band(opt, causal, s, &band)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  for (const RowStrides* r : {&L.q, &L.k, &L.v, &L.o, &L.dO, &L.dq, &L.dk, &L.dv})
    if ((st = check_strides(s, *r)) != FA_OK) return st;
  if ((st = check_ws(s, deterministic, workspace, workspace_bytes)) != FA_OK) return st;
  // Build every descriptor before enqueueing anything.
  BwdLaunch a;
  if ((st = make_bwd_launch(&a, q, k, v, dO, dq, dk, dv, s, L, scale, band, dtype,
                            deterministic, workspace)) != FA_OK)
    return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const WsLayout w = ws_layout(s, deterministic);
  auto* base = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_bwd_preprocess(o, L.o, dO, L.dO, lse,
                                        reinterpret_cast<float*>(base + w.lse2),
                                        reinterpret_cast<float*>(base + w.di), a.dq_accum, s.N,
                                        s.H, s.BH(), s.D, dtype == FA_BF16, cs);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if ((e = launch_bwd_dkdv(a, cs)) != cudaSuccess) return FA_ERR_CUDA;
  if (deterministic) return from_cuda(launch_bwd_dq(a, cs));
  return from_cuda(launch_dq_convert(a.dq_accum, dq, L.dq, s.N, s.H, s.BH(), s.D, scale,
                                     dtype == FA_BF16, cs));
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int D, float scale, int causal, fa_dtype dtype, void* stream) {
  const Shape s{B, H, N, D};
  return fwd_impl(q, k, v, o, lse, s, contiguous_layout(s), scale, causal, nullptr, dtype,
                  stream);
}

fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int D, const fa_layout* layout, float scale, int causal,
                         fa_dtype dtype, void* stream) {
  if (!layout) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, Shape{B, H, N, D}, from_abi(*layout), scale, causal, nullptr,
                  dtype, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int N, int D, const fa_layout* layout, const fa_options* options,
                    float scale, int causal, fa_dtype dtype, void* stream) {
  const Shape s{B, H, N, D};
  return fwd_impl(q, k, v, o, lse, s, layout ? from_abi(*layout) : contiguous_layout(s), scale,
                  causal, options, dtype, stream);
}

size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int D) {
  const Shape s{B, H, N, D};
  if (check_shape(s, FA_BF16) != FA_OK) return 0;
  return fwd8_ws_bytes(s);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int D, const fa_layout* layout, const fa_options* options,
                     const float* descale_q, const float* descale_k, const float* descale_v,
                     float scale, int causal, void* workspace, size_t workspace_bytes,
                     void* stream) {
  const Shape s{B, H, N, D};
  return fwd8_impl(q, k, v, o, lse, s, layout ? from_abi(*layout) : contiguous_layout(s),
                   options, descale_q, descale_k, descale_v, scale, causal, workspace,
                   workspace_bytes, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int D, int deterministic) {
  const Shape s{B, H, N, D};
  if (check_shape(s, FA_BF16) != FA_OK) return 0;
  return ws_layout(s, deterministic).total;
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int H, int N,
                            int D, fa_dtype dtype, int deterministic, void* workspace,
                            size_t workspace_bytes, void* stream) {
  const Shape s{B, H, N, D};
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  if ((st = check_ws(s, deterministic, workspace, workspace_bytes)) != FA_OK) return st;
  const WsLayout w = ws_layout(s, deterministic);
  auto* base = static_cast<uint8_t*>(workspace);
  const Layout L = contiguous_layout(s);
  return from_cuda(launch_bwd_preprocess(
      o, L.o, dO, L.dO, lse, reinterpret_cast<float*>(base + w.lse2),
      reinterpret_cast<float*>(base + w.di),
      deterministic ? nullptr : reinterpret_cast<float*>(base + w.dq), N, H, s.BH(), D,
      dtype == FA_BF16, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                      void* dv, int B, int H, int N, int D, float scale, int causal,
                      fa_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                      void* stream) {
  const Shape s{B, H, N, D};
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) ||
      !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if ((st = check_ws(s, deterministic, workspace, workspace_bytes)) != FA_OK) return st;
  BwdLaunch a;
  Band band;
  if ((st = make_band(nullptr, causal, s, &band)) != FA_OK) return st;
  if ((st = make_bwd_launch(&a, q, k, v, dO, nullptr, dk, dv, s, contiguous_layout(s), scale,
                            band, dtype, deterministic, workspace)) != FA_OK)
    return st;
  return from_cuda(launch_bwd_dkdv(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B,
                    int H, int N, int D, float scale, int causal, fa_dtype dtype, void* workspace,
                    size_t workspace_bytes, void* stream) {
  const Shape s{B, H, N, D};
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq))
    return FA_ERR_INVALID_ARG;
  if ((st = check_ws(s, 1, workspace, workspace_bytes)) != FA_OK) return st;
  BwdLaunch a;
  Band band;
  if ((st = make_band(nullptr, causal, s, &band)) != FA_OK) return st;
  if ((st = make_bwd_launch(&a, q, k, v, dO, dq, nullptr, nullptr, s, contiguous_layout(s),
                            scale, band, dtype, 1, workspace)) != FA_OK)
    return st;
  return from_cuda(launch_bwd_dq(a, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd_dq_convert(void* dq, int B, int H, int N, int D, float scale, fa_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream) {
  const Shape s{B, H, N, D};
  fa_status st = check_shape(s, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(dq)) return FA_ERR_INVALID_ARG;
  if ((st = check_ws(s, 0, workspace, workspace_bytes)) != FA_OK) return st;
  const WsLayout w = ws_layout(s, 0);
  const float* acc = reinterpret_cast<const float*>(static_cast<uint8_t*>(workspace) + w.dq);
  return from_cuda(launch_dq_convert(acc, dq, contiguous_layout(s).dq, N, H, s.BH(), D, scale,
                                     dtype == FA_BF16, static_cast<cudaStream_t>(stream)));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                 float scale, int causal, fa_dtype dtype, int deterministic, void* workspace,
                 size_t workspace_bytes, void* stream) {
  const Shape s{B, H, N, D};
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, s, contiguous_layout(s), scale, causal,
                  nullptr, dtype, deterministic, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int D, const fa_layout* layout, float scale, int causal,
                         fa_dtype dtype, int deterministic, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!layout) return FA_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, Shape{B, H, N, D}, from_abi(*layout), scale,
                  causal, nullptr, dtype, deterministic, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                    const fa_layout* layout, const fa_options* options, float scale, int causal,
                    fa_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                    void* stream) {
  const Shape s{B, H, N, D};
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, s,
                  layout ? from_abi(*layout) : contiguous_layout(s), scale, causal, options, dtype,
                  deterministic, workspace, workspace_bytes, stream);
}

fa_status fa_device_error(void* stream, int* code) {
  if (!code) return FA_ERR_INVALID_ARG;
  uint32_t* p = error_word_ptr();
  if (!p) return FA_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  *code = v == 0 ? FA_OK : FA_ERR_TIMEOUT;
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 2000000) return FA_ERR_INVALID_ARG;
  uint32_t* p = error_word_ptr();
  if (!p) return FA_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (launch_wait_selftest(p, static_cast<uint64_t>(limit_us) * 1000ull, cs) != cudaSuccess)
    return FA_ERR_CUDA;
  int code = FA_OK;
  fa_status st = fa_device_error(stream, &code);
  if (st != FA_OK) return st;
  return static_cast<fa_status>(code);
}

}  // extern "C"
