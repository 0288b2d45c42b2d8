// fa_fwd.cu -- exact attention forward for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, head), walking the
// key/value tiles with an online softmax ("FlashAttention from scratch"
// walkthrough, l189.com, sec. 2.2 and 2.4; "FlashAttention 深入", online
// softmax).  Parallelism is over query tiles as well as (batch, head), the
// sequence-dimension split of FlashAttention-2 ("FlashAttention 深入", v2).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (= TMEM lane t).  Reads S
//              from TMEM, keeps the running max m and sum l in fp32
//              (walkthrough sec. 5.2), writes P as 16-bit pairs back into the
//              same TMEM columns, rescales O in TMEM when m grows, and runs
//              the epilogue (O / l through a swizzled smem tile and a TMA
//              store; LSE = ln 2 * (m + log2 l)).
//   warp 4     TMA producer: Q once, K and V tiles into two smem stages.
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S
//              buffers, then O += P_{j-1} V_{j-1} with P read from TMEM.
//              S_{j+1} is issued before PV_j so the tensor core computes the
//              next scores while the softmax warps work on the current ones.
//
// TMEM columns: [0,128) S/P buffer 0, [128,256) S/P buffer 1, [256,256+D) O,
// [256+D, 256+3D/2) Q.  The tensor core reads its operands from shared memory
// at roughly 64 bytes per clock, so every product keeps its A operand in TMEM
// (Q for S = Q K^T, P for O += P V) and reads only B (K or V) from shared
// memory: one 4 KB B slice per 64-cycle instruction keeps it fed.
//
// Softmax bookkeeping works in log2 units: scores are multiplied by
// scale*log2(e) and exponentiated with ex2.  The reference maximum m is only
// moved when the tile maximum exceeds it by more than 8 (a factor of 256);
// P then stays below 256, and O / l and the LSE are unchanged because both
// use the same m.  Rows whose maximum barely moves never touch O in TMEM.
//
// Causal mask (walkthrough sec. 5.3): query i sees keys j <= i.  Key tiles
// past the diagonal are never loaded; the diagonal tile and a ragged last
// tile are masked element-wise.  Within a head, the longest query tiles go first.
#include <climits>

#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kFwdThreads = 192;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdSmem {
  static constexpr int kBlocks = D / 64;             // 64-element column blocks
  static constexpr int kBlockBytes = kTile * 128;    // 128 rows x 128 B
  static constexpr int kTileBytes = kBlocks * kBlockBytes;
  alignas(1024) uint8_t q[kTileBytes];  // reused as the O staging tile
  alignas(1024) uint8_t k[2][kTileBytes];
  alignas(1024) uint8_t v[2][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, drain, qt_full;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort_flag) {
  bool ok = mbar_wait(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kFwdThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdLaunch p) {
  using Smem = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int n_q_tiles = (p.N + kTile - 1) / kTile;
  // Head-major order, so that the CTAs in flight share one head's K and V in
  // L2; under the causal mask the longest query tiles of a head go first.
  const int bh = static_cast<int>(blockIdx.x / n_q_tiles);
  const int qt = kCausal ? n_q_tiles - 1 - static_cast<int>(blockIdx.x % n_q_tiles)
                         : static_cast<int>(blockIdx.x % n_q_tiles);
  const int q0 = qt * kTile;
  const int n_kv = (p.N + kTile - 1) / kTile;
  const int n_tiles = kCausal ? min(n_kv, qt + 1) : n_kv;

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    mbar_init(&s.o_done, 1);
    mbar_init(&s.drain, 1);
    mbar_init(&s.qt_full, 128);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t tO = tbase + 256;
  const uint32_t tQ = tbase + 256 + D;  // Q as the A operand of S = Q K^T (D/2 columns)
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.map_q);
      tma_prefetch_desc(&p.map_k);
      tma_prefetch_desc(&p.map_v);
      mbar_arrive_expect_tx(&s.q_full, Smem::kTileBytes);
      for (int kb = 0; kb < Smem::kBlocks; ++kb)
        tma_load_3d(s.q + kb * Smem::kBlockBytes, &p.map_q, &s.q_full, kb * 64, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t u = static_cast<uint32_t>(j >> 1);
        if (j >= 2 && !mbar_wait(&s.k_empty[st], (u - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(&s.k_full[st], Smem::kTileBytes);
        for (int kb = 0; kb < Smem::kBlocks; ++kb)
          tma_load_3d(s.k[st] + kb * Smem::kBlockBytes, &p.map_k, &s.k_full[st], kb * 64,
                      j * kTile, bh);
        if (j >= 2 && !mbar_wait(&s.v_empty[st], (u - 1) & 1, p.err, abort_flag)) {
          issued = j * 2 + 1;
          break;
        }
        mbar_arrive_expect_tx(&s.v_full[st], Smem::kTileBytes);
        for (int kb = 0; kb < Smem::kBlocks; ++kb)
          tma_load_3d(s.v[st] + kb * Smem::kBlockBytes, &p.map_v, &s.v_full[st], kb * 64,
                      j * kTile, bh);
        issued = j * 2 + 2;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's smem goes away.
        int zero = 0;
        mbar_wait(&s.q_full, 0, p.err, &zero, 100000000ull);
        for (int t = max(0, issued - 4); t < issued; ++t) {
          const int j = t >> 1, st = j & 1;
          mbar_wait((t & 1) ? &s.v_full[st] : &s.k_full[st], (j >> 1) & 1, p.err, &zero,
                    100000000ull);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ab = kBf16 ? 1u : 0u;
      constexpr uint32_t idS = idesc_f16(128, 128, ab, 0, 0);
      constexpr uint32_t idPV = idesc_f16(128, D, ab, 0, 1);
      // Operand descriptors are built once and advanced by constant offsets.
      const uint64_t dk0 = smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(s.v[0]), Smem::kBlockBytes, 1024);
      bool ok = mbar_wait(&s.qt_full, 0, p.err, abort_flag);
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int st = j & 1;
          const uint32_t u = static_cast<uint32_t>(j >> 1);
          if (!mbar_wait(&s.k_full[st], u & 1, p.err, abort_flag)) break;
          tc_fence_after();
          const uint64_t dk = desc_add(dk0, st * Smem::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Smem::kBlockBytes + (kk & 3) * 32;
            tc_mma_ts(tbase + st * 128, tQ + kk * 8, desc_add(dk, off), idS, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s.s_full[st]);
          tc_commit(&s.k_empty[st]);
        }
        if (j >= 1) {
          const int jj = j - 1, st = jj & 1;
          const uint32_t u = static_cast<uint32_t>(jj >> 1);
          if (!mbar_wait(&s.p_full[st], u & 1, p.err, abort_flag)) break;
          if (!mbar_wait(&s.v_full[st], u & 1, p.err, abort_flag)) break;
          tc_fence_after();
          const uint64_t dv = desc_add(dv0, st * Smem::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            tc_mma_ts(tO, tbase + st * 128 + kk * 8, desc_add(dv, kk * 16 * 128), idPV,
                      (jj > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&s.o_done);
          tc_commit(&s.v_empty[st]);
        }
      }
      // Every MMA issued above completes before TMEM is released.
      tc_commit(&s.drain);
      int zero = 0;
      mbar_wait(&s.drain, 0, p.err, &zero, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // row within the tile and TMEM lane
    const int i = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    float m = -INFINITY;  // reference maximum, log2 units
    float l = 0.f;        // running sum of 2^(t - m)
    // Q into TMEM, so that S = Q K^T reads only K from shared memory: thread
    // r moves row r out of the swizzled tile (16-byte chunk c of a 128-byte
    // row sits at chunk c ^ (r & 7)); the 16-bit pairs keep their order.
    bool ok = warp_wait(&s.q_full, 0, p.err, abort_flag);
    if (ok) {
#pragma unroll
      for (int kb = 0; kb < Smem::kBlocks; ++kb) {
        uint32_t w[32];
        const uint8_t* row = s.q + kb * Smem::kBlockBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) * 16));
          w[c * 4] = v.x;
          w[c * 4 + 1] = v.y;
          w[c * 4 + 2] = v.z;
          w[c * 4 + 3] = v.w;
        }
        tmem_st32(tQ + lane_off + kb * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.qt_full);
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int st = j & 1;
      const uint32_t u = static_cast<uint32_t>(j >> 1);
      if (!warp_wait(&s.s_full[st], u & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kTile];
      {
        // All four loads in flight before the single wait.
        uint32_t raw[kTile / 32][32];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tbase + lane_off + st * 128 + c * 32, raw[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
#pragma unroll
          for (int t = 0; t < 32; ++t) sv[c * 32 + t] = __uint_as_float(raw[c][t]);
      }
      // Scores -> log2 units.  With a positive scale this is folded into the
      // exponent below (one FFMA per score); otherwise scale first.
      if (!pos_scale) {
#pragma unroll
        for (int c = 0; c < kTile; ++c) sv[c] *= sl2;
      }
      const int k0 = j * kTile;
      const bool diag = kCausal && (k0 + kTile - 1 > q0);
      if (diag || k0 + kTile > p.N) {
        const int last = (kCausal ? min(i, p.N - 1) : p.N - 1) - k0;  // last visible column
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (c > last) sv[c] = -INFINITY;
      }
      // Row maximum with eight independent chains (short dependency depth).
      float mxs[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mxs[t] = sv[t];
#pragma unroll
      for (int c = 8; c < kTile; c += 8)
#pragma unroll
        for (int t = 0; t < 8; ++t) mxs[t] = fmaxf(mxs[t], sv[c + t]);
      const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                             fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
      const float m_tile = pos_scale ? mx * sl2 : mx;
      const float m_new = fmaxf(m, m_tile);
      const bool need = m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
        l *= alpha;
        m = m_new;
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O currently holds sum_{j' < j} P V; it must be final before scaling.
        if (!warp_wait(&s.o_done, (j - 1) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
          tmem_st32(tO + lane_off + c * 32, o);
        }
      }
      const float mneg = (m == -INFINITY) ? 0.f : -m;
      float sums[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial row sums
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x0 = sv[h * 64 + 2 * c], x1 = sv[h * 64 + 2 * c + 1];
          const float p0 = ex2_approx(pos_scale ? fmaf(x0, sl2, mneg) : x0 + mneg);
          const float p1 = ex2_approx(pos_scale ? fmaf(x1, sl2, mneg) : x1 + mneg);
          sums[(c & 1) * 2] += p0;
          sums[(c & 1) * 2 + 1] += p1;
          pk[c] = pack2<kBf16>(p0, p1);
        }
        tmem_st32(tbase + lane_off + st * 128 + h * 32, pk);
      }
      l += (sums[0] + sums[1]) + (sums[2] + sums[3]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[st]);
    }

    // ---------------------------------------------------------- epilogue
    // Every softmax thread takes the same branch (a timeout in one warp must
    // not leave the others waiting at the barrier below).
    const bool mine = ok && warp_wait(&s.o_done, (n_tiles - 1) & 1, p.err, abort_flag);
    if (named_bar_and(1, 128, mine)) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack2<kBf16>(__uint_as_float(o[2 * t]) * inv_l,
                               __uint_as_float(o[2 * t + 1]) * inv_l);
        // 32 columns = four 16-byte chunks of this row, 128-byte swizzle
        uint8_t* blk = s.q + (c >> 1) * Smem::kBlockBytes + r * 128;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int cc = (c & 1) * 4 + ch;
          *reinterpret_cast<uint4*>(blk + ((cc ^ (r & 7)) * 16)) =
              make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (tid == 0) {
        for (int kb = 0; kb < Smem::kBlocks; ++kb)
          tma_store_3d(&p.map_o, s.q + kb * Smem::kBlockBytes, kb * 64, q0, bh);
        tma_store_commit();
        tma_store_wait_all();
      }
      if (i < p.N) p.lse[static_cast<long long>(bh) * p.N + i] = (m + lg2_approx(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, kBf16, kCausal>;
  const int smem = static_cast<int>(sizeof(FwdSmem<D>)) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long n_q_tiles = (a.N + kTile - 1) / kTile;
  const long long grid = n_q_tiles * a.BH;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(grid), kFwdThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s) {
  if (a.D == 64) {
    if (a.bf16) return a.causal ? launch_fwd_t<64, true, true>(a, s) : launch_fwd_t<64, true, false>(a, s);
    return a.causal ? launch_fwd_t<64, false, true>(a, s) : launch_fwd_t<64, false, false>(a, s);
  }
  if (a.bf16) return a.causal ? launch_fwd_t<128, true, true>(a, s) : launch_fwd_t<128, true, false>(a, s);
  return a.causal ? launch_fwd_t<128, false, true>(a, s) : launch_fwd_t<128, false, false>(a, s);
}

}  // namespace fa
