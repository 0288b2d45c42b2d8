// fa_bwd.cu -- exact attention backward for sm_103a: recompute P from Q, K
// and the forward's log-sum-exp instead of storing it ("FlashAttention from
// scratch" walkthrough, l189.com, sec. 3.3; "FlashAttention 深入", backward
// recomputation).
//
//   preprocess  Di = rowsum(dO * O) (fp32), the full-row statistic of the
//               softmax Jacobian; LSE rescaled to log2 units; both padded to
//               whole 128-row tiles (+inf / 0) so the tile kernels can copy
//               them with one bulk copy.  Also zeroes the fp32 dQ accumulator.
//   dkdv        one CTA per 128-key tile, software-pipelined over 64-row
//               query tiles (D = 64 or 128):
//                 S^T  = K Q^T            (TMEM)      P^T = exp2(S^T*c - lse2)
//                 dP^T = V dO^T           (TMEM)      dS^T = P^T (dP^T - Di)
//                 dV  += P^T dO           (A = P^T packed into TMEM)
//                 dK  += dS^T Q           (A = dS^T packed into TMEM)
//                 dQ^T = K^T dS^T         (atomic mode, into TMEM; drained
//                                          with fp32 atomics)
//   dq          deterministic mode: one CTA per 128-query tile looping over
//               key tiles, dQ accumulated in TMEM, no atomics.
//   dq_convert  dQ = scale * accumulator, rounded to the input type.
//
// Every wait is bounded.
#include <climits>

#include "fa_band.cuh"
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort_flag) {
  bool ok = mbar_wait(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Write 32 consecutive 16-bit values (16 packed words) of tile row r,
// columns [32*c32, 32*c32 + 32), into a 128-byte-swizzled tile made of
// 64-column blocks of 128 rows.
__device__ __forceinline__ void store_row_chunk_sw128(uint8_t* tile, int r, int c32,
                                                      const uint32_t (&pk)[16]) {
  uint8_t* row = tile + (c32 >> 1) * (kTile * 128) + r * 128;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    const int cc = (c32 & 1) * 4 + ch;
    *reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) * 16)) =
        make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
  }
}

// ---------------------------------------------------------------------------
// preprocess
// ---------------------------------------------------------------------------
// One group of D/8 threads per row; each thread handles 8 columns.
template <int D, bool kBf16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                             RowStrides so,
                                                             const uint16_t* __restrict__ dO,
                                                             RowStrides sdo,
                                                             const float* __restrict__ lse,
                                                             float* __restrict__ lse2,
                                                             float* __restrict__ di,
                                                             float* __restrict__ dq_accum, int N,
                                                             int Npad, int H, long long BH) {
  pdl_wait();
  constexpr int G = D / 8;  // threads per row
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long prow = gtid / G;  // padded row index over BH * Npad
  const int part = static_cast<int>(gtid % G);
  if (prow >= BH * Npad) return;
  const long long bh = prow / Npad;
  const int n = static_cast<int>(prow % Npad);
  float acc = 0.f;
  if (n < N) {
    const long long b = bh / H, h = bh % H;
    const long long row = bh * N + n;
    const uint4 a = *reinterpret_cast<const uint4*>(o + b * so.batch + h * so.head + n * so.seq +
                                                    part * 8);
    const uint4 g = *reinterpret_cast<const uint4*>(dO + b * sdo.batch + h * sdo.head +
                                                    n * sdo.seq + part * 8);
    const uint32_t* aa = reinterpret_cast<const uint32_t*>(&a);
    const uint32_t* gg = reinterpret_cast<const uint32_t*>(&g);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 x = unpack2<kBf16>(aa[t]), y = unpack2<kBf16>(gg[t]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    if (dq_accum) {
      float4* z = reinterpret_cast<float4*>(dq_accum + row * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, G);
  if (part == 0) {
    di[prow] = acc;
    lse2[prow] = (n < N) ? lse[bh * N + n] * kLog2e : INFINITY;
  }
}

// ---------------------------------------------------------------------------
// dK / dV, software-pipelined over 64-row query tiles (D = 64 or 128)
// ---------------------------------------------------------------------------
// With 64-row query tiles the scores and their gradient take 64 TMEM columns
// each, so NB tiles' S^T / dP^T fit beside the dV and dK accumulators (NB = 2
// at D = 128, 3 at D = 64):
//   TMEM [128b, 128b + 64)       buffer b: S^T of tile i (b = i % NB), then
//                                dQ^T of tile i - 1 once S^T is consumed
//   TMEM [128b + 64, 128b + 128) buffer b: dP^T of tile i; then, for each
//                                32-query half, P^T and dS^T packed over it
//   TMEM [128 NB, 128 NB + D) dV, [128 NB + D, 128 NB + 2D) dK
// Two warps issue the products, each running its loop with all 32 lanes (the
// operands stay warp-uniform) while one elected lane issues every product
// and commit.  The score warp issues S^T, dP^T(i) as soon
// as buffer i % NB is free; the gradient warp, once tile i's P^T / dS^T are
// in TMEM, issues dQ^T(i-1) and then dV, dK(i).  Any stall of an issuing
// thread (even a wait on a barrier that has already completed) leaves the
// tensor core idle for a few hundred cycles while its next products travel
// to it; with two issuers the other one's queued products fill that gap.
// dQ^T(i-1) takes the S^T columns of tile i once those are consumed; the
// four dQ warps drain it before S^T(i+2) reuses the buffer.  Q / dO (with
// their LSE / Di rows) come through a three-stage ring, dS^T for dQ through
// a three-stage shared buffer; eight warps do the elementwise work.  dV and
// dK take their A operands (P^T, dS^T) from TMEM, so they read only dO or Q
// from shared memory; the score and dQ^T products read both operands from
// shared memory, which bounds them at 48 cycles per 128 x 64 x 16 product.
// dQ is formed transposed, dQ^T = K^T dS^T (M = D), so TMEM lane = column d
// and each atomic warp instruction covers 32 consecutive floats of one dQ row.
// At D = 64 the dQ^T product still runs with M = 128: output row m depends
// only on A row m, so rows 64..127 (read past K's tile in shared memory) are
// computed and never drained.
// Warps 0-7 elementwise, 8-11 buffer / dQ, 12 producer, 13-14 MMA (and at
// D = 64 an idle warp 15).  At D = 64 the launch reserves 128 registers a
// thread for 16 warps (four share each SM sub-partition's 16384); warpgroup
// 3 (warps 12-15) keeps kPipeLowRegs and the elementwise warpgroups take
// kPipeHighRegs: 256 x 144 + 128 x 128 + 128 x 88 = 64512 of the 65536
// reserved, 32 x (144 + 144 + 128 + 88) = 16128 on each sub-partition.  (At
// D = 128 the same split made the kernel slower.)
template <int D>
constexpr int kPipeThreads = D == 64 ? 512 : 480;
constexpr uint32_t kPipeLowRegs = 88, kPipeHighRegs = 144;
constexpr int kQ64 = 64;

template <int D, bool kSparse, bool kResident>
struct DkdvPipeSmem {
  // TMEM buffers for S^T / dP^T: as many as fit beside dV and dK (D = 64:
  // 3 x 128 + 2 x 64 = 512 columns; D = 128: 2 x 128 + 2 x 128)
  static constexpr int kBufs = D == 64 ? 3 : 2;
  // Q / dO stages: one more than the buffers, so that a tile's loads start
  // before the buffer it will use is free
  static constexpr int kQStages = kBufs + 1;
  // K / V buffers: a resident CTA loads its next key tile's while this one runs
  static constexpr int kKVBufs = kResident ? 2 : 1;
  static constexpr int kDBlocks = D / 64;      // 64-column blocks of a row
  static constexpr int kKBlock = kTile * 128;  // 128 rows x 128 B
  static constexpr int kQBlock = kQ64 * 128;   // 64 rows x 128 B
  alignas(1024) uint8_t k[kKVBufs][kDBlocks * kKBlock];  // [buffer][D block][128 keys][64 d]
  alignas(1024) uint8_t v[kKVBufs][kDBlocks * kKBlock];
  alignas(1024) uint8_t q[kQStages][kDBlocks * kQBlock];  // [stage][D block][64 queries][64 d]
  alignas(1024) uint8_t dO[kQStages][kDBlocks * kQBlock];
  alignas(1024) uint8_t dst[3][kKBlock];       // [tile % 3][128 keys][64 queries]
  alignas(16) float lse2[kQStages][kQ64];
  alignas(16) float di[kQStages][kQ64];
  // D = 64, atomic mode: drained dQ tiles [64 queries][D] for the bulk
  // reductions, double-buffered
  alignas(1024) float dq_stage[D == 64 ? 2 : 1][D == 64 ? kQ64 * D : 1];
  uint64_t kv_full[kKVBufs], kv_empty[kKVBufs];
  uint64_t qdo_full[kQStages], qdo_empty[kQStages], s_full[kBufs], s_read[kBufs], p_full[kBufs];
  uint64_t buf_ready[kBufs];
  uint64_t dq_full[3], tmem_free[kBufs], ds_last, acc_full, epi_read, drain[2];
  uint64_t last_issued;  // resident: a unit's last dV, dK issued
  uint64_t stage_full[2], stage_free[2];
  uint32_t tmem_base;
  int abort_flag;
  uint32_t q_tiles[kSparse ? 2 * kMaxSparseTiles / 32 : 1];  // block-sparse: 64-row query tiles
};

template <int D, bool kBf16, bool kAlibi, bool kAtomicDq, bool kSparse, bool kResident>
__global__ void __launch_bounds__(kPipeThreads<D>, 1)
    bwd_dkdv_pipe_kernel(const __grid_constant__ BwdLaunch p) {
  static_assert(!kResident || (D == 64 && !kSparse),
                "resident CTAs: D = 64 (two K / V buffers fit) and dense bands");
  pdl_wait();
  using Smem = DkdvPipeSmem<D, kSparse, kResident>;
  constexpr int kDB = Smem::kDBlocks;
  constexpr int kNB = Smem::kBufs;     // S^T / dP^T buffers: tile gi uses buffer gi % kNB
  constexpr int kQS = Smem::kQStages;  // Q / dO stages: tile gi uses stage gi % kQS
  constexpr int kKVB = Smem::kKVBufs;  // K / V buffers: unit k uses buffer k % kKVB
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_kt = (p.N + kTile - 1) / kTile;
  const int Npad = n_kt * kTile;
  const int n_q64 = (p.N + kQ64 - 1) / kQ64;
  const long long n_units = static_cast<long long>(n_kt) * p.BH;
  const int wl = p.band.win_left, wr = p.band.win_right;
  // A unit is one key tile of one (batch, head).  Head-major order, longest
  // key tiles first within a head: the CTAs in flight share one head's Q, dO
  // and dQ accumulator in L2 (tile-major instead when the streamed operands
  // all fit in L2).  A CTA of the grid takes unit blockIdx.x; a resident
  // CTA c of G takes units k G + c (k even) and k G + G - 1 - c (k odd).
  auto unit_of = [&](int k) -> long long {
    if constexpr (!kResident) return blockIdx.x;
    const long long G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
  };
  auto has_unit = [&](int k) { return kResident ? unit_of(k) < n_units : k == 0; };
  struct Unit {
    int bh, hh, bb, k0;  // slice, its TMA coordinates (head, batch), first key
    int first, last;     // 64-row query tiles whose band reaches the key tile
  };
  // (32-bit division when the unit count allows: a 64-bit one is a long
  // instruction sequence, and every role decodes each unit.  Not in the
  // atomic-dQ kernel with one unit per CTA: it decodes once per role, and
  // with this path its compiled loops measured 30 % slower at D = 128.)
  const bool units32 = (kResident || !kAtomicDq) && n_units <= 0xffffffffLL;
  auto decode = [&](long long u) {
    Unit w;
    if (units32) {
      const uint32_t u32 = static_cast<uint32_t>(u);
      const uint32_t d = static_cast<uint32_t>(p.tile_major ? p.BH : n_kt);
      const uint32_t q = u32 / d, r = u32 - q * d;
      w.bh = static_cast<int>(p.tile_major ? r : q);
      w.k0 = static_cast<int>(p.tile_major ? q : r) * kTile;
    } else {
      w.bh = static_cast<int>(p.tile_major ? u % p.BH : u / n_kt);
      w.k0 = static_cast<int>(p.tile_major ? u / p.BH : u % n_kt) * kTile;
    }
    w.hh = w.bh % p.H;
    w.bb = w.bh / p.H;
    band_query_tiles(w.k0, kTile, kQ64, n_q64, wl, wr, w.first, w.last);
    return w;
  };
  auto walk_of = [&](const Unit& w) {
    return TileWalk<kSparse>{w.first, w.last, n_q64, TileSet{s.q_tiles, n_q64}};
  };
  // fn(k, unit, walk) for this CTA's units in turn, while it returns true.
  // Each role numbers the tiles of all its units in one sequence (gi) and
  // every ring and buffer below is indexed by it.  A dense band reaches
  // every key tile from at least one query tile (the tile holding the
  // tile's first key), so a resident CTA's units are never empty.
  auto for_each_unit = [&](auto&& fn) {
    for (int k = 0; has_unit(k); ++k) {
      const Unit w = decode(unit_of(k));
      if (!fn(k, w, walk_of(w))) return false;
    }
    return true;
  };
  if constexpr (kSparse) {  // the mask's 128-row blocks hold 64-row tiles 2b, 2b + 1
    const Unit w = decode(blockIdx.x);
    fill_tile_set(s.q_tiles, n_q64, [&](int it) {
      return it >= w.first && it <= w.last &&
             block_kept(p.band, w.bh, p.H, n_kt, it >> 1, w.k0 / kTile);
    });
  }
  __syncthreads();

  if (tid == 0) {
    for (int i = 0; i < kKVB; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < kQS; ++i) {
      mbar_init(&s.qdo_full[i], 1);
      mbar_init(&s.qdo_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&s.dq_full[i], 1);
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 256);
      mbar_init(&s.s_read[i], 8);  // one arrival per elementwise warp
      // four buffer warps and the tcgen05.commit that retires dV, dK(gi - kNB)
      mbar_init(&s.buf_ready[i], 5);
      mbar_init(&s.tmem_free[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.drain[i], 1);
      mbar_init(&s.stage_full[i], 2);  // the two buffer warps holding dQ rows d < 64
      mbar_init(&s.stage_free[i], 1);  // the thread that issues the reductions
    }
    mbar_init(&s.ds_last, 256);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.epi_read, 1);
    mbar_init(&s.last_issued, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 12) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t tdV = tbase + kNB * 128, tdK = tdV + D;
  volatile int* abort_flag = &s.abort_flag;
  constexpr uint32_t ab = kBf16 ? 1u : 0u;

  if (warp >= 12) {
    // D = 64: the producer and MMA warps give registers to the elementwise
    // warpgroups (warp 15 only does this)
    if constexpr (D == 64) setmaxnreg_dec<kPipeLowRegs>();
    if (warp == 12) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int kv_loads = 0, issued = 0;  // units whose K / V, tiles whose Q / dO were requested
        int gi = 0;
        for_each_unit([&](int k, const Unit& w, const TileWalk<kSparse>& walk) -> bool {
          const int kvb = k % kKVB;
          // buffer kvb was last read by the products of unit k - kKVB
          if (k >= kKVB && !mbar_wait(&s.kv_empty[kvb], ((k - kKVB) / kKVB) & 1, p.err, abort_flag))
            return false;
          mbar_arrive_expect_tx(&s.kv_full[kvb], 2 * kDB * Smem::kKBlock);
          for (int kb = 0; kb < kDB; ++kb) {
            tma_load_4d(s.k[kvb] + kb * Smem::kKBlock, &p.map_k, &s.kv_full[kvb], kb * 64, w.k0,
                        w.hh, w.bb);
            tma_load_4d(s.v[kvb] + kb * Smem::kKBlock, &p.map_v, &s.kv_full[kvb], kb * 64, w.k0,
                        w.hh, w.bb);
          }
          kv_loads = k + 1;
          const int n = walk.count();
          for (int i = 0, qt = walk.first(); i < n; ++i, qt = walk.next(qt), ++gi) {
            const int st = gi % kQS;
            if (gi >= kQS &&
                !mbar_wait(&s.qdo_empty[st], ((gi - kQS) / kQS) & 1, p.err, abort_flag))
              return false;
            // Atomic mode: buffer 0's first phase completes before the tile
            // that reuses the buffer lands, so that the buffer warps' wait
            // for it implies that phase (the drains do for later tiles): a
            // buffer warp running ahead cannot arrive for tile kNB in place
            // of a sibling still to arrive for tile 0.
            if (kAtomicDq && gi == kNB && !mbar_wait(&s.buf_ready[0], 0, p.err, abort_flag))
              return false;
            const int q0 = qt * kQ64;
            mbar_arrive_expect_tx(&s.qdo_full[st], 2 * kDB * Smem::kQBlock + 2 * kQ64 * 4);
            for (int kb = 0; kb < kDB; ++kb) {
              tma_load_4d(s.q[st] + kb * Smem::kQBlock, &p.map_q64, &s.qdo_full[st], kb * 64, q0,
                          w.hh, w.bb);
              tma_load_4d(s.dO[st] + kb * Smem::kQBlock, &p.map_do64, &s.qdo_full[st], kb * 64, q0,
                          w.hh, w.bb);
            }
            const long long off = static_cast<long long>(w.bh) * Npad + q0;
            bulk_load(s.lse2[st], p.lse + off, kQ64 * 4, &s.qdo_full[st]);
            bulk_load(s.di[st], p.di + off, kQ64 * 4, &s.qdo_full[st]);
            issued = gi + 1;
          }
          return true;
        });
        if (*abort_flag) {
          int zero = 0;
          for (int t = max(0, kv_loads - kKVB); t < kv_loads; ++t)
            mbar_wait(&s.kv_full[t % kKVB], (t / kKVB) & 1, p.err, &zero, 100000000ull);
          for (int t = max(0, issued - kQS); t < issued; ++t)
            mbar_wait(&s.qdo_full[t % kQS], (t / kQS) & 1, p.err, &zero, 100000000ull);
        }
      }
    } else if (warp == 13) {
      // ------------------------------------------------------------ score products
      {
        const bool leader = elect_one_sync();
        auto leader_commit = [&](uint64_t* bar) {
          if (leader) tc_commit(bar);
        };
        constexpr uint32_t idS = idesc_f16(128, kQ64, ab, 0, 0);  // keys x queries, over d
        int gi = 0;
        for_each_unit([&](int k, const Unit&, const TileWalk<kSparse>& walk) -> bool {
          const int kvb = k % kKVB;
          if (!mbar_wait(&s.kv_full[kvb], (k / kKVB) & 1, p.err, abort_flag)) return false;
          const uint32_t k_addr = smem_u32(s.k[kvb]), v_addr = smem_u32(s.v[kvb]);
          const int n = walk.count();
          for (int i = 0; i < n; ++i, ++gi) {
            const int b = gi % kNB, st = gi % kQS;
            // A unit's products follow the previous unit's last dV, dK into
            // the tensor core's queue: the epilogue waits for those, not for
            // scores the elementwise warps need only after it.
            if (kResident && i == 0 && k > 0 &&
                !mbar_wait(&s.last_issued, (k - 1) & 1, p.err, abort_flag))
              return false;
            // Buffer b may take tile gi once buf_ready(gi) completes: one wait
            // here instead of three (each wait of this thread costs tensor time).
            if (!mbar_wait(&s.buf_ready[b], (gi / kNB) & 1, p.err, abort_flag)) return false;
            tc_fence_after();
            const uint32_t q_addr = smem_u32(s.q[st]), do_addr = smem_u32(s.dO[st]);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t ka = (kk >> 2) * Smem::kKBlock + (kk & 3) * 32;
              const uint32_t kq = (kk >> 2) * Smem::kQBlock + (kk & 3) * 32;
              if (leader)
                tc_mma_ss(tbase + b * 128, desc_add(smem_desc_sw128(k_addr, 16, 1024), ka),
                          desc_add(smem_desc_sw128(q_addr, 16, 1024), kq), idS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t ka = (kk >> 2) * Smem::kKBlock + (kk & 3) * 32;
              const uint32_t kq = (kk >> 2) * Smem::kQBlock + (kk & 3) * 32;
              if (leader)
                tc_mma_ss(tbase + b * 128 + 64, desc_add(smem_desc_sw128(v_addr, 16, 1024), ka),
                          desc_add(smem_desc_sw128(do_addr, 16, 1024), kq), idS, kk > 0 ? 1u : 0u);
            }
            leader_commit(&s.s_full[b]);
          }
          return true;
        });
        leader_commit(&s.drain[0]);
        int zero = 0;
        mbar_wait(&s.drain[0], 0, p.err, &zero, 100000000ull);
      }
    } else if (warp == 14) {
      // ------------------------------------------------------------ gradient products
      {
        const bool leader = elect_one_sync();
        auto leader_commit = [&](uint64_t* bar) {
          if (leader) tc_commit(bar);
        };
        constexpr uint32_t idKV = idesc_f16(128, D, ab, 0, 1);    // keys x d, over queries
        // d x queries, over keys; M = 128 at D = 64 too (rows past D unused)
        constexpr uint32_t idQ = idesc_f16(128, kQ64, ab, 1, 1);
        // dQ^T(j) = K^T dS^T(j), into the S^T columns of buffer (j + 1) % kNB,
        // with K from buffer kvb.
        auto issue_dq = [&](int j, int kvb) {
          const uint32_t k_addr = smem_u32(s.k[kvb]);
          const uint32_t dst_addr = smem_u32(s.dst[j % 3]);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            if (leader)
              tc_mma_ss(tbase + ((j + 1) % kNB) * 128,
                        desc_add(smem_desc_sw128(k_addr, Smem::kKBlock, 1024), kk * 16 * 128),
                        desc_add(smem_desc_sw128(dst_addr, Smem::kKBlock, 1024), kk * 16 * 128),
                        idQ, kk > 0 ? 1u : 0u);
          leader_commit(&s.dq_full[j % 3]);
        };
        int gi = 0;
        int kvb_prev = 0;        // K / V buffer of tile gi - 1
        bool prev_last = false;  // tile gi - 1 was the last of its unit
        const bool ok = for_each_unit([&](int k, const Unit&, const TileWalk<kSparse>& walk) -> bool {
          const int kvb = k % kKVB;
          const int n = walk.count();
          for (int i = 0; i < n; ++i, ++gi) {
            const int b = gi % kNB, st = gi % kQS;
            if (kAtomicDq && gi >= 1) {
              // S^T(gi) is in the elementwise warps' registers: dQ^T(gi - 1) can
              // take its columns (their previous occupant, dQ^T(gi - 1 - kNB), was
              // drained before S^T(gi) was issued), and dS^T(gi - 1) reached
              // shared memory before that signal.  It runs while the
              // elementwise step of tile gi does, off the chain that frees
              // buffer b for S^T(gi + 2).
              if (!mbar_wait(&s.s_read[b], (gi / kNB) & 1, p.err, abort_flag)) return false;
              tc_fence_after();
              issue_dq(gi - 1, kvb_prev);
              // the last product on the previous unit's K: its buffer is free
              // for unit k + 1 once this completes
              if (kResident && prev_last) leader_commit(&s.kv_empty[kvb_prev]);
            }
            if (!mbar_wait(&s.p_full[b], (gi / kNB) & 1, p.err, abort_flag)) return false;
            tc_fence_after();
            const uint32_t q_addr = smem_u32(s.q[st]), do_addr = smem_u32(s.dO[st]);
            // dV += P^T dO : A = P^T packed in TMEM over the dP^T columns.  The
            // first tile of a unit overwrites: the epilogue of the previous
            // unit read dV, dK before its threads signalled p_full(gi).
#pragma unroll
            for (int kk = 0; kk < kQ64 / 16; ++kk)
              if (leader)
                tc_mma_ts(tdV, tbase + b * 128 + 64 + (kk >> 1) * 32 + (kk & 1) * 8,
                          desc_add(smem_desc_sw128(do_addr, Smem::kQBlock, 1024), kk * 16 * 128),
                          idKV, (i > 0 || kk > 0) ? 1u : 0u);
            // dK += dS^T Q : A = dS^T packed in TMEM beside P^T
#pragma unroll
            for (int kk = 0; kk < kQ64 / 16; ++kk)
              if (leader)
                tc_mma_ts(tdK, tbase + b * 128 + 64 + (kk >> 1) * 32 + 16 + (kk & 1) * 8,
                          desc_add(smem_desc_sw128(q_addr, Smem::kQBlock, 1024), kk * 16 * 128),
                          idKV, (i > 0 || kk > 0) ? 1u : 0u);
            leader_commit(&s.qdo_empty[st]);
            // dV, dK(gi) done frees buffer b for tile gi + kNB: the commit
            // arrives on buf_ready(gi + kNB) itself, so the score warp wakes on
            // the tensor core's arrival, not on a relay.
            leader_commit(&s.buf_ready[b]);
            if (kResident && i == n - 1) {
              __syncwarp();
              if (leader) mbar_arrive(&s.last_issued);
            }
            kvb_prev = kvb;
            prev_last = i == n - 1;
          }
          // dV, dK of this unit are complete once this arrives: the epilogue
          // may read them.  The score products on this unit's K and V all
          // completed before its last P^T / dS^T existed.
          leader_commit(&s.acc_full);
          if (kResident && !kAtomicDq) leader_commit(&s.kv_empty[kvb]);
          return true;
        });
        // The CTA's last tile's dQ^T goes into buffer gi % kNB, once
        // dQ^T(gi - 1 - kNB) has left it and the last dS^T is in shared memory.
        if (ok && kAtomicDq && !*abort_flag && gi > 0) {
          const int j = gi - 1;
          if (mbar_wait(&s.ds_last, 0, p.err, abort_flag) &&
              (j < kNB || mbar_wait(&s.tmem_free[(j + 1) % kNB], ((j - kNB) / kNB) & 1, p.err,
                                    abort_flag))) {
            tc_fence_after();
            issue_dq(j, kvb_prev);
          }
        }
        leader_commit(&s.drain[1]);
        int zero = 0;
        mbar_wait(&s.drain[1], 0, p.err, &zero, 100000000ull);
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ buffer warps
    // Buffer gi % kNB may take S^T, dP^T(gi) once dV, dK(gi - kNB) are done
    // (the last readers of its P^T / dS^T; their tcgen05.commit arrives on
    // buf_ready(gi) directly), dQ^T(gi - 1 - kNB) has left its S^T columns
    // (atomic mode) and Q / dO(gi) have landed.  These warps see to the last
    // two, arrive on buf_ready(gi), and in atomic mode drain dQ^T (TMEM lane
    // = column d of dQ) into the fp32 accumulator.
    const int quad = warp & 3;
    const int d = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    int n_tiles = 0;  // tiles of all this CTA's units
    for (int k = 0; has_unit(k); ++k) n_tiles += walk_of(decode(unit_of(k))).count();
    // The drains run kNB + 1 tiles behind, into the next unit: the tile
    // drained next is query tile qt_d of unit wd, with left_d tiles of it
    // (this one included) still to drain.
    int kd = 0, qt_d = 0, left_d = 0;
    Unit wd{};
    for (int gi = 0; gi < n_tiles + (kAtomicDq ? kNB + 1 : 0); ++gi) {
      const int b = gi % kNB;
      const int j = gi - 1 - kNB;  // dQ^T(j) sits in the S^T columns of buffer (j + 1) % kNB = b
      const bool drain = kAtomicDq && j >= 0 && j < n_tiles;
      uint32_t g[2][32];
      if (drain) {
        if (!warp_wait(&s.dq_full[j % 3], (j / 3) & 1, p.err, abort_flag)) break;
        tc_fence_after();
        tmem_ld32(tbase + lane_off + b * 128, g[0]);
        tmem_ld32(tbase + lane_off + b * 128 + 32, g[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s.tmem_free[b]);  // for the last tile's dQ^T
      }
      if (gi < n_tiles) {
        if (!warp_wait(&s.qdo_full[gi % kQS], (gi / kQS) & 1, p.err, abort_flag)) break;
        __syncwarp();
        if (lane == 0) {
          // Buffer b's previous phase (tile gi - kNB) must be complete
          // before this warp arrives for tile gi: else a warp running ahead
          // could complete it in place of a sibling still behind.  (Atomic
          // mode: implied by the producer's wait before tile kNB and by the
          // drain waits.  A wait that gives up has set the abort flag, so
          // every later wait fails.)
          if (!kAtomicDq && gi >= kNB)
            mbar_wait(&s.buf_ready[b], ((gi - kNB) / kNB) & 1, p.err, abort_flag);
          mbar_arrive(&s.buf_ready[b]);
          // the first kNB tiles have no dV, dK(gi - kNB) to wait for
          if (gi < kNB && warp == 8) mbar_arrive(&s.buf_ready[b]);
        }
      }
      if (drain) {
        while (left_d == 0 && has_unit(kd)) {
          wd = decode(unit_of(kd++));
          left_d = walk_of(wd).count();
          qt_d = walk_of(wd).first();
        }
        const int q0 = qt_d * kQ64;
        --left_d;
        qt_d = walk_of(wd).next(qt_d);
        if constexpr (D == 64) {
          // Stage the tile in shared memory ([query][d], rows d < 64 come
          // from quadrants 0 and 1) and add it into the accumulator with one
          // bulk tensor reduction instead of 64 atomics per thread; rows
          // past N fall outside the tensor map and are dropped.
          const int sb = j & 1;
          if (quad < 2) {
            if (j >= 2 && !warp_wait(&s.stage_free[sb], ((j >> 1) - 1) & 1, p.err, abort_flag))
              break;
            float* stage = s.dq_stage[sb];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int c = 0; c < 32; ++c) stage[(h * 32 + c) * D + d] = __uint_as_float(g[h][c]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.stage_full[sb]);
          } else if (quad == 2) {
            // Warp 10 (its TMEM rows hold no dQ at D = 64) issues the
            // reduction, so the staging warps go straight on to the next
            // buffer.
            bool issued = true;  // one lane issues; the warp leaves the loop together
            if (lane == 0) {
              issued = mbar_wait(&s.stage_full[sb], (j >> 1) & 1, p.err, abort_flag);
              if (issued) {
                tma_reduce_add_4d(&p.map_dqacc, s.dq_stage[sb], 0, q0, wd.hh, wd.bb);
                tma_store_commit();
                // the reduction of tile j - 1 has read its buffer: free it
                tma_store_wait_read_all_but_newest();
                if (j >= 1) mbar_arrive(&s.stage_free[(j - 1) & 1]);
              }
            }
            if (!__all_sync(0xffffffffu, issued)) break;
          }
        } else {
          float* dst = p.dq_accum + (static_cast<long long>(wd.bh) * p.N + q0) * D + d;
          const int nq = d < D ? min(kQ64, p.N - q0) : 0;  // lanes past D hold no dQ
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (h * 32 + c < nq)
                atomicAdd(dst + static_cast<long long>(h * 32 + c) * D, __uint_as_float(g[h][c]));
        }
      }
    }
    // the last bulk reductions must have read shared memory before it goes
    if (kAtomicDq && D == 64 && warp == 10 && lane == 0) tma_store_wait_all();
  } else {
    if constexpr (D == 64) setmaxnreg_inc<kPipeHighRegs>();
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, query-column half
    const int r = quad * 32 + lane;                // key row (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    int gi = 0;
    int epi_last = -3;  // resident: the last tile before the latest epilogue
    // resident, thread 0: the latest epilogue's store has still to be
    // waited for and epi_read signalled (done before anyone waits on it)
    bool epi_signal = false;
    auto signal_epi_read = [&] {
      if (kResident && tid == 0 && epi_signal) {
        tma_store_wait_read_all();
        mbar_arrive(&s.epi_read);
        epi_signal = false;
      }
    };
    for_each_unit([&](int k, const Unit& w, const TileWalk<kSparse>& walk) -> bool {
      const int k0 = w.k0;
      const float nslope2 = kAlibi ? alibi_nslope2(p.band, w.bh, p.H) : 0.f;
      const int n = walk.count();
      bool ok = true;
      for (int i = 0, qt = walk.first(); i < n; ++i, qt = walk.next(qt), ++gi) {
        const int b = gi % kNB, st = gi % kQS;  // buffer, Q / dO stage
        const int sd = gi % 3;                   // dS^T stage
        const int q0 = qt * kQ64;
        // S^T(gi) was issued after dV, dK(gi - kNB), the last readers of the
        // P^T / dS^T columns of buffer b, had completed.
        if (!warp_wait(&s.s_full[b], (gi / kNB) & 1, p.err, abort_flag) ||
            !warp_wait(&s.qdo_full[st], (gi / kQS) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[32], dr[32];
        tmem_ld32(tbase + lane_off + b * 128 + half * 32, sr);
        tmem_ld32(tbase + lane_off + b * 128 + 64 + half * 32, dr);
        tmem_ld_wait();
        if (kAtomicDq) {
          // S^T(gi) has left TMEM (and dS^T(gi - 1), stored in the previous
          // iteration, is in shared memory): dQ^T(gi - 1) may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.s_read[b]);
        }
        const bool cut = band_cuts(q0, kQ64, k0, kTile, wl, wr);
        // ALiBi on a tile wholly on one side of the diagonal: |key - q| is
        // linear in the column, the bias B + D e (e = column of this half)
        const bool below = k0 + kTile - 1 <= q0, above = q0 + kQ64 - 1 <= k0;
        const bool lin = kAlibi && (below || above);
        uint32_t pk[16], dk[16];
        if (!cut && (!kAlibi || lin)) {
          // P = 2^(S * scale * log2 e - LSE2 [+ bias]) and dS = P (dP - Di),
          // two columns per packed instruction: the elementwise warps share
          // their SM sub-partitions with the MMA-issuing warps, so every
          // instruction saved here is issue time given back to the tensor core.
          const uint64_t nsl2 = f32x2(-sl2, -sl2), neg1 = f32x2(-1.f, -1.f);
          const float qk = static_cast<float>(q0 + half * 32 - (k0 + r));  // query - key at e = 0
          const float slope = below ? nslope2 : -nslope2;
          const uint64_t nb2 = f32x2(-slope * qk, -slope * qk), nd2 = f32x2(-slope, -slope);
#pragma unroll
          for (int t = 0; t < 32; t += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(&s.lse2[st][half * 32 + t]);
            const float4 d4 = *reinterpret_cast<const float4*>(&s.di[st][half * 32 + t]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = t + 2 * h;
              uint64_t l2 = h ? f32x2(l4.z, l4.w) : f32x2(l4.x, l4.y);
              if (lin)  // LSE2 - bias
                l2 = fma_f32x2(f32x2(static_cast<float>(e), static_cast<float>(e + 1)), nd2,
                               add_f32x2(l2, nb2));
              // -z = LSE2 [- bias] - S * scale_log2
              const float2 nz = split_f32x2(
                  fma_f32x2(f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2, l2));
              const float p0 = ex2_approx(-nz.x), p1 = ex2_approx(-nz.y);
              const uint64_t dd =
                  fma_f32x2(h ? f32x2(d4.z, d4.w) : f32x2(d4.x, d4.y), neg1,
                            f32x2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])));
              const float2 ds = split_f32x2(mul_f32x2(f32x2(p0, p1), dd));
              pk[e / 2] = pack2<kBf16>(p0, p1);
              dk[e / 2] = pack2<kBf16>(ds.x, ds.y);
            }
          }
        } else {
          // a tile the band cuts, or an ALiBi bias: key k0 + r, query q
          const int key = k0 + r;
#pragma unroll
          for (int t = 0; t < 32; t += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(&s.lse2[st][half * 32 + t]);
            const float4 d4 = *reinterpret_cast<const float4*>(&s.di[st][half * 32 + t]);
            const float ll[4] = {l4.x, l4.y, l4.z, l4.w};
            const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
            float pv[4], dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = q0 + half * 32 + t + e;
              float z = fmaf(__uint_as_float(sr[t + e]), sl2, -ll[e]);
              if (kAlibi) z = fmaf(nslope2, fabsf(static_cast<float>(key - q)), z);
              float pe = ex2_approx(z);
              if (cut && !band_visible(q, key, wl, wr)) pe = 0.f;
              pv[e] = pe;
              dsv[e] = pe * (__uint_as_float(dr[t + e]) - dd[e]);
            }
            pk[t / 2] = pack2<kBf16>(pv[0], pv[1]);
            pk[t / 2 + 1] = pack2<kBf16>(pv[2], pv[3]);
            dk[t / 2] = pack2<kBf16>(dsv[0], dsv[1]);
            dk[t / 2 + 1] = pack2<kBf16>(dsv[2], dsv[3]);
          }
        }
        // P^T and dS^T over this warp's own 32 dP^T columns (already read):
        // P^T in the first 16, dS^T in the next 16.
        tmem_st16(tbase + lane_off + b * 128 + 64 + half * 32, pk);
        tmem_st16(tbase + lane_off + b * 128 + 64 + half * 32 + 16, dk);
        tmem_st_wait();
        tc_fence_before();
        // P(gi) also publishes dS^T(gi - 1), stored and fenced below in the
        // previous iteration; dV, dK(gi) need only the TMEM operands.
        mbar_arrive(&s.p_full[b]);
        if (kAtomicDq) {
          // dQ^T(gi - 3) was the last reader of dS^T buffer gi % 3; resident,
          // the two tiles after an epilogue find its dK, dV tiles there until
          // their bulk stores have read them.
          signal_epi_read();
          if ((gi >= 3 && !warp_wait(&s.dq_full[sd], ((gi - 3) / 3) & 1, p.err, abort_flag)) ||
              (kResident && gi - epi_last <= 2 &&
               !warp_wait(&s.epi_read, (k - 1) & 1, p.err, abort_flag))) {
            ok = false;
            break;
          }
          store_row_chunk_sw128(s.dst[sd], r, half, dk);
          fence_proxy_async_smem();
        }
      }
      if (kAtomicDq && ok && !has_unit(k + 1)) mbar_arrive(&s.ds_last);

      // -------------------------------------------------------- epilogue
      // dK, dV staged in shared memory: the free Q / dO ring (16 or 32 KB
      // of 32 or 48 each) of a CTA with one unit; a resident CTA's ring
      // already holds its next unit's tiles, so it takes the dS^T buffers
      // of tiles gl - 2 and gl - 1 (gl: this unit's last tile, gi - 1) once
      // their dQ^T products and the previous epilogue's stores have read them.
      const int gl = gi - 1;
      uint8_t* dk_tile = kResident ? s.dst[(gl + 1) % 3] : s.q[0];
      uint8_t* dv_tile = kResident ? s.dst[(gl + 2) % 3] : s.dO[0];
      // (polled: the elementwise warps are idle until dV, dK are complete, and
      // a sleeping wait wakes later)
      bool done = ok && __all_sync(0xffffffffu, mbar_wait_poll(&s.acc_full, k & 1, p.err, abort_flag));
      signal_epi_read();
      if (kResident && done && k > 0) done = warp_wait(&s.epi_read, (k - 1) & 1, p.err, abort_flag);
      if (kResident && kAtomicDq) {
        for (int j = max(0, gl - 2); done && j < gl; ++j)
          done = warp_wait(&s.dq_full[j % 3], (j / 3) & 1, p.err, abort_flag);
      }
      if (!named_bar_and(1, 256, done)) return false;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kDB; ++c) {  // this warp's D / 2 columns, 32 at a time
        const int c32 = half * kDB + c;
        uint32_t a[32], g[32];
        if (n > 0) {
          tmem_ld32(tdV + lane_off + c32 * 32, a);
          tmem_ld32(tdK + lane_off + c32 * 32, g);
          tmem_ld_wait();
        } else {  // a key tile the block mask leaves unseen: dK = dV = 0
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = g[e] = 0u;
        }
        uint32_t pa[16], pb[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          pa[t] = pack2<kBf16>(__uint_as_float(a[2 * t]), __uint_as_float(a[2 * t + 1]));
          pb[t] = pack2<kBf16>(__uint_as_float(g[2 * t]) * p.scale,
                               __uint_as_float(g[2 * t + 1]) * p.scale);
        }
        store_row_chunk_sw128(dv_tile, r, c32, pa);
        store_row_chunk_sw128(dk_tile, r, c32, pb);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (tid == 0) {
        for (int kb = 0; kb < kDB; ++kb) {
          tma_store_4d(&p.map_dv, dv_tile + kb * Smem::kKBlock, kb * 64, k0, w.hh, w.bb);
          tma_store_4d(&p.map_dk, dk_tile + kb * Smem::kKBlock, kb * 64, k0, w.hh, w.bb);
        }
        tma_store_commit();
        if constexpr (kResident) {
          epi_signal = true;
        } else {
          tma_store_wait_all();
        }
      }
      epi_last = gl;
      return true;
    });
    if (kResident && tid == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// deterministic dQ, software-pipelined over 64-key tiles (D = 64 or 128)
// ---------------------------------------------------------------------------
// One CTA per 128-row query tile.  dQ accumulates in TMEM over the key tiles
// in a fixed order, so the result does not depend on scheduling:
//   TMEM [128b, 128b + 64)       buffer b: S of key tile i (b = i % 3)
//   TMEM [128b + 64, 128b + 128) buffer b: dP of tile i, then dS packed over
//                                each elementwise warp's own 32 columns
//   TMEM [384, 384 + D)          dQ
// The score warp issues S = Q K^T and dP = dO V^T of tile i once buffer
// i % 3 is free (dQ(i - 3), the last reader of its dS, done; K, V(i)
// landed, confirmed by a relay warp so the issuing thread waits once per
// tile; the two issuing warps run their loops whole, one elected lane
// issuing, and poll their barriers rather than sleep); eight warps form
// dS = P (dP - Di), P = 2^(S * scale * log2 e -
// LSE2), one query row per thread so its LSE and Di sit in registers; the
// gradient warp issues dQ += dS K with dS read from TMEM.  Q and dO are
// loaded once; K and V come through a four-stage ring.
constexpr int kDqPipeThreads = 384;  // warps 0-7 elementwise, 8 relay, 9 producer, 10-11 MMA
constexpr int kK64 = 64;

template <int D, bool kSparse>
struct DqPipeSmem {
  // TMEM buffers for S / dP (3 x 128 columns beside dQ's D) and K / V
  // stages (one more, so that a tile's loads start before its buffer is free)
  static constexpr int kBufs = 3;
  static constexpr int kKVStages = kBufs + 1;
  static constexpr int kDBlocks = D / 64;
  static constexpr int kQBlock = kTile * 128;  // 128 rows x 128 B
  static constexpr int kKBlock = kK64 * 128;   // 64 rows x 128 B
  alignas(1024) uint8_t q[kDBlocks * kQBlock];  // [D block][128 queries][64 d]; then dQ
  alignas(1024) uint8_t dO[kDBlocks * kQBlock];
  alignas(1024) uint8_t k[kKVStages][kDBlocks * kKBlock];  // [stage][D block][64 keys][64 d]
  alignas(1024) uint8_t v[kKVStages][kDBlocks * kKBlock];
  alignas(16) float lse2[kTile];
  alignas(16) float di[kTile];
  uint64_t q_full, kv_full[kKVStages], kv_empty[kKVStages], s_full[kBufs], p_full[kBufs],
      buf_ready[kBufs];
  uint64_t all_done, drain[2];
  uint32_t tmem_base;
  int abort_flag;
  uint32_t k_tiles[kSparse ? 2 * kMaxSparseTiles / 32 : 1];  // block-sparse: 64-key tiles
};

template <int D, bool kBf16, bool kAlibi, bool kSparse>
__global__ void __launch_bounds__(kDqPipeThreads, 1)
    bwd_dq_pipe_kernel(const __grid_constant__ BwdLaunch p) {
  pdl_wait();
  using Smem = DqPipeSmem<D, kSparse>;
  constexpr int kDB = Smem::kDBlocks;
  constexpr int kNB = Smem::kBufs;       // S / dP buffers: tile it uses buffer it % kNB
  constexpr int kKS = Smem::kKVStages;   // K / V stages: tile it uses stage it % kKS
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_qt = (p.N + kTile - 1) / kTile;
  const int Npad = n_qt * kTile;
  const int n_k64 = (p.N + kK64 - 1) / kK64;
  // Head-major; when keys are bounded on the right only (causal) later
  // query tiles see more keys and go first.
  // (tile-major instead when the streamed operands all fit in L2)
  const int bh = static_cast<int>(p.tile_major ? blockIdx.x % p.BH : blockIdx.x / n_qt);
  const int hh = bh % p.H, bb = bh / p.H;  // TMA coordinates of (batch, head)
  const int wl = p.band.win_left, wr = p.band.win_right;
  const int tile_idx = static_cast<int>(p.tile_major ? blockIdx.x / p.BH : blockIdx.x % n_qt);
  const int qt = (wl < 0 && wr >= 0) ? n_qt - 1 - tile_idx : tile_idx;
  const int q0 = qt * kTile;
  int it_begin, it_last;  // 64-key tiles this query tile's band reaches
  band_key_tiles(q0, kTile, kK64, n_k64, wl, wr, it_begin, it_last);
  const TileWalk<kSparse> walk{it_begin, it_last, n_k64, TileSet{s.k_tiles, n_k64}};
  if constexpr (kSparse)  // the mask's 128-key blocks hold 64-key tiles 2b, 2b + 1
    fill_tile_set(s.k_tiles, n_k64, [&](int t) {
      return t >= it_begin && t <= it_last && block_kept(p.band, bh, p.H, n_qt, qt, t >> 1);
    });
  __syncthreads();
  const int n_it = walk.count();

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kKS; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 256);
      // the relay warp and the tcgen05.commit that retires dQ(it - kNB)
      mbar_init(&s.buf_ready[i], 2);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&s.drain[i], 1);
    mbar_init(&s.all_done, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t tdQ = tbase + kNB * 128;
  volatile int* abort_flag = &s.abort_flag;
  constexpr uint32_t ab = kBf16 ? 1u : 0u;

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&s.q_full, 2 * kDB * Smem::kQBlock + 2 * kTile * 4);
      for (int kb = 0; kb < kDB; ++kb) {
        tma_load_4d(s.q + kb * Smem::kQBlock, &p.map_q, &s.q_full, kb * 64, q0, hh, bb);
        tma_load_4d(s.dO + kb * Smem::kQBlock, &p.map_do, &s.q_full, kb * 64, q0, hh, bb);
      }
      const long long off = static_cast<long long>(bh) * Npad + q0;
      bulk_load(s.lse2, p.lse + off, kTile * 4, &s.q_full);
      bulk_load(s.di, p.di + off, kTile * 4, &s.q_full);
      int issued = 0;
      for (int it = 0, t = walk.first(); it < n_it; ++it, t = walk.next(t)) {
        const int st = it % kKS;
        if (it >= kKS && !mbar_wait(&s.kv_empty[st], ((it - kKS) / kKS) & 1, p.err, abort_flag))
          break;
        mbar_arrive_expect_tx(&s.kv_full[st], 2 * kDB * Smem::kKBlock);
        for (int kb = 0; kb < kDB; ++kb) {
          tma_load_4d(s.k[st] + kb * Smem::kKBlock, &p.map_k64, &s.kv_full[st], kb * 64,
                      t * kK64, hh, bb);
          tma_load_4d(s.v[st] + kb * Smem::kKBlock, &p.map_v64, &s.kv_full[st], kb * 64,
                      t * kK64, hh, bb);
        }
        issued = it + 1;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's smem goes away.
        int zero = 0;
        mbar_wait(&s.q_full, 0, p.err, &zero, 100000000ull);
        for (int t = max(0, issued - kKS); t < issued; ++t)
          mbar_wait(&s.kv_full[t % kKS], (t / kKS) & 1, p.err, &zero, 100000000ull);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ relay
    // Buffer it % kNB takes S, dP(it) once K, V(it) have landed (seen here)
    // and dQ(it - kNB) is done (its tcgen05.commit arrives on buf_ready).
    for (int it = 0; it < n_it; ++it) {
      if (!warp_wait(&s.kv_full[it % kKS], (it / kKS) & 1, p.err, abort_flag)) break;
      if (lane == 0) {
        mbar_arrive(&s.buf_ready[it % kNB]);
        if (it < kNB) mbar_arrive(&s.buf_ready[it % kNB]);  // no dQ(it - kNB) to wait for
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ score products
    {
      const bool leader = elect_one_sync();
      auto leader_commit = [&](uint64_t* bar) {
        if (leader) tc_commit(bar);
      };
      constexpr uint32_t idS = idesc_f16(128, kK64, ab, 0, 0);  // queries x keys, over d
      const uint32_t q_addr = smem_u32(s.q), do_addr = smem_u32(s.dO);
      bool ok = mbar_wait_poll(&s.q_full, 0, p.err, abort_flag);
      for (int it = 0; ok && it < n_it; ++it) {
        const int b = it % kNB, st = it % kKS;
        if (!mbar_wait_poll(&s.buf_ready[b], (it / kNB) & 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(s.k[st]), v_addr = smem_u32(s.v[st]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oq = (kk >> 2) * Smem::kQBlock + (kk & 3) * 32;
          const uint32_t ok_ = (kk >> 2) * Smem::kKBlock + (kk & 3) * 32;
          if (leader) tc_mma_ss(tbase + b * 128, desc_add(smem_desc_sw128(q_addr, 16, 1024), oq),
                    desc_add(smem_desc_sw128(k_addr, 16, 1024), ok_), idS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oq = (kk >> 2) * Smem::kQBlock + (kk & 3) * 32;
          const uint32_t ok_ = (kk >> 2) * Smem::kKBlock + (kk & 3) * 32;
          if (leader) tc_mma_ss(tbase + b * 128 + 64, desc_add(smem_desc_sw128(do_addr, 16, 1024), oq),
                    desc_add(smem_desc_sw128(v_addr, 16, 1024), ok_), idS, kk > 0 ? 1u : 0u);
        }
        leader_commit(&s.s_full[b]);
      }
      leader_commit(&s.drain[0]);
      int zero = 0;
      mbar_wait_poll(&s.drain[0], 0, p.err, &zero, 100000000ull);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ gradient products
    {
      const bool leader = elect_one_sync();
      auto leader_commit = [&](uint64_t* bar) {
        if (leader) tc_commit(bar);
      };
      constexpr uint32_t idQ = idesc_f16(128, D, ab, 0, 1);  // queries x d, over keys
      for (int it = 0; it < n_it; ++it) {
        const int b = it % kNB, st = it % kKS;
        if (!mbar_wait_poll(&s.p_full[b], (it / kNB) & 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(s.k[st]);
        // dQ += dS K : A = dS packed in TMEM over the dP columns (keys 32h ..
        // 32h + 31 in columns 32h .. 32h + 15), B = K MN-major (d contiguous)
#pragma unroll
        for (int kk = 0; kk < kK64 / 16; ++kk)
          if (leader) tc_mma_ts(tdQ, tbase + b * 128 + 64 + (kk >> 1) * 32 + (kk & 1) * 8,
                    desc_add(smem_desc_sw128(k_addr, Smem::kKBlock, 1024), kk * 16 * 128), idQ,
                    (it > 0 || kk > 0) ? 1u : 0u);
        leader_commit(&s.kv_empty[st]);  // S, dP(it) completed before dS(it) existed
        leader_commit(&s.buf_ready[b]);  // frees buffer b for tile it + 2
      }
      // The score products all completed before the last dS existed, so
      // this commit covers every product of the CTA.
      leader_commit(&s.all_done);
      leader_commit(&s.drain[1]);
      int zero = 0;
      mbar_wait_poll(&s.drain[1], 0, p.err, &zero, 100000000ull);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, key-column half
    const int r = quad * 32 + lane;                // query row (TMEM lane)
    const int i = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const float nslope2 = kAlibi ? alibi_nslope2(p.band, bh, p.H) : 0.f;
    bool ok = warp_wait(&s.q_full, 0, p.err, abort_flag);
    const float lse2 = s.lse2[r], dii = s.di[r];  // +inf / 0 for rows past N
    for (int it = 0, t = walk.first(); ok && it < n_it; ++it, t = walk.next(t)) {
      const int b = it % kNB;
      const int k0 = t * kK64;
      if (!warp_wait(&s.s_full[b], (it / kNB) & 1, p.err, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[32], dr[32];
      tmem_ld32(tbase + lane_off + b * 128 + half * 32, sr);
      tmem_ld32(tbase + lane_off + b * 128 + 64 + half * 32, dr);
      tmem_ld_wait();
      const bool cut = band_cuts(q0, kTile, k0, kK64, wl, wr) || k0 + kK64 > p.N;
      // ALiBi on a tile wholly on one side of the diagonal: |key - i| is
      // linear in the column, the bias B + D e (e = column of this half)
      const bool below = k0 + kK64 - 1 <= q0, above = q0 + kTile - 1 <= k0;
      const bool lin = kAlibi && (below || above);
      uint32_t dk[16];
      if (!cut && (!kAlibi || lin)) {
        // two columns per packed instruction: -z = LSE2 [- bias] -
        // S * scale_log2, dS = P (dP - Di)
        const uint64_t nsl2 = f32x2(-sl2, -sl2);
        const float kq = static_cast<float>(k0 + half * 32 - i);  // key - query at e = 0
        const float sd = above ? nslope2 : -nslope2;
        const uint64_t lb2 = f32x2(lse2 - sd * kq, lse2 - sd * kq), nd2 = f32x2(-sd, -sd);
        const uint64_t l2 = f32x2(lse2, lse2);
        const uint64_t neg1 = f32x2(-1.f, -1.f), d2 = f32x2(dii, dii);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t off =
              lin ? fma_f32x2(f32x2(static_cast<float>(e), static_cast<float>(e + 1)), nd2, lb2)
                  : l2;
          const float2 nz = split_f32x2(
              fma_f32x2(f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2, off));
          const float p0 = ex2_approx(-nz.x), p1 = ex2_approx(-nz.y);
          const uint64_t dd =
              fma_f32x2(d2, neg1, f32x2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])));
          const float2 ds = split_f32x2(mul_f32x2(f32x2(p0, p1), dd));
          dk[e / 2] = pack2<kBf16>(ds.x, ds.y);
        }
      } else {
        // a tile the band cuts, a ragged last tile, or an ALiBi bias
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float d2v[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int key = k0 + half * 32 + e + u;
            float z = fmaf(__uint_as_float(sr[e + u]), sl2, -lse2);
            if (kAlibi) z = fmaf(nslope2, fabsf(static_cast<float>(key - i)), z);
            float pe = ex2_approx(z);
            if (key >= p.N || (cut && !band_visible(i, key, wl, wr))) pe = 0.f;
            d2v[u] = pe * (__uint_as_float(dr[e + u]) - dii);
          }
          dk[e / 2] = pack2<kBf16>(d2v[0], d2v[1]);
        }
      }
      // dS over the first 16 of this warp's own 32 dP columns (already read)
      tmem_st16(tbase + lane_off + b * 128 + 64 + half * 32, dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[b]);
    }

    // ---------------------------------------------------------- epilogue
    // A query tile the block mask leaves without keys has dQ = 0; Q, the
    // output stage, has landed (q_full) and no product reads it any more.
    const bool done = ok && warp_wait(&s.all_done, 0, p.err, abort_flag);
    if (named_bar_and(1, 256, done)) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kDB; ++c) {  // this warp's D / 2 columns, 32 at a time
        const int c32 = half * kDB + c;
        uint32_t g[32];
        if (n_it > 0) {
          tmem_ld32(tdQ + lane_off + c32 * 32, g);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) g[e] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<kBf16>(__uint_as_float(g[2 * e]) * p.scale,
                               __uint_as_float(g[2 * e + 1]) * p.scale);
        store_row_chunk_sw128(s.q, r, c32, pk);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (tid == 0) {
        for (int kb = 0; kb < kDB; ++kb)
          tma_store_4d(&p.map_dq, s.q + kb * Smem::kQBlock, kb * 64, q0, hh, bb);
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ convert
// ---------------------------------------------------------------------------
// acc is [BH][N][D] fp32; dq gets scale * acc in the caller's layout.  One
// thread per 8 consecutive elements of a row.  The row -> (batch, head,
// position) split uses 32-bit division whenever the row count allows: with
// 64-bit division the index arithmetic, not HBM, set the kernel's pace.
template <bool kBf16, int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         uint16_t* __restrict__ dq, RowStrides sdq,
                                                         int N, int H, long long n8, float scale) {
  pdl_wait();
  constexpr int g = D / 8;  // threads per row
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const bool rows32 = n8 / g <= 0xffffffffLL;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8;
       t += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * t];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * t + 1];
    uint4 o;
    o.x = pack2<kBf16>(a.x * scale, a.y * scale);
    o.y = pack2<kBf16>(a.z * scale, a.w * scale);
    o.z = pack2<kBf16>(b.x * scale, b.y * scale);
    o.w = pack2<kBf16>(b.z * scale, b.w * scale);
    const long long row = t / g;  // over BH * N
    long long n;
    int bh;
    if (rows32) {
      const uint32_t r = static_cast<uint32_t>(row), q = r / static_cast<uint32_t>(N);
      bh = static_cast<int>(q);
      n = r - q * static_cast<uint32_t>(N);
    } else {
      bh = static_cast<int>(row / N);
      n = row - static_cast<long long>(bh) * N;
    }
    const int bb = bh / H, hh = bh - bb * H;
    *reinterpret_cast<uint4*>(dq + bb * sdq.batch + hh * sdq.head + n * sdq.seq + (t % g) * 8) = o;
  }
}

// ---------------------------------------------------------------------------
// bounded-wait self test: one barrier nobody signals
// ---------------------------------------------------------------------------
__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, err, &abort_flag, limit_ns);
}

template <int D, bool kBf16, bool kAlibi, bool kSparse>
cudaError_t launch_dq_t(const BwdLaunch& a, cudaStream_t st) {
  auto kern = bwd_dq_pipe_kernel<D, kBf16, kAlibi, kSparse>;
  const int smem = static_cast<int>(sizeof(DqPipeSmem<D, kSparse>)) + 1024;
  static AttrCache configured;
  cudaError_t e = ensure_dynamic_smem(kern, smem, configured);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((a.N + kTile - 1) / kTile) * a.BH;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  BwdLaunch b = a;  // streamed per head: K and V
  b.tile_major = tile_major_order(a.band, 4LL * a.BH * a.N * a.D);
  return launch_pdl(kern, static_cast<unsigned>(grid), kDqPipeThreads, smem, st, b);
}

// Every backward kernel is launched with programmatic stream serialization
// (launch_pdl) and starts with pdl_wait(): the launch of each of the short
// kernels of a backward pass overlaps the tail of the one before it, and a
// kernel that waits never signals early, so its waiting CTAs do not take SMs
// from a grid still running (B8 H12 N1024 D64 causal, forward + backward
// 115.8 -> 109.0 us; B32 H16 N512 D64, 232.5 -> 225.6 us).
template <int D, bool kBf16, bool kAlibi, bool kAtomic, bool kSparse, bool kResident>
cudaError_t launch_dkdv_grid(const BwdLaunch& b, long long grid, cudaStream_t st) {
  auto kern = bwd_dkdv_pipe_kernel<D, kBf16, kAlibi, kAtomic, kSparse, kResident>;
  const int smem = static_cast<int>(sizeof(DkdvPipeSmem<D, kSparse, kResident>)) + 1024;
  static AttrCache configured;
  cudaError_t e = ensure_dynamic_smem(kern, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, static_cast<unsigned>(grid), kPipeThreads<D>, smem, st, b);
}

template <int D, bool kBf16, bool kAlibi, bool kAtomic, bool kSparse>
cudaError_t launch_dkdv_pipe_t(const BwdLaunch& a, cudaStream_t st) {
  const long long n_kt = (a.N + kTile - 1) / kTile;
  const long long units = n_kt * a.BH;
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  BwdLaunch b = a;  // streamed per head: Q, dO and, atomic mode, the fp32 dQ accumulator
  b.tile_major = tile_major_order(a.band, (kAtomic ? 8LL : 4LL) * a.BH * a.N * a.D);
  if constexpr (D == 64 && !kSparse) {
    // Short sequences (at most 32 key tiles) with more key tiles than SMs:
    // resident CTAs, one per SM, each loading its next key tile while it
    // works on this one (a CTA per key tile spends about a third of its
    // time starting, loading K, V and storing dK, dV at these lengths).
    if (n_kt <= 32) {
      int sms = 0;
      const cudaError_t e = sm_count(&sms);
      if (e != cudaSuccess) return e;
      if (units > sms) return launch_dkdv_grid<D, kBf16, kAlibi, kAtomic, kSparse, true>(b, sms, st);
    }
  }
  return launch_dkdv_grid<D, kBf16, kAlibi, kAtomic, kSparse, false>(b, units, st);
}

template <int D, bool kBf16, bool kSparse>
cudaError_t launch_dkdv_ds(const BwdLaunch& a, cudaStream_t st) {
  const bool atomic = a.dq_accum != nullptr;
  const bool alibi = a.band.alibi != nullptr;
  if (alibi)
    return atomic ? launch_dkdv_pipe_t<D, kBf16, true, true, kSparse>(a, st)
                  : launch_dkdv_pipe_t<D, kBf16, true, false, kSparse>(a, st);
  return atomic ? launch_dkdv_pipe_t<D, kBf16, false, true, kSparse>(a, st)
                : launch_dkdv_pipe_t<D, kBf16, false, false, kSparse>(a, st);
}

template <int D, bool kBf16>
cudaError_t launch_dkdv_d(const BwdLaunch& a, cudaStream_t st) {
  return a.band.block_mask ? launch_dkdv_ds<D, kBf16, true>(a, st)
                           : launch_dkdv_ds<D, kBf16, false>(a, st);
}

template <int D, bool kBf16>
cudaError_t launch_dq_d(const BwdLaunch& a, cudaStream_t st) {
  const bool alibi = a.band.alibi != nullptr;
  if (a.band.block_mask)
    return alibi ? launch_dq_t<D, kBf16, true, true>(a, st) : launch_dq_t<D, kBf16, false, true>(a, st);
  return alibi ? launch_dq_t<D, kBf16, true, false>(a, st) : launch_dq_t<D, kBf16, false, false>(a, st);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, RowStrides so, const void* dO, RowStrides sdo,
                                  const float* lse, float* lse2, float* di, float* dq_accum, int N,
                                  int H, long long BH, int D, int bf16, cudaStream_t st) {
  const int Npad = (N + kTile - 1) / kTile * kTile;
  const long long threads = BH * Npad * (D / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
  const auto* o16 = static_cast<const uint16_t*>(o);
  const auto* d16 = static_cast<const uint16_t*>(dO);
  const unsigned g = static_cast<unsigned>(blocks);
  auto kern = D == 64 ? (bf16 ? bwd_preprocess_kernel<64, true> : bwd_preprocess_kernel<64, false>)
                      : (bf16 ? bwd_preprocess_kernel<128, true> : bwd_preprocess_kernel<128, false>);
  return launch_pdl(kern, g, 256, 0, st, o16, so, d16, sdo, lse, lse2, di, dq_accum, N, Npad, H,
                    BH);
}

cudaError_t launch_bwd_dkdv(const BwdLaunch& a, cudaStream_t st) {
  if (a.D == 64) return a.bf16 ? launch_dkdv_d<64, true>(a, st) : launch_dkdv_d<64, false>(a, st);
  return a.bf16 ? launch_dkdv_d<128, true>(a, st) : launch_dkdv_d<128, false>(a, st);
}

cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t st) {
  if (a.D == 64) return a.bf16 ? launch_dq_d<64, true>(a, st) : launch_dq_d<64, false>(a, st);
  return a.bf16 ? launch_dq_d<128, true>(a, st) : launch_dq_d<128, false>(a, st);
}

cudaError_t launch_dq_convert(const float* acc, void* dq, RowStrides sdq, int N, int H,
                              long long BH, int D, float scale, int bf16, cudaStream_t st) {
  const long long n8 = BH * N * D / 8;
  int sms = 0;
  const cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  long long blocks = (n8 + 255) / 256;  // grid-stride, at most 16 CTAs per SM
  if (blocks > 16LL * sms) blocks = 16LL * sms;
  if (blocks < 1) blocks = 1;
  auto* d16 = static_cast<uint16_t*>(dq);
  const unsigned g = static_cast<unsigned>(blocks);
  auto kern = D == 64 ? (bf16 ? dq_convert_kernel<true, 64> : dq_convert_kernel<false, 64>)
                      : (bf16 ? dq_convert_kernel<true, 128> : dq_convert_kernel<false, 128>);
  return launch_pdl(kern, g, 256, 0, st, acc, d16, sdq, N, H, n8, scale);
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa
