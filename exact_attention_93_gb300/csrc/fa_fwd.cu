// fa_fwd.cu -- exact attention forward for sm_103a.
//
// A work unit is two 128-row query tiles (A and B, adjacent in one
// (batch, head)); a CTA computes one unit, or several in turn (below),
// walking the key/value tiles with an online softmax
// ("FlashAttention from scratch" walkthrough, l189.com, sec. 2.2 and 2.4;
// "FlashAttention 深入", online softmax).  Parallelism is over query tiles
// as well as (batch, head), the sequence-dimension split of FlashAttention-2
// ("FlashAttention 深入", v2).
//
// Warp roles (384 threads; warps 10 and 11 only lend their registers to
// the softmax warps, see kFwdThreads):
//   warps 0-3  softmax for tile A, warps 4-7 softmax for tile B: thread t of
//              a group owns query row t of its tile (= TMEM lane t).  Reads S
//              from TMEM, keeps the running max m and sum l in fp32
//              (walkthrough sec. 5.2), writes P as 16-bit pairs back into the
//              same TMEM columns, rescales O in TMEM when m grows, and runs
//              the epilogue (O / l through a swizzled smem tile and a TMA
//              store; LSE = ln 2 * (m + log2 l)).
//   warp 8     TMA producer: a unit's two Q tiles once (into one of two
//              buffer sets when the CTA runs several units), K and V tiles
//              into two smem stages.
//   warp 9     MMA issuer: with 16-bit operands the whole warp runs the
//              issue loop, so that its operands stay warp-uniform, and one
//              elected lane issues each product and commit (8-bit operands:
//              lane 0 alone).  For key tile j it issues
//                O_A += P_A(j) V_j, S_A(j+1) = Q_A K_{j+1}^T,
//                O_B += P_B(j) V_j, S_B(j+1) = Q_B K_{j+1}^T,
//              so while one group's softmax works on its scores the tensor
//              core runs the other group's products.
//
// TMEM columns: [0,128) S/P of tile A, [128,256) S/P of tile B,
// [256,256+D) O of tile A, [256+D,256+2D) O of tile B.
//
// Softmax bookkeeping works in log2 units: scores are multiplied by
// scale*log2(e) and exponentiated with ex2.  The reference maximum m is only
// moved when the tile maximum exceeds it by more than 8 (a factor of 256);
// P then stays below 256, and O / l and the LSE are unchanged because both
// use the same m.  Rows whose maximum barely moves never touch O in TMEM.
//
// Visible keys (fa_band.cuh): query i sees keys i - left .. i + right, the
// causal mask (walkthrough sec. 5.3) being right = 0.  Each query tile
// multiplies only the key tiles its band reaches; tiles the band cuts, and a
// ragged last tile, are masked element-wise.  The pair's two tiles share one
// K/V stream over the union of their key-tile ranges.  With an ALiBi slope
// (flash_attn_func alibi_slopes) every score gets -slope * |i - j| added
// before the softmax.  The grid runs head-major, the longest query-tile
// pairs of a head first, so the CTAs in flight share one head's K and V in L2
// (tile-major for short causal sequences whose K and V all fit in L2).
//
// Work units: a CTA may process several query-tile pairs in turn.  With
// short sequences the per-CTA costs (barrier set-up, TMEM allocation, the
// first loads, the epilogue, the launch of the next CTA) weigh as much as
// the key-tile loop, so the grid then holds one resident CTA per SM: the
// next unit's Q and first K/V land and its first scores are computed while
// the softmax warps still run the previous unit's epilogue.  All barrier
// phases count across units.
//
// 8-bit operands (the FP8 forward FlashAttention-3 adds, which the "Flash
// Attention" wiki page and the v3 row of "FlashAttention 深入" list): Q, K
// and V^T arrive as e4m3 bytes, both products run as kind::f8f6f4 (K = 32
// per step), P goes into TMEM as e4m3 (four keys per column) at a scale
// that keeps it below 256 and small weights normal, and O leaves in bf16
// through its own staging buffers.  Per-(batch, head) descale factors scale
// the scores (Q, K) and O (V).
#include <climits>

#include "fa_band.cuh"
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

// 12 warps: 0-7 softmax, 8 producer, 9 MMA, 10-11 idle.  The launch
// reserves 168 registers a thread (three warps share each SM sub-partition's
// 16384); warpgroup 2 (warps 8-11) gives up all but kFwdLowRegs and the two
// softmax warpgroups take kFwdHighRegs: 256 x 208 + 128 x 80 = 63488 of the
// 384 x 168 = 64512 reserved, and 32 x (208 + 208 + 80) = 15872 registers on
// each sub-partition.
constexpr int kFwdThreads = 384;
constexpr uint32_t kFwdLowRegs = 80, kFwdHighRegs = 208;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, bool kSparse, bool kFp8>
struct FwdSmem {
  static constexpr int kRowBytes = kFp8 ? D : 2 * D;  // one Q or K row
  // Q and K tiles: 128-byte column blocks (128-byte swizzle), or, for 8-bit
  // D = 64, one block of 64-byte rows (64-byte swizzle)
  static constexpr int kBlocks = kRowBytes >= 128 ? kRowBytes / 128 : 1;
  static constexpr int kBlockBytes = kTile * (kRowBytes >= 128 ? 128 : kRowBytes);
  static constexpr int kTileBytes = kBlocks * kBlockBytes;  // also V^T: D rows x 128 B
  static constexpr int kOBlocks = D / 64;                   // 16-bit O: 64-column blocks
  static constexpr int kOBlockBytes = kTile * 128;          // 128 rows x 128 B
  // O staging of its own (8-bit operands, or D = 64 where it fits beside the
  // tiles); 16-bit D = 128 stages O in the tile's spent Q buffer
  static constexpr bool kOwnStage = kFp8 || D == 64;
  // Q buffer sets: with O staged apart, a resident CTA loads the next unit's
  // Q into the other set while the current unit runs
  static constexpr int kQSets = kOwnStage ? 2 : 1;
  // tiles A and B; with 16-bit operands each is reused as its O staging
  alignas(1024) uint8_t q[kQSets][2][kTileBytes];  // [set][tile]
  alignas(1024) uint8_t k[2][kTileBytes];
  alignas(1024) uint8_t v[2][kTileBytes];  // 8-bit: V^T, D rows x 128 keys
  alignas(1024) uint8_t o[kOwnStage ? 2 : 1][kOwnStage ? kOBlocks * kOBlockBytes : 16];
  uint64_t q_full[kQSets], q_empty[kQSets];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2];  // per query tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  // block-sparse: key tiles of tile A, of tile B, and their union
  uint32_t key_tiles[kSparse ? 3 : 1][kSparse ? kMaxSparseTiles / 32 : 1];
};

// The key tiles one CTA multiplies: for each query tile t a range
// [lo_t, hi_t] (dense) or a set (block-sparse), and the K/V stream over
// their union in increasing order.  Every walk ends at the sentinel n.
template <bool kSparse>
struct KeyWalk {
  int lo0, hi0, lo1, hi1, last, n;
  TileSet a, b, u;
  __device__ __forceinline__ int first() const { return kSparse ? u.next(0) : lo0; }
  __device__ __forceinline__ int next(int j) const {
    return kSparse ? u.next(j + 1) : (j + 1 <= last ? j + 1 : n);
  }
  __device__ __forceinline__ bool has(int t, int j) const {
    if (kSparse) return t ? b.has(j) : a.has(j);
    return t ? (j >= lo1 && j <= hi1) : (j >= lo0 && j <= hi0);
  }
  __device__ __forceinline__ int first_of(int t) const {
    if (kSparse) return t ? b.next(0) : a.next(0);
    return t ? (lo1 <= hi1 ? lo1 : n) : (lo0 <= hi0 ? lo0 : n);
  }
  __device__ __forceinline__ int next_of(int t, int j) const {
    if (kSparse) return t ? b.next(j + 1) : a.next(j + 1);
    return j + 1 <= (t ? hi1 : hi0) ? j + 1 : n;
  }
  __device__ __forceinline__ int count_of(int t) const {
    if (kSparse) return t ? b.count() : a.count();
    return t ? max(0, hi1 - lo1 + 1) : max(0, hi0 - lo0 + 1);
  }
};

// One work unit: query tiles 2 pt and 2 pt + 1 of (batch, head) bh.
struct FwdUnit {
  int bh, hh, bb, pt;  // hh, bb: TMA coordinates of (batch, head)
  int lo[2], hi[2];    // key tiles [lo_t, hi_t] of query tile 2 pt + t (lo > hi: none)
  int n_q_here;        // query tiles inside the sequence (1 or 2)
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort_flag) {
  bool ok = mbar_wait(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// The two products in either operand width.
template <bool kFp8>
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                       uint32_t acc) {
  if constexpr (kFp8)
    tc_mma_ss_f8(d, a, b, id, acc);
  else
    tc_mma_ss(d, a, b, id, acc);
}

template <bool kFp8>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                       uint32_t acc) {
  if constexpr (kFp8)
    tc_mma_ts_f8(d, a, b, id, acc);
  else
    tc_mma_ts(d, a, b, id, acc);
}

// kBf16: the 16-bit type of O (and of Q, K, V unless kFp8, where they are
// e4m3 bytes and V arrives transposed).  kResident: the CTAs stay resident
// and take several work units each; otherwise each CTA takes one.
template <int D, bool kBf16, bool kAlibi, bool kSparse, bool kFp8, bool kResident>
__global__ void __launch_bounds__(kFwdThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdLaunch p) {
  // Launched with programmatic stream serialization: the CTAs of one
  // forward start while the previous kernel finishes, and wait here before
  // reading Q, K, V (back-to-back B8 H12 N1024 forwards 33.1 -> 30.3 us).
  pdl_wait_and_release();
  using Smem = FwdSmem<D, kSparse, kFp8>;
  static_assert(!kResident || (Smem::kOwnStage && !kSparse),
                "resident CTAs: dense, O staged apart from Q");
  constexpr int kColsPerBlock = kFp8 ? 128 : 64;  // elements in a 128-byte block
  // 8-bit D = 64: Q and K rows are 64 bytes, in 64-byte-swizzled tiles
  constexpr bool kRows64 = Smem::kRowBytes < 128;
  // P = 2^(x - m + kPOffset) with the reference maximum m lagging the true
  // one by at most kThreshold, so P < 2^(kThreshold + kPOffset) = 256.
  // 16-bit P keeps the largest lag; 8-bit P (e4m3, largest finite 448,
  // subnormal below 2^-6) spends half of it on the offset so that weights
  // down to 2^-10 of the row maximum stay normal.
  constexpr float kThreshold = kFp8 ? 4.0f : 8.0f;
  constexpr float kPOffset = kFp8 ? 4.0f : 0.0f;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int n_q_tiles = (p.N + kTile - 1) / kTile;
  const int n_pairs = (n_q_tiles + 1) / 2;
  const int n_kv = (p.N + kTile - 1) / kTile;
  const long long n_units = static_cast<long long>(n_pairs) * p.BH;
  const int wl = p.band.win_left, wr = p.band.win_right;
  // With keys bounded on the right only (causal), later pairs see more keys:
  // they go first.
  const bool later_longer = wl < 0 && wr >= 0;
  // With G CTAs, CTA c takes unit k G + c in even rounds k and k G + G-1-c in
  // odd ones: one unit each when the grid covers them all; resident CTAs
  // walk the longest-first order back and forth, so that long and short
  // units even out over the rounds.
  auto unit_of = [&](int k) -> long long {
    const long long G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? G - 1 - c : c);
  };
  // (32-bit division when the unit count allows: a 64-bit one is a long
  // instruction sequence, and every role decodes each unit)
  const bool units32 = n_units <= 0xffffffffLL;
  auto decode = [&](long long u, FwdUnit& w) {
    int idx;
    if (units32) {
      const uint32_t u32 = static_cast<uint32_t>(u);
      const uint32_t d = static_cast<uint32_t>(p.tile_major ? p.BH : n_pairs);
      const uint32_t q = u32 / d, rem = u32 - q * d;
      w.bh = static_cast<int>(p.tile_major ? rem : q);
      idx = static_cast<int>(p.tile_major ? q : rem);
    } else {
      w.bh = static_cast<int>(p.tile_major ? u % p.BH : u / n_pairs);
      idx = static_cast<int>(p.tile_major ? u / p.BH : u % n_pairs);
    }
    w.hh = w.bh % p.H;
    w.bb = w.bh / p.H;
    w.pt = later_longer ? n_pairs - 1 - idx : idx;
    // lo and hi never decrease from tile A to B, and each range holds the
    // tile's diagonal, so their union is contiguous.
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int qt = 2 * w.pt + t;
      if (qt >= n_q_tiles) {
        w.lo[t] = 1;
        w.hi[t] = 0;
      } else {
        band_key_tiles(qt * kTile, kTile, kTile, n_kv, wl, wr, w.lo[t], w.hi[t]);
      }
    }
    w.n_q_here = w.hi[1] >= w.lo[1] ? 2 : 1;
  };
  auto walk_of = [&](const FwdUnit& w) {
    return KeyWalk<kSparse>{w.lo[0], w.hi[0], w.lo[1], w.hi[1], max(w.hi[0], w.hi[1]), n_kv,
                            TileSet{s.key_tiles[0], n_kv},
                            TileSet{s.key_tiles[kSparse ? 1 : 0], n_kv},
                            TileSet{s.key_tiles[kSparse ? 2 : 0], n_kv}};
  };
  // Calls fn(k, u) for this CTA's units in order while it returns true.  A
  // CTA with one unit runs it as straight-line code: a loop around the
  // softmax would hold more of its state in registers.
  auto for_each_unit = [&](auto&& fn) {
    if constexpr (kResident) {
      for (int k = 0;; ++k) {
        const long long u = unit_of(k);
        if (u >= n_units || !fn(k, u)) break;
      }
    } else {
      fn(0, static_cast<long long>(blockIdx.x));
    }
  };
  if constexpr (kSparse) {
    // One unit per CTA: the block mask, intersected with each tile's band
    // range.
    FwdUnit w;
    decode(blockIdx.x, w);
    const int qa = 2 * w.pt, qb = 2 * w.pt + 1;
    auto in_a = [&](int j) {
      return j >= w.lo[0] && j <= w.hi[0] && block_kept(p.band, w.bh, p.H, n_kv, qa, j);
    };
    auto in_b = [&](int j) {
      return j >= w.lo[1] && j <= w.hi[1] && block_kept(p.band, w.bh, p.H, n_kv, qb, j);
    };
    fill_tile_set(s.key_tiles[0], n_kv, in_a);
    fill_tile_set(s.key_tiles[1], n_kv, in_b);
    fill_tile_set(s.key_tiles[2], n_kv, [&](int j) { return in_a(j) || in_b(j); });
  }

  if (tid == 0) {
    for (int i = 0; i < Smem::kQSets; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_done[i], 1);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;
  if (warp >= 8) {
    // The producer and MMA warps need few registers: their warpgroup
    // gives some to the softmax warpgroups (warps 10 and 11 only do this).
    setmaxnreg_dec<kFwdLowRegs>();
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&p.map_q);
        tma_prefetch_desc(&p.map_k);
        tma_prefetch_desc(&p.map_v);
        uint32_t kv = 0;      // K/V tiles loaded so far, over all units (ring position)
        int q_rounds = 0;     // Q loads issued
        long long loads = 0;  // K and V loads issued (K of ring position n is load 2n)
        for_each_unit([&](int k, long long u) -> bool {
          FwdUnit w;
          decode(u, w);
          const KeyWalk<kSparse> walk = walk_of(w);
          // The running counters are copied in and out, so that the key-tile
          // loop works on registers.
          uint32_t ring = kv;
          long long n_loads = loads;
          // Unit k's Q goes into set k % kQSets once the last S product of the
          // unit that used the set before has read it.
          const int qs = k % Smem::kQSets, q_use = k / Smem::kQSets;
          if (q_use > 0 && !mbar_wait(&s.q_empty[qs], (q_use - 1) & 1, p.err, abort_flag))
            return false;
          mbar_arrive_expect_tx(&s.q_full[qs], w.n_q_here * Smem::kTileBytes);
          for (int t = 0; t < w.n_q_here; ++t)
            for (int kb = 0; kb < Smem::kBlocks; ++kb)
              tma_load_4d(s.q[qs][t] + kb * Smem::kBlockBytes, &p.map_q, &s.q_full[qs],
                          kb * kColsPerBlock, (2 * w.pt + t) * kTile, w.hh, w.bb);
          q_rounds = k + 1;
          bool stop = false;
          for (int j = walk.first(); j < walk.n; j = walk.next(j), ++ring) {
            const int st = ring & 1;
            const uint32_t use = ring >> 1;  // earlier uses of this stage
            if (ring >= 2 && !mbar_wait(&s.k_empty[st], (use - 1) & 1, p.err, abort_flag)) {
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&s.k_full[st], Smem::kTileBytes);
            for (int kb = 0; kb < Smem::kBlocks; ++kb)
              tma_load_4d(s.k[st] + kb * Smem::kBlockBytes, &p.map_k, &s.k_full[st],
                          kb * kColsPerBlock, j * kTile, w.hh, w.bb);
            ++n_loads;
            if (ring >= 2 && !mbar_wait(&s.v_empty[st], (use - 1) & 1, p.err, abort_flag)) {
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&s.v_full[st], Smem::kTileBytes);
            if constexpr (kFp8) {
              // V^T rows d = 0..D-1, keys j*128 .. j*128+127
              tma_load_4d(s.v[st], &p.map_v, &s.v_full[st], j * kTile, 0, w.hh, w.bb);
            } else {
              for (int kb = 0; kb < Smem::kBlocks; ++kb)
                tma_load_4d(s.v[st] + kb * Smem::kBlockBytes, &p.map_v, &s.v_full[st], kb * 64,
                            j * kTile, w.hh, w.bb);
            }
            ++n_loads;
          }
          kv = ring;
          loads = n_loads;
          return !stop;
        });
        if (*abort_flag) {
          // Let copies already in flight land before the CTA's smem goes away.
          int zero = 0;
          for (int r = max(0, q_rounds - Smem::kQSets); r < q_rounds; ++r)
            mbar_wait(&s.q_full[r % Smem::kQSets], (r / Smem::kQSets) & 1, p.err, &zero,
                      100000000ull);
          for (long long t = loads > 4 ? loads - 4 : 0; t < loads; ++t) {
            const long long n = t >> 1;  // ring position
            const int st = static_cast<int>(n & 1);
            mbar_wait((t & 1) ? &s.v_full[st] : &s.k_full[st], static_cast<uint32_t>((n >> 1) & 1),
                      p.err, &zero, 100000000ull);
          }
        }
      }
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // 16-bit operands: every lane computes the same descriptors and waits
      // on the same barriers; only the elected lane issues.  (A single-lane
      // branch made each product's operands per-thread values to be moved into
      // uniform registers first: issuing a group's sixteen products then took
      // longer than the tensor core took to run them.)  8-bit operands keep
      // the single-lane loop.
      if (!kFp8 || lane == 0) {
        const bool leader = kFp8 ? true : elect_one_sync();
        auto leader_commit = [&](uint64_t* bar) {
          if (leader) tc_commit(bar);
        };
        constexpr uint32_t ab = kBf16 ? 1u : 0u;
        constexpr uint32_t idS = kFp8 ? idesc_e4m3(128, 128) : idesc_f16(128, 128, ab, 0, 0);
        // P V: 16-bit V is MN-major (D contiguous); 8-bit V^T is K-major
        constexpr uint32_t idPV = kFp8 ? idesc_e4m3(128, D) : idesc_f16(128, D, ab, 0, 1);
        // Operand descriptors are built once and advanced by constant offsets.
        const uint64_t dq0 = kRows64 ? smem_desc_sw64(smem_u32(s.q[0][0]), 16, 512)
                                     : smem_desc_sw128(smem_u32(s.q[0][0]), 16, 1024);
        const uint64_t dk0 = kRows64 ? smem_desc_sw64(smem_u32(s.k[0]), 16, 512)
                                     : smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
        const uint64_t dv0 =
            smem_desc_sw128(smem_u32(s.v[0]), kFp8 ? 16 : Smem::kBlockBytes, 1024);
        // One product step covers 32 bytes of each row: 16 elements of 16 bits,
        // 32 of 8 bits.
        constexpr int kStepElems = kFp8 ? 32 : 16;
        // P step kk of V tile stage st: 16-bit V advances kStepElems rows of
        // 128 bytes, 8-bit V^T 32 bytes within each row.
        auto v_step = [](uint64_t dv, int kk) {
          return kFp8 ? desc_add(dv, kk * 32) : desc_add(dv, kk * kStepElems * 128);
        };
        uint32_t kv_run = 0;              // K/V tiles of earlier units (ring position)
        int base0_run = 0, base1_run = 0;  // P V products of tiles A, B in earlier units
        for_each_unit([&](int k, long long u) -> bool {
          FwdUnit w;
          decode(u, w);
          const KeyWalk<kSparse> walk = walk_of(w);
          const int qs = k % Smem::kQSets, q_use = k / Smem::kQSets;  // this unit's Q set
          // register copies of the running counters for this unit's loops
          const uint32_t kv = kv_run;
          const int base0 = base0_run, base1 = base1_run;
          // S products of this unit still to issue; with resident CTAs the
          // last one's commit hands the Q buffers to the next unit's loads.
          [[maybe_unused]] int s_left = walk.count_of(0) + walk.count_of(1);
          // S_t = Q_t K^T into tile t's S columns, K from stage kst
          auto issue_s = [&](int t, int kst) {
            const uint64_t dq = desc_add(dq0, (qs * 2 + t) * Smem::kTileBytes);
            const uint64_t dk = desc_add(dk0, kst * Smem::kTileBytes);
  #pragma unroll
            for (int kk = 0; kk < Smem::kRowBytes / 32; ++kk) {
              const uint32_t off = (kk >> 2) * Smem::kBlockBytes + (kk & 3) * 32;
              if (leader) mma_ss<kFp8>(tbase + t * 128, desc_add(dq, off), desc_add(dk, off), idS,
                           kk > 0 ? 1u : 0u);
            }
            leader_commit(&s.s_full[t]);
            if constexpr (kResident)
              if (--s_left == 0) leader_commit(&s.q_empty[qs]);
          };
          const int jf = walk.first();
          // with nothing to multiply (an empty block-sparse pair) no K arrives
          bool ok = mbar_wait_poll(&s.q_full[qs], q_use & 1, p.err, abort_flag) &&
                    (jf >= walk.n || mbar_wait_poll(&s.k_full[kv & 1], (kv >> 1) & 1, p.err, abort_flag));
          if (!ok) return false;
          if (jf >= walk.n) {
            if constexpr (kResident) leader_commit(&s.q_empty[qs]);
            return true;
          }
          tc_fence_after();
          for (int t = 0; t < 2; ++t)
            if (walk.has(t, jf)) issue_s(t, kv & 1);
          leader_commit(&s.k_empty[kv & 1]);
          int n_stream = 0;  // key tiles in this unit's K/V stream
          if constexpr (!kSparse) {
            // dense: each tile's key tiles are the range [lo_t, hi_t]
            const int j_first = jf, j_last = walk.last;
            for (int j = j_first; ok && j <= j_last; ++j) {
              const uint32_t g = kv + static_cast<uint32_t>(j - j_first);  // ring position of j
              const int st = g & 1;
              if (!mbar_wait_poll(&s.v_full[st], (g >> 1) & 1, p.err, abort_flag)) {
                ok = false;
                break;
              }
              bool k_next = false;  // K_{j+1} has landed
              for (int t = 0; ok && t < 2; ++t) {
                // (selects, not indexing: a dynamic index would put w in local memory)
                const int lt = t ? w.lo[1] : w.lo[0], ht = t ? w.hi[1] : w.hi[0];
                const bool active = j >= lt && j <= ht;
                // S_t(j+1) is next: after PV_t(j), or as the first product of
                // a tile whose range starts at j + 1
                const bool s_next = active ? j + 1 <= ht : (j + 1 == lt && lt <= ht);
                if (active) {
                  if (!mbar_wait_poll(&s.p_full[t], ((t ? base1 : base0) + j - lt) & 1, p.err,
                                 abort_flag)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  // O_t += P_t(j) V_j, with P read from tile t's S columns
                  const uint64_t dv = desc_add(dv0, st * Smem::kTileBytes);
  #pragma unroll
                  for (int kk = 0; kk < kTile / kStepElems; ++kk)
                    if (leader) mma_ts<kFp8>(tbase + 256 + t * D, tbase + t * 128 + kk * 8, v_step(dv, kk),
                                 idPV, (j > lt || kk > 0) ? 1u : 0u);
                  leader_commit(&s.o_done[t]);
                }
                if (s_next) {
                  if (!k_next) {
                    if (!mbar_wait_poll(&s.k_full[(g + 1) & 1], ((g + 1) >> 1) & 1, p.err,
                                   abort_flag)) {
                      ok = false;
                      break;
                    }
                    tc_fence_after();
                    k_next = true;
                  }
                  issue_s(t, (g + 1) & 1);  // after the PV product that read P_t(j)
                }
              }
              leader_commit(&s.v_empty[st]);
              if (k_next) leader_commit(&s.k_empty[(g + 1) & 1]);
            }
            n_stream = j_last - j_first + 1;
          } else {
            // block-sparse: each tile's key tiles are a set; counters give the
            // p_full phases
            int c0 = 0, c1 = 0;  // P V products issued for tile A, B
            for (int j = jf, jn = 0; ok && j < walk.n; j = jn, ++n_stream) {
              jn = walk.next(j);  // the stream's next key tile
              const uint32_t g = kv + static_cast<uint32_t>(n_stream);
              const int st = g & 1;
              if (!mbar_wait_poll(&s.v_full[st], (g >> 1) & 1, p.err, abort_flag)) {
                ok = false;
                break;
              }
              bool k_next = false;  // K of tile jn has landed
              for (int t = 0; ok && t < 2; ++t) {
                const bool active = walk.has(t, j);
                // S_t of tile jn follows PV_t(j), or starts a tile that joins at jn
                const bool s_next = jn < walk.n && walk.has(t, jn);
                if (active) {
                  const int ct = t ? c1 : c0;
                  if (!mbar_wait_poll(&s.p_full[t], ((t ? base1 : base0) + ct) & 1, p.err, abort_flag)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  // O_t += P_t(j) V_j, with P read from tile t's S columns
                  const uint64_t dv = desc_add(dv0, st * Smem::kTileBytes);
  #pragma unroll
                  for (int kk = 0; kk < kTile / kStepElems; ++kk)
                    if (leader) mma_ts<kFp8>(tbase + 256 + t * D, tbase + t * 128 + kk * 8, v_step(dv, kk),
                                 idPV, (ct > 0 || kk > 0) ? 1u : 0u);
                  leader_commit(&s.o_done[t]);
                  if (t)
                    ++c1;
                  else
                    ++c0;
                }
                if (s_next) {
                  if (!k_next) {
                    if (!mbar_wait_poll(&s.k_full[(g + 1) & 1], ((g + 1) >> 1) & 1, p.err,
                                   abort_flag)) {
                      ok = false;
                      break;
                    }
                    tc_fence_after();
                    k_next = true;
                  }
                  issue_s(t, (g + 1) & 1);  // after the PV product that read P_t(j)
                }
              }
              leader_commit(&s.v_empty[st]);
              if (k_next) leader_commit(&s.k_empty[(g + 1) & 1]);
            }
          }
          kv_run = kv + static_cast<uint32_t>(n_stream);
          base0_run = base0 + walk.count_of(0);
          base1_run = base1 + walk.count_of(1);
          return ok;
        });
        // Every MMA issued above completes before TMEM is released.
        leader_commit(&s.drain);
        int zero = 0;
        mbar_wait(&s.drain, 0, p.err, &zero, 100000000ull);
      }
    }
  } else {
    setmaxnreg_inc<kFwdHighRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;          // query tile of this group (0 = A, 1 = B)
    const int r = tid & 127;          // row within the tile and TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + t * 128, tO = tbase + 256 + t * D;
    int base_run = 0;  // key tiles of this query tile in earlier units (barrier phases)
    for_each_unit([&](int k, long long u) -> bool {
      const int base = base_run;
      FwdUnit w;
      decode(u, w);
      const KeyWalk<kSparse> walk = walk_of(w);
      const int bh = w.bh, hh = w.hh, bb = w.bb;
      const int q0 = (2 * w.pt + t) * kTile;
      const int i = q0 + r;
      const int n_tiles = walk.count_of(t);
      const float nslope2 = kAlibi ? alibi_nslope2(p.band, bh, p.H) : 0.f;
      // 8-bit operands carry per-(batch, head) dequantisation factors: Q and K
      // scale the scores, V scales O.
      float sl2 = p.scale_log2, v_descale = 1.f;
      if constexpr (kFp8) {
        if (p.descale_q) sl2 *= p.descale_q[bh];
        if (p.descale_k) sl2 *= p.descale_k[bh];
        if (p.descale_v) v_descale = p.descale_v[bh];
      }
      const bool pos_scale = sl2 > 0.f;
      float m = -INFINITY;  // reference maximum, log2 units
      float l = 0.f;        // running sum of 2^(t - m), the LSE's
      // The sum O is divided by, for 16-bit P.  O is made of P values
      // rounded to 8 (bf16) or 11 (fp16) bits; dividing by their exact sum
      // l would move O by the rounding of P times the V rows themselves,
      // which is 2^-8 |V| where one key dominates a row: with a lagging
      // reference maximum that key's P lies anywhere in [1, 256).  So lo
      // takes the rounded value of each tile's largest P instead of its
      // exact one, and, on tiles the mask cuts in a query tile whose rows
      // see at most 128 keys (where every weight can be large), the rounded
      // value of every P: the weights that dominate O then sum to one as
      // rounded.  The LSE keeps the exact sum l.
      float lo = 0.f;
      const bool few_keys = [&] {
        // the visible-key count of row i is concave in i: its minimum over
        // the tile is at an end row (block masks that drop tiles: few)
        if (kSparse && walk.count_of(t) < (t ? w.hi[1] - w.lo[1] : w.hi[0] - w.lo[0]) + 1)
          return true;
        auto count = [&](int row) {
          const int first = wl < 0 ? 0 : max(0, row - wl);
          const int last = min(p.N - 1, wr < 0 ? p.N - 1 : row + wr);
          return last - first + 1;
        };
        return min(count(q0), count(min(q0 + kTile, p.N) - 1)) <= kTile;
      }();
      bool ok = true;
      for (int jj = 0, j = walk.first_of(t); jj < n_tiles; ++jj, j = walk.next_of(t, j)) {
        if (!warp_wait(&s.s_full[t], (base + jj) & 1, p.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kTile];
        {
          // All four loads in flight before the single wait.
          uint32_t raw[kTile / 32][32];
#pragma unroll
          for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tS + lane_off + c * 32, raw[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kTile / 32; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) sv[c * 32 + e] = __uint_as_float(raw[c][e]);
        }
        // Scores -> log2 units.  With a positive scale and no bias this is
        // folded into the exponent below (one packed FMA per two scores);
        // otherwise scale (and add the ALiBi bias) first.
        const int k0 = j * kTile;
        const bool prescale = kAlibi || !pos_scale;
        if (kAlibi) {
          const float d0 = static_cast<float>(k0 - i);  // key - query at column 0 (exact)
          const bool below = k0 + kTile - 1 <= q0, above = k0 >= q0 + kTile - 1;
          if (below || above) {
            // The whole tile lies on one side of the diagonal: |key - i| is
            // linear in the column, so the bias is B + D c, two columns per
            // packed FMA.
            const float sd = above ? nslope2 : -nslope2;
            const uint64_t b2 = f32x2(sd * d0, sd * d0), dd2 = f32x2(sd, sd), s2 = f32x2(sl2, sl2);
#pragma unroll
            for (int c = 0; c < kTile; c += 2) {
              const uint64_t bias = fma_f32x2(f32x2(static_cast<float>(c), static_cast<float>(c + 1)),
                                              dd2, b2);
              const float2 x = split_f32x2(fma_f32x2(f32x2(sv[c], sv[c + 1]), s2, bias));
              sv[c] = x.x;
              sv[c + 1] = x.y;
            }
          } else {
#pragma unroll
            for (int c = 0; c < kTile; ++c)
              sv[c] = fmaf(sv[c], sl2, nslope2 * fabsf(d0 + static_cast<float>(c)));
          }
        } else if (!pos_scale) {
#pragma unroll
          for (int c = 0; c < kTile; ++c) sv[c] *= sl2;
        }
        const bool masked =
            band_cuts(q0, kTile, k0, kTile, p.band.win_left, p.band.win_right) || k0 + kTile > p.N;
        if (masked) {
          // this row's visible keys are first .. last
          const int wl_ = p.band.win_left, wr_ = p.band.win_right;
          const int first = wl_ < 0 ? 0 : i - wl_;
          const int last = min(p.N - 1, wr_ < 0 ? p.N - 1 : i + wr_);
          const int cf = first - k0, cl = last - k0;  // visible columns cf .. cl
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (c < cf || c > cl) sv[c] = -INFINITY;
        }
        // Row maximum: eight independent chains of three-input max.
        float mxs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxs[e] = sv[e];
#pragma unroll
        for (int c = 8; c < kTile; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            mxs[e] = c + 8 < kTile ? fmax3(mxs[e], sv[c + e], sv[c + 8 + e]) : fmaxf(mxs[e], sv[c + e]);
        const float mx = fmax3(fmax3(mxs[0], mxs[1], mxs[2]), fmax3(mxs[3], mxs[4], mxs[5]),
                               fmaxf(mxs[6], mxs[7]));
        const float m_tile = prescale ? mx : mx * sl2;
        const float m_new = fmaxf(m, m_tile);
        const bool need = m_new > m + kThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
          l *= alpha;
          lo *= alpha;
          m = m_new;
        }
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
          // O currently holds sum_{j' < j} P V; it must be final before scaling.
          if (!warp_wait(&s.o_done[t], (base + jj - 1) & 1, p.err, abort_flag)) {
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
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
        const float mneg = (m == -INFINITY) ? 0.f : kPOffset - m;
        // P = 2^(x * mult - m), two columns per packed FMA / add; the softmax
        // warps share issue slots with the MMA warp, so fewer instructions
        // here keep the tensor core fed.
        const float mult = prescale ? 1.f : sl2;
        const uint64_t mult2 = f32x2(mult, mult), mneg2 = f32x2(mneg, mneg);
        // the tile's largest P as the loop below computes it, and as rounded
        float pmax_corr = 0.f;
        if constexpr (!kFp8) {
          const float pmax = ex2_approx(fmaf(mx, mult, mneg));
          pmax_corr = unpack2<kBf16>(pack2<kBf16>(pmax, 0.f)).x - pmax;
        }
        uint64_t sums[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};  // independent partial row sums
        uint32_t pk8[kFp8 ? 32 : 1];  // 8-bit P: four keys per column
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 z = split_f32x2(
                fma_f32x2(f32x2(sv[h * 64 + 2 * c], sv[h * 64 + 2 * c + 1]), mult2, mneg2));
            const float p0 = ex2_approx(z.x), p1 = ex2_approx(z.y);
            sums[c & 1] = add_f32x2(sums[c & 1], f32x2(p0, p1));
            if constexpr (kFp8) {
              const uint32_t b2 = pack2_e4m3(p0, p1);
              if (c & 1)
                pk8[h * 16 + (c >> 1)] |= b2 << 16;
              else
                pk8[h * 16 + (c >> 1)] = b2;
            } else {
              pk[c] = pack2<kBf16>(p0, p1);
            }
          }
          if constexpr (!kFp8) tmem_st32(tS + lane_off + h * 32, pk);
        }
        if constexpr (kFp8) tmem_st32(tS + lane_off, pk8);
        const float2 s0 = split_f32x2(sums[0]), s1 = split_f32x2(sums[1]);
        const float tile_sum = (s0.x + s0.y) + (s1.x + s1.y);
        l += tile_sum;
        if constexpr (kFp8) {
          lo += tile_sum;
        } else if (masked && few_keys) {
          // every P as rounded, read back from TMEM (rare tiles: the
          // registers of the loop above are free by now)
          tmem_st_wait();
          uint64_t rs = f32x2(0.f, 0.f);
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t pr[32];
            tmem_ld32(tS + lane_off + h * 32, pr);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float2 q2 = unpack2<kBf16>(pr[c]);
              rs = add_f32x2(rs, f32x2(q2.x, q2.y));
            }
          }
          const float2 r2 = split_f32x2(rs);
          lo += r2.x + r2.y;
        } else {
          lo += tile_sum + pmax_corr;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&s.p_full[t]);
      }

      // ---------------------------------------------------------- epilogue
      // Every thread of the group takes the same branch (a timeout in one warp
      // must not leave the others waiting at the barrier below), and the same
      // decision to go on to the next unit.
      bool group_ok = ok;
      if (q0 < p.N) {
        // A tile the block mask empties has O = 0 and LSE = -inf; its smem
        // stage may be written once its Q load has landed.
        const bool have = n_tiles > 0;
        const bool mine =
            ok && (have ? warp_wait(&s.o_done[t], (base + n_tiles - 1) & 1, p.err, abort_flag)
                        : warp_wait(&s.q_full[k % Smem::kQSets], (k / Smem::kQSets) & 1, p.err,
                                    abort_flag));
        group_ok = named_bar_and(1 + t, 128, mine);
        if (group_ok) {
          tc_fence_after();
          const float inv_l = lo > 0.f ? v_descale / lo : 0.f;
          // 16-bit D = 128: this tile's Q is no longer read
          uint8_t* stage = Smem::kOwnStage ? s.o[t] : s.q[0][t];
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (have) {
              tmem_ld32(tO + lane_off + c * 32, o);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack2<kBf16>(__uint_as_float(o[2 * e]) * inv_l,
                                   __uint_as_float(o[2 * e + 1]) * inv_l);
            // 32 columns = four 16-byte chunks of this row, 128-byte swizzle
            uint8_t* blk = stage + (c >> 1) * Smem::kOBlockBytes + r * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const int cc = (c & 1) * 4 + ch;
              *reinterpret_cast<uint4*>(blk + ((cc ^ (r & 7)) * 16)) =
                  make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + t, 128);
          if (r == 0) {
            for (int kb = 0; kb < Smem::kOBlocks; ++kb)
              tma_store_4d(&p.map_o, stage + kb * Smem::kOBlockBytes, kb * 64, q0, hh, bb);
            tma_store_commit();
            tma_store_wait_all();
          }
          if (i < p.N)
            p.lse[static_cast<long long>(bh) * p.N + i] =
                have ? (m - kPOffset + lg2_approx(l)) * kLn2 : -INFINITY;
        }
      }
      base_run = base + n_tiles;
      return group_ok;
    });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool kBf16, bool kAlibi, bool kSparse, bool kFp8, bool kResident>
cudaError_t launch_fwd_grid(const FwdLaunch& b, long long grid, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, kBf16, kAlibi, kSparse, kFp8, kResident>;
  const int smem = static_cast<int>(sizeof(FwdSmem<D, kSparse, kFp8>)) + 1024;
  static AttrCache configured;
  cudaError_t e = ensure_dynamic_smem(kern, smem, configured);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, static_cast<unsigned>(grid), kFwdThreads, smem, stream, b);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, bool kBf16, bool kAlibi, bool kSparse, bool kFp8 = false>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  const long long n_q_tiles = (a.N + kTile - 1) / kTile;
  const long long units = (n_q_tiles + 1) / 2 * a.BH;
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  FwdLaunch b = a;  // streamed per head: K and V
  b.tile_major = tile_major_order(a.band, 2LL * a.BH * a.N * a.D * (kFp8 ? 1 : 2));
  // Resident CTAs, one per SM, for short sequences (at most 32 key tiles)
  // with more units than SMs; the next unit's loads need the O staging of
  // their own.
  if constexpr (FwdSmem<D, kSparse, kFp8>::kOwnStage && !kSparse) {
    if (n_q_tiles <= 32) {
      int sms = 0;
      const cudaError_t e = sm_count(&sms);
      if (e != cudaSuccess) return e;
      if (units > sms) return launch_fwd_grid<D, kBf16, kAlibi, kSparse, kFp8, true>(b, sms, stream);
    }
  }
  return launch_fwd_grid<D, kBf16, kAlibi, kSparse, kFp8, false>(b, units, stream);
}

// V^T for the 8-bit forward: the P V product wants its B operand K-major
// (keys contiguous), so each (batch, head)'s [N, D] byte matrix is rewritten
// as [D, ld] once per call.  A CTA (D / 16 warps) moves one 128-key x D-column
// tile; warp w takes columns 16w .. 16w+15, lane l keys 4l .. 4l+3: four
// 16-byte row loads, a 4 x 4 byte transpose per word (byte permutes) and
// sixteen 4-byte stores, each warp-wide store covering 128 consecutive bytes
// of one V^T row.
__global__ void __launch_bounds__(256) transpose_v8_kernel(const uint8_t* __restrict__ v,
                                                           RowStrides sv, uint8_t* __restrict__ vt,
                                                           int N, long long ld, int H, int D,
                                                           int n_key_tiles) {
  const int bh = static_cast<int>(blockIdx.x / n_key_tiles);
  const int k0 = static_cast<int>(blockIdx.x % n_key_tiles) * kTile;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const long long b = bh / H, h = bh % H;
  const uint8_t* src = v + b * sv.batch + h * sv.head + w * 16;
  uint4 row[4];  // keys k0 + 4l + i, columns 16w .. 16w+15
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = k0 + 4 * l + i;
    row[i] = key < N ? __ldg(reinterpret_cast<const uint4*>(src + key * sv.seq))
                     : make_uint4(0u, 0u, 0u, 0u);
  }
  const int kg = k0 + 4 * l;  // first key of this lane's group (a multiple of 4)
  if (kg >= ld) return;       // ld is a multiple of 16: the group lies wholly inside
  uint8_t* dst = vt + static_cast<long long>(bh) * D * ld + kg;
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // columns 16w + 4c .. 16w + 4c + 3
    const uint32_t w0 = (&row[0].x)[c], w1 = (&row[1].x)[c], w2 = (&row[2].x)[c],
                   w3 = (&row[3].x)[c];
    // rows of keys -> rows of columns
    const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w0, w1, 0x7362);
    const uint32_t t2 = __byte_perm(w2, w3, 0x5140), t3 = __byte_perm(w2, w3, 0x7362);
    const uint32_t out[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                             __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(16 * w + 4 * c + e) * ld) = out[e];
  }
}

}  // namespace

cudaError_t launch_transpose_v8(const void* v, RowStrides sv, void* vt, int N, long long ld, int H,
                                long long BH, int D, cudaStream_t s) {
  if ((D != 64 && D != 128) || ld < N || (ld & 15) != 0) return cudaErrorInvalidValue;
  const long long tiles = (N + kTile - 1) / kTile;
  if (tiles * BH > INT_MAX) return cudaErrorInvalidConfiguration;
  transpose_v8_kernel<<<static_cast<unsigned>(tiles * BH), D * 2, 0, s>>>(
      static_cast<const uint8_t*>(v), sv, static_cast<uint8_t*>(vt), N, ld, H, D,
      static_cast<int>(tiles));
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd8_d(const FwdLaunch& a, cudaStream_t s) {
  const bool alibi = a.band.alibi != nullptr, sparse = a.band.block_mask != nullptr;
  if (sparse)
    return alibi ? launch_fwd_t<D, true, true, true, true>(a, s)
                 : launch_fwd_t<D, true, false, true, true>(a, s);
  return alibi ? launch_fwd_t<D, true, true, false, true>(a, s)
               : launch_fwd_t<D, true, false, false, true>(a, s);
}

template <int D, bool kBf16>
cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t s) {
  const bool alibi = a.band.alibi != nullptr, sparse = a.band.block_mask != nullptr;
  if (sparse)
    return alibi ? launch_fwd_t<D, kBf16, true, true>(a, s) : launch_fwd_t<D, kBf16, false, true>(a, s);
  return alibi ? launch_fwd_t<D, kBf16, true, false>(a, s) : launch_fwd_t<D, kBf16, false, false>(a, s);
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s) {
  if (a.fp8) {
    if (!a.bf16) return cudaErrorInvalidValue;
    return a.D == 64 ? launch_fwd8_d<64>(a, s) : launch_fwd8_d<128>(a, s);
  }
  if (a.D == 64) return a.bf16 ? launch_fwd_d<64, true>(a, s) : launch_fwd_d<64, false>(a, s);
  return a.bf16 ? launch_fwd_d<128, true>(a, s) : launch_fwd_d<128, false>(a, s);
}

}  // namespace fa
