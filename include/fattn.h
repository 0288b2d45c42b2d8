/*
 * fattn.h -- libfattn: exact tiled attention on one sm_103a GPU (C ABI).
 *
 * Computes O = softmax(scale * Q K^T [+ causal mask]) V exactly, tile by tile
 * with an online softmax, and its gradients by recomputing P from Q, K and
 * the saved per-row log-sum-exp instead of storing the N x N matrix.
 *
 * Sources for what is computed (the pages this library follows):
 *   [WALK] "FlashAttention from scratch in PyTorch" walkthrough (l189.com
 *          news 1255901): sec. 1.1 standard attention, sec. 2.2 online
 *          softmax, sec. 2.4 tiling loop, sec. 3.1 forward with the saved
 *          log-sum-exp, sec. 3.3 recompute backward and softmax Jacobian,
 *          sec. 5.2 fp32 statistics, sec. 5.3 causal mask.
 *   [DEEP] "FlashAttention 深入" (LLM interview guide): online softmax,
 *          backward recomputation, v2 sequence-dimension parallelism.
 *   [API]  claire-chang.com FlashAttention introduction: the flash_attn_func
 *          argument list (softmax_scale, causal, deterministic).
 *   [WIKI] "Flash Attention" wiki page (aiboss88.com): implementation
 *          section, FlashAttention-3's FP8 forward; [DEEP] v1 -> v3 table
 *          (v3 adds FP8).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *   Layout   Q, K, V, O, dO, dQ, dK, dV are [B, H, N, D] arrays of 16-bit
 *            floats, D innermost ([WALK] sec. 1.1, "Q, K, V: (batch, heads,
 *            seq_len, dim)"): contiguous for the plain entry points, any
 *            strides (fa_layout) for the *_strided ones.  LSE and Di are
 *            contiguous fp32 [B, H, N].
 *            Q, K and V share N (self-attention).
 *   Types    FA_BF16 or FA_FP16, the same for every 16-bit array of a call.
 *            Accumulation and softmax statistics are fp32 ([WALK] sec. 5.2).
 *   Shapes   B, H, N >= 1; D is 64 or 128; B * H <= 2^31 - 1 and
 *            B * H * N * D < 2^40.
 *   Pointers Device pointers, 16-byte aligned (TMA requirement).  The caller
 *            owns every buffer; the library allocates no device memory.
 *   Streams  `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *            call only enqueues work and returns; results are ready once the
 *            stream reaches that point.
 *   Errors   Arguments are checked before anything is enqueued.  A failed
 *            check returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED and
 *            enqueues nothing.  A failed launch returns FA_ERR_CUDA.  Kernels
 *            bound every internal wait; a wait that runs out records
 *            FA_ERR_TIMEOUT in a device-side error word that fa_device_error()
 *            reads.
 *   Threads  Calls may come from several host threads; the only shared state
 *            is the device error word and the lazily fetched driver entry
 *            point for building TMA descriptors.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size, bad scale   */
  FA_ERR_UNSUPPORTED = 2, /* D not in {64, 128}, unknown dtype               */
  FA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed              */
  FA_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait                */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/* Version of this interface (incremented on any signature change). */
int fa_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(fa_status s);

/*
 * Element strides of one [B, H, N, D] operand whose D elements are
 * contiguous: element (b, h, n, d) lives at base + b*batch + h*head + n*seq + d
 * (in elements, not bytes).  The contiguous layout is {H*N*D, N*D, D}; the
 * [API] flash_attn_func layout (batch, seqlen, nheads, headdim) is
 * {N*H*D, D, H*D}; a packed (batch, seqlen, 3, nheads, headdim) QKV tensor
 * gives Q, K and V with {3*N*H*D, D, 3*H*D} at offsets 0, H*D and 2*H*D.
 * Each stride must be a non-negative multiple of 8 (16 bytes, a TMA rule),
 * and every element must lie less than 2^40 bytes from its base.
 * Outputs must not overlap each other or themselves (not checked).
 */
typedef struct {
  long long batch, head, seq;
} fa_strides;

/* The strides of every operand of a call.  fa_fwd_strided reads q, k, v and
 * o; fa_bwd_strided reads all eight.  LSE, Di and the workspace keep their
 * fixed contiguous layouts. */
typedef struct {
  fa_strides q, k, v, o, dO, dq, dk, dv;
} fa_layout;

/*
 * Options of flash_attn_func beyond causal ([API]):
 *   window_left, window_right  sliding-window local attention: query i sees
 *                              keys i - left .. i + right inclusive; -1 is
 *                              no bound on that side, (-1, -1) is full
 *                              attention.  Values below -1 are invalid.
 *                              With causal != 0 the window is intersected
 *                              with the causal mask.
 *   alibi_slopes               NULL, or a device array of fp32 slopes, [H]
 *                              (alibi_per_batch = 0) or [B, H] (= 1): the
 *                              score of query i and key j gets
 *                              -slope * |i - j| added after scaling.
 *                              4-byte aligned; read by the kernels, not
 *                              validated.
 *   block_mask                 NULL, or a device array of bytes over blocks
 *                              of 128 x 128 scores, [T][T] for every head
 *                              (block_mask_per_head = 0) or [H][T][T] (= 1),
 *                              T = ceil(N / 128): query block a multiplies
 *                              key block b only when the byte [a][b] is
 *                              nonzero (block-sparse attention, the
 *                              extension [DEEP] and [WALK] report).  It
 *                              combines with causal, the window and ALiBi;
 *                              a row left with no visible key gets O = 0,
 *                              LSE = -inf and no gradient.  T may be at most
 *                              16384 (FA_ERR_UNSUPPORTED beyond).
 */
typedef struct {
  int window_left, window_right;
  const float* alibi_slopes;
  int alibi_per_batch;
  const unsigned char* block_mask;
  int block_mask_per_head;
} fa_options;

/*
 * Forward pass ([WALK] sec. 2.4 and 3.1; [DEEP] online softmax).
 *
 *   o[b,h,i,:]  = sum_j P_ij V[b,h,j,:],  P = softmax_j(scale * Q_i . K_j)
 *   lse[b,h,i]  = ln sum_j exp(scale * Q_i . K_j)   (natural log, scaled scores)
 *
 * With causal != 0 query i sees keys j <= i only ([WALK] sec. 5.3); tiles
 * above the diagonal are skipped.  `scale` must be finite (the usual value is
 * 1/sqrt(D), [API] softmax_scale default).  Writes o and lse only.
 * Deterministic: the same inputs give bit-identical outputs.
 *
 * The forward kernel (of every fa_fwd* call) is launched with programmatic
 * stream serialization: its CTAs may start while the preceding kernel in
 * the stream finishes, and wait for that kernel's completion before
 * reading anything.  Stream order is kept for every caller; a following
 * kernel that itself allows overlap must, as always, wait
 * (cudaGridDependencySynchronize) before reading o or lse.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int D, float scale, int causal, fa_dtype dtype, void* stream);

/*
 * fa_fwd on operands in any layout described by `layout` (see fa_strides);
 * the arithmetic, and so the result, is bit-identical to fa_fwd on the same
 * values stored contiguously.  layout == NULL or a bad stride returns
 * FA_ERR_INVALID_ARG before anything is enqueued.
 */
fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int D, const fa_layout* layout, float scale, int causal,
                         fa_dtype dtype, void* stream);

/*
 * The general forward: operands in `layout` (NULL: contiguous) and the
 * window / ALiBi `options` (NULL: none).  fa_fwd and fa_fwd_strided are
 * this with NULL options.  A bad window bound or a misaligned slope pointer
 * returns FA_ERR_INVALID_ARG before anything is enqueued.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int N, int D, const fa_layout* layout, const fa_options* options,
                    float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Workspace bytes fa_fwd_fp8 needs: B*H*D*ld bytes (V transposed, ld = N
 * rounded up to 16), rounded up to 256.  Returns 0 for invalid sizes
 * (D not in {64, 128} included).
 */
size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int D);

/*
 * FP8 forward ([WIKI] implementation section; [DEEP] v3): fa_fwd_ex with Q,
 * K and V given as e4m3 bytes (OCP FP8 E4M3: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, largest finite 448, no infinities) and
 * per-(batch, head) dequantisation factors:
 *
 *   Q~ = descale_q[b,h] * Q,  K~ = descale_k[b,h] * K,  V~ = descale_v[b,h] * V
 *   o, lse = the fa_fwd_ex result for Q~, K~, V~   (o in bf16)
 *
 *   q, k, v     device, e4m3 bytes [B, H, N, D] in `layout` (strides in
 *               bytes, multiples of 16; NULL: contiguous).  D is 64 or 128
 *               (FA_ERR_UNSUPPORTED otherwise).
 *   o           device, bf16 [B, H, N, D] in layout->o (elements, multiples
 *               of 8).   lse: device fp32 [B, H, N], natural log.
 *   descale_*   NULL (factor 1) or device fp32 [B][H], 4-byte aligned, read
 *               by the kernels and not validated (finite values expected).
 *   options     window, ALiBi and block mask exactly as for fa_fwd_ex.
 *   workspace   device, fa_fwd_fp8_workspace_size(...) bytes, 256-byte
 *               aligned; overwritten (it holds V transposed to [B,H,D,ld]).
 *
 * Scores and the softmax statistics are exact products accumulated in
 * fp32, as for 16-bit inputs.  The probabilities P enter the P V product
 * rounded to e4m3, each relative to the row maximum known when its tile is
 * processed and scaled by a power of two so that weights down to 2^-10 of
 * that maximum stay normal; the row sum uses the unrounded P.  So o differs
 * from the exact result by at most about 2^-4 of sum_j P_ij |V~_jd| (the
 * e4m3 half-ulp) plus the bf16 rounding of o; lse carries no P rounding.
 * Deterministic: the same inputs give bit-identical outputs.
 */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int D, const fa_layout* layout, const fa_options* options,
                     const float* descale_q, const float* descale_k, const float* descale_v,
                     float scale, int causal, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Workspace bytes fa_bwd needs, laid out as (each part 256-byte aligned):
 *   lse2      fp32 [B*H][Npad]   LSE * log2(e); +inf for padding rows
 *   di        fp32 [B*H][Npad]   Di = rowsum(dO * O); 0 for padding rows
 *   dq_accum  fp32 [B*H][N][D]   only when deterministic == 0
 * where Npad is N rounded up to a multiple of 128.  Returns 0 for invalid
 * sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int D, int deterministic);

/*
 * Backward pass ([WALK] sec. 3.3; [DEEP] backward recomputation): given the
 * forward's o and lse and the upstream gradient dO, writes dq, dk, dv.
 *
 *   P_ij  = exp(scale * Q_i . K_j - lse_i)        recomputed, never stored
 *   Di    = sum_d dO_id O_id                      (= sum_j P_ij dP_ij)
 *   dV_j  = sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i . V_j - Di)
 *   dQ_i  = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
 *
 * deterministic == 0: dQ is accumulated with fp32 atomics into the workspace
 *   and converted at the end (fast; summation order varies run to run).
 * deterministic != 0: a second pass computes dQ one query tile at a time with
 *   no atomics; results are bit-identical across runs ([API] deterministic).
 * `workspace` must hold fa_bwd_workspace_size(...) bytes, 256-byte aligned;
 * its contents on entry do not matter.
 *
 * Its kernels are launched with programmatic stream serialization: each may
 * start while the kernel before it in the stream finishes, and waits for
 * that kernel's completion before reading anything (as fa_fwd's does).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                 float scale, int causal, fa_dtype dtype, int deterministic, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * fa_bwd on operands in any layout described by `layout`; bit-identical to
 * fa_bwd on the same values stored contiguously.  The workspace is the same
 * size and layout as for fa_bwd.
 */
fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int D, const fa_layout* layout, float scale, int causal,
                         fa_dtype dtype, int deterministic, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * The general backward, matching fa_fwd_ex: the same `layout` and
 * `options` (and causal) as the forward that produced o and lse.  The
 * gradients are those of the windowed, biased attention; the slopes get no
 * gradient.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                    const fa_layout* layout, const fa_options* options, float scale, int causal,
                    fa_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * The stages fa_bwd enqueues, for callers that schedule or time them
 * separately.  fa_bwd(...) is exactly fa_bwd_preprocess, then fa_bwd_dkdv,
 * then fa_bwd_dq_convert (deterministic == 0) or fa_bwd_dq (otherwise), all
 * on one stream with one workspace.
 */

/* Fills lse2 and di in the workspace (and zeroes dq_accum when
 * deterministic == 0) from o, dO and the forward's lse. */
fa_status fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int H, int N,
                            int D, fa_dtype dtype, int deterministic, void* workspace,
                            size_t workspace_bytes, void* stream);

/* One pass over key tiles, each looping over query tiles: writes dk and dv.
 * When deterministic == 0 it also adds sum_j dS_ij K_j (without the scale
 * factor) into the workspace's dq_accum with fp32 atomics. */
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                      void* dv, int B, int H, int N, int D, float scale, int causal,
                      fa_dtype dtype, int deterministic, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Deterministic dQ: one query tile per CTA looping over key tiles, no
 * atomics.  Needs lse2 and di in the workspace. */
fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B,
                    int H, int N, int D, float scale, int causal, fa_dtype dtype, void* workspace,
                    size_t workspace_bytes, void* stream);

/* dq = scale * dq_accum (the workspace of a deterministic == 0 call),
 * rounded to dtype. */
fa_status fa_bwd_dq_convert(void* dq, int B, int H, int N, int D, float scale, fa_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass without any device allocation by the caller or the library.
 * The pages describe nothing like it; it exists for callers that cannot hand
 * over a workspace -- for example a plug-in run inside another framework's
 * execution step that receives only its tensors and no allocator, or a
 * latency-bound caller that cannot afford cudaMalloc (which may synchronise
 * the whole device) in the middle of a step.
 *
 * Computes exactly what fa_bwd(..., deterministic = 1, ...) computes, with the
 * same kernels; its scratch (the padded log2-LSE and Di rows, 8 bytes per
 * query row rounded up to 128-row tiles, i.e. 8 * B*H*ceil(N/128)*128 bytes
 * plus alignment) lives in one fixed array of FA_NOALLOC_SCRATCH_BYTES that
 * the library places in device memory on every GPU where it is loaded, held
 * until the process exits.
 *   - Shapes whose scratch would not fit return FA_ERR_UNSUPPORTED before
 *     anything is enqueued (B*H*ceil(N/128)*128 may be at most 2^20 rows).
 *   - The first call on a device resolves the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     A cudaDeviceReset replaces the device's context and with it that
 *     address: the first call after it resolves the address again (so it,
 *     too, should come before any capture).
 *   - Every call on a device shares the one array, and each call overwrites
 *     it completely.  Calls whose work can overlap on the GPU (different
 *     streams, no ordering between them) race on it: order them on one stream.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define FA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int D, float scale, int causal, fa_dtype dtype,
                         void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * bounded waits write.  *code receives FA_OK or FA_ERR_TIMEOUT.  Returns
 * FA_ERR_CUDA if the synchronisation or the read fails.
 */
fa_status fa_device_error(void* stream, int* code);

/*
 * Failure-detection self test: enqueues one small kernel that waits on a
 * barrier nothing ever signals, with a limit of `limit_us` microseconds
 * (1 <= limit_us <= 2000000), then reads the error word as fa_device_error
 * does.  Returns FA_ERR_TIMEOUT when the wait ran out as intended; the
 * context stays usable.
 */
fa_status fa_selftest_wait_timeout(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
