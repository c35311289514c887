/*
 * dflash2.h — C ABI of the GB300 (sm_103a) library for the block-local tail of the
 * DFlash2 speculative-decoding drafter.
 *
 * The library computes two things, on one GPU, for B independent draft blocks of G rows
 * (an anchor row followed by G-1 mask rows):
 *
 *  1. the two-tap dynamic grouped depthwise convolution wrapped around each drafter
 *     sublayer. kernel_projection of the RMS-normed sublayer input emits
 *     D[t, side, tap, group] for both sides at once; side 0 is applied before the
 *     sublayer (prepare) and side 1 after it (finish):
 *         Conv_side(y)[t, c] = sum_tau (base[side, tau, c] + D[t, side, tau, c / gs]) * y[t - tau, c]
 *     with t block-local and y[-1] = 0, so nothing is read across a block boundary.
 *     (dflash2.ts of "@mlx-bun/inference 1.0.0": header comment, #coefficients, #conv;
 *      MAX API "max.pipelines.architectures.dflash2_qwen3_5": DFlash2GroupedConv,
 *      prepare, finish, DFlash2TransformerBlock.)
 *
 *  2. the candidate-path selector: the head GEMM over rows 1..G-1 with a fused top-K per
 *     row, z = hidden_projection(h), the low-rank bilinear edge scores
 *         S[b, l, p, c] = unary[b, l, c] + sum_r pred_book[pid(b,l,p), r] * z[b, l, r] * succ_book[cand[b, l, c], r]
 *     (pid(b, 0, p) = anchor[b], pid(b, l, p) = cand[b, l-1, p]) and the greedy
 *     left-to-right walk over S.
 *     (MAX API: DFlash2CandidateSelector, score_edges, select_path,
 *      DFlash2Qwen3_5.compute_candidates; dflash2.ts: #select.)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer is a DEVICE pointer owned by the caller, unless stated otherwise. The
 *    library never allocates device memory per call; scratch comes from caller-owned
 *    workspaces whose size a *_workspace_bytes() query returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *    default stream). A return value reports host-side validation and launch only.
 *  - Device-side faults the kernels can detect (an id outside [0, V), a bounded wait that
 *    ran out) are recorded in a device error word instead of trapping;
 *    dflash2_poll_error() reads and clears it.
 *  - dtype: DFLASH2_BF16 (production: bf16 storage, fp32 arithmetic and accumulation,
 *    tcgen05 kind::f16) or DFLASH2_F32 (fp32 storage; elementwise work in fp32, the GEMMs
 *    on tcgen05 kind::tf32).
 *  - Tensors are dense, row-major, with the innermost dimension last, and 16-byte aligned.
 *  - The first call of an entry point on a device sets kernel attributes; make it before
 *    capturing the calls into a CUDA graph.
 *  - Errors: DFLASH2_ERR_INVALID_ARG for a NULL required pointer, a misaligned pointer or a
 *    shape outside the documented limits; DFLASH2_ERR_UNSUPPORTED for taps != 2 (two-tap
 *    only, as dflash2.ts readConfig demands); DFLASH2_ERR_WORKSPACE for a workspace smaller
 *    than the query returns; DFLASH2_ERR_CUDA if a launch failed. Nothing is launched when
 *    an error is returned. dflash2_last_error_message() describes the last failure of the
 *    calling thread.
 */
#ifndef DFLASH2_H_
#define DFLASH2_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH2_API __attribute__((visibility("default")))
#else
#define DFLASH2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH2_OK = 0,
  DFLASH2_ERR_INVALID_ARG = -1,
  DFLASH2_ERR_UNSUPPORTED = -2,
  DFLASH2_ERR_CUDA = -3,
  DFLASH2_ERR_WORKSPACE = -4,
  DFLASH2_ERR_TIMEOUT = -5,  /* device: a bounded wait gave up */
  DFLASH2_ERR_BAD_INDEX = -6 /* device: a token id outside [0, V) was read */
} dflash2_status;

typedef enum { DFLASH2_BF16 = 0, DFLASH2_F32 = 1 } dflash2_dtype;

/* Library version, e.g. 100 for 0.1.0. */
DFLASH2_API int dflash2_version(void);

/* Human-readable name of a status code (static storage). */
DFLASH2_API const char* dflash2_status_string(int status);

/* Description of the last error returned to the calling host thread (thread-local storage). */
DFLASH2_API const char* dflash2_last_error_message(void);

/* Synchronises `stream`, then returns and clears the device error word of the current
 * device (DFLASH2_OK if no kernel recorded an error), or DFLASH2_ERR_CUDA if the
 * synchronisation itself failed. */
DFLASH2_API int dflash2_poll_error(void* stream);

/* ------------------------------------------------------------------------------------
 * Conv, pre-sublayer side (MAX DFlash2GroupedConv.prepare; dflash2.ts #block:
 * n = rms(x); coef = #coefficients(n); a = #conv(n, coef, 0)).
 *
 *   x        [B, G, H] dtype  the sublayer input (residual stream), one dense G-row block
 *                             per draft block (MAX forward_block: the block axis is a
 *                             reshape of the token axis).
 *   norm_w   [H] dtype or NULL. Non-NULL: n = x / sqrt(mean(x^2) + eps) * norm_w is
 *                             computed first. NULL: x is already normalised (n = x).
 *   eps      RMSNorm epsilon.
 *   w_kp     [2*taps*groups, H] dtype, kernel_projection weight stored (out, in); output
 *                             column o = (side*taps + tap)*groups + group.
 *   base     [2, taps, H] fp32 base kernel (side, tap, channel).
 *   B >= 1, 2 <= G <= 64, H % 64 == 0, group_size % 8 == 0, H % group_size == 0,
 *   groups = H / group_size, taps == 2.
 *   out      [B, G, H] dtype   a = side-0 conv of n (fp32 arithmetic, rounded to dtype).
 *   coef1    [B, G, taps, groups] dtype  side 1's deltas D[t, 1, tap, g], WITHOUT the base
 *                             kernel (finish adds base[1] back).
 *   d_full   [B, G, 2, taps, groups] fp32 or NULL: the full projection D (diagnostics).
 *   workspace / workspace_bytes: at least dflash2_conv_prepare_workspace_bytes(...) bytes
 *                             of device memory, 256-byte aligned; contents are scratch.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API size_t dflash2_conv_prepare_workspace_bytes(int B, int G, int H, int group_size, int dtype);
/* Number of kernels one dflash2_conv_prepare call launches for this shape (with_norm: norm_w
 * given; kernel_projection and the side-0 pass are one kernel up to 128 bf16 rows, two above) and
 * one dflash2_conv_finish call (with_next_norm: next_norm_w given): with the next norm, finish is a
 * single fused kernel up to 256 rows or where its tiles fit, else a side-1 pass and a norm pass.
 * -1 for a shape the calls reject. Host-only; launches nothing. */
DFLASH2_API int dflash2_conv_prepare_launches(int B, int G, int H, int group_size, int dtype, int with_norm);
DFLASH2_API int dflash2_conv_finish_launches(int B, int G, int H, int group_size, int dtype, int with_next_norm);
DFLASH2_API int dflash2_conv_prepare(const void* x, const void* norm_w, float eps, const void* w_kp, const float* base,
                         int B, int G, int H, int group_size, int taps, int dtype, void* out, void* coef1,
                         float* d_full, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Conv, post-sublayer side plus the residual add (MAX DFlash2GroupedConv.finish and
 * DFlash2TransformerBlock: r += conv.finish(h); dflash2.ts #block: x = x + #conv(out, coef, 1)
 * with the add in fp32).
 *
 *   y         [B, G, H] dtype   the sublayer output.
 *   coef1     [B, G, taps, groups] dtype  from dflash2_conv_prepare.
 *   base      [2, taps, H] fp32 (side 1 is used).
 *   residual  [B, G, H] dtype or NULL. out = residual + Conv_1(y) (fp32 add, one rounding),
 *                             or out = Conv_1(y) when NULL. out may alias residual.
 *   out       [B, G, H] dtype.
 *   next_norm_w [H] dtype or NULL; next_n dtype or NULL (both or neither):
 *             next_n[b, t - next_row0, :] = rms(out[b, t, :]) * next_norm_w for
 *             t in [next_row0, G), i.e. a [B, G - next_row0, H] tensor. next_row0 = 0 feeds
 *             the next conv site's prepare (norm_w = NULL); next_row0 = 1 with the final
 *             norm gives the head's input h (rows 1..G-1, dflash2.ts #block).
 *             Requires H <= 8192 (one thread per 8 channels of a row reduces the row).
 * ---------------------------------------------------------------------------------- */
DFLASH2_API int dflash2_conv_finish(const void* y, const void* coef1, const float* base, int B, int G, int H,
                        int group_size, int taps, int dtype, const void* residual, void* out,
                        const void* next_norm_w, float eps, void* next_n, int next_row0, void* stream);

/* ------------------------------------------------------------------------------------
 * Head GEMM + fused top-K + hidden_projection (MAX DFlash2Qwen3_5.compute_candidates and
 * DFlash2CandidateSelector's proj(h); dflash2.ts #block: logits = head(h), z = selProj(h),
 * #select's per-row top-K). Full-vocabulary logits are never written to memory.
 *
 *   h         [M, H] dtype   the normed drafter rows (M = B * (G - 1), rows 1..G-1 of each block).
 *   w_head    [V, H] dtype   the borrowed head, stored (out, in).
 *   bias      [V] fp32 or NULL, added to every logit.
 *   w_proj    [R, H] dtype or NULL (then z must be NULL): hidden_projection weight.
 *   cand      [M, K] int32   the K best vocabulary ids per row, by value descending; equal
 *                            values keep the lower id first (the same rule decides the K-th place).
 *   unary     [M, K] fp32    their logits.
 *   z         [M, R] fp32 or NULL: h @ w_proj^T.
 *   logits    [M, V] fp32 or NULL: every logit (diagnostics only; costs M*V*4 bytes of writes).
 *   1 <= K <= 16, K <= V, H % 64 == 0, R % 16 == 0 and R <= 256 when w_proj is given.
 *   workspace: at least dflash2_head_topk_workspace_bytes(M, H, V, K, R) bytes.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API size_t dflash2_head_topk_workspace_bytes(int M, int H, int V, int K, int R);
DFLASH2_API int dflash2_head_topk(const void* h, int M, int H, const void* w_head, int V, const float* bias, const void* w_proj,
                      int R, int K, int dtype, int32_t* cand, float* unary, float* z, float* logits,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Head + top-K over a draft vocabulary (dflash2.ts #block: a target that declares its draft
 * vocabulary projects the head onto those rows only; #select: `ids` maps the columns of the
 * logits over the draft vocabulary to token ids before the codebook gathers).
 *
 *   w_listed   [V_listed, H] dtype   the head rows of the listed vocabulary, in listed order.
 *   vocab_ids  [V_listed] int32      the token id of each listed row (required).
 *   bias_listed [V_listed] fp32 or NULL.
 *   cand       [M, K] int32          TOKEN ids (vocab_ids of the chosen rows), ordered by value
 *                                    descending; equal values keep the earlier listed row first.
 *   Everything else (h, w_proj/z, unary, logits [M, V_listed], workspace sized by
 *   dflash2_head_topk_workspace_bytes(M, H, V_listed, K, R)) is as for dflash2_head_topk.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API int dflash2_head_topk_vocab(const void* h, int M, int H, const void* w_listed, int V_listed,
                                        const int32_t* vocab_ids, const float* bias_listed, const void* w_proj, int R,
                                        int K, int dtype, int32_t* cand, float* unary, float* z, float* logits,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Allocation-free variant of dflash2_head_topk. The pages describe no counterpart: this entry
 * point exists for callers that cannot allocate device memory when they run the head — a
 * latency-bound serving loop where a cudaMalloc would stall every other stream of the device, a
 * host runtime whose allocator is not CUDA-aware, and plug-in hosts that only hand over the input
 * and output buffers. Arguments and results are those of dflash2_head_topk without the
 * workspace: the top-K scratch lives in a fixed 8 MiB device array inside the library, held on
 * every device that loads the library until the process exits.
 *  - Calls whose scratch would exceed 8 MiB are rejected with DFLASH2_ERR_INVALID_ARG (960 rows
 *    need about 4.7 MB on a 152-SM GB300).
 *  - All calls on a device share the array and it keeps the last call's contents; nothing in it
 *    needs to start at zero. Calls that overlap on the GPU race on it: keep them on one stream.
 *  - The first call on a device looks up the array's address; make it before any stream capture.
 *    The address is cached per device index: it belongs to the device's primary context (the one
 *    the CUDA runtime uses) and stays valid until cudaDeviceReset; callers that bind another
 *    context with the driver API, or reset the device, must not call this entry point afterwards.
 *  - Never calls cudaMalloc, cudaFree or any allocating library routine.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API int dflash2_head_topk_noalloc(const void* h, int M, int H, const void* w_head, int V, const float* bias,
                                          const void* w_proj, int R, int K, int dtype, int32_t* cand, float* unary,
                                          float* z, float* logits, void* stream);

/* ------------------------------------------------------------------------------------
 * Edge scores, optionally fused with the greedy walk (MAX DFlash2CandidateSelector.score_edges
 * and select_path; dflash2.ts #select).
 *
 *   cand      [B, steps, K] int32 candidate ids (from dflash2_head_topk, M = B * steps).
 *   unary     [B, steps, K] fp32.
 *   z         [B, steps, R] fp32.
 *   anchors   [B] int32, the last verified token of each block.
 *   pred_book, succ_book [V, R] dtype  predecessor / successor codebooks.
 *   1 <= steps <= 63, 1 <= K <= 32, 8 <= R <= 128 with R % 8 == 0.
 *   S         [B, steps, K, K] fp32 indexed [b, l, p, c], or NULL.
 *   path      [B, steps] int32 or NULL: the greedy walk (slot 0 reads row p = 0; slot l reads
 *             the row of the position chosen at l-1; ties go to the lowest position).
 *   At least one of S and path must be non-NULL. An id outside [0, V) sets
 *   DFLASH2_ERR_BAD_INDEX and reads as a zero codebook row.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API int dflash2_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                        const void* pred_book, const void* succ_book, int B, int steps, int K, int R, int V,
                        int dtype, float* S, int32_t* path, void* stream);

/* The greedy walk alone, over a given S (MAX DFlash2CandidateSelector.select_path without a
 * sampler). S [B, steps, K, K] fp32, cand [B, steps, K] int32 -> path [B, steps] int32.
 * 1 <= steps, 1 <= K <= 32. */
DFLASH2_API int dflash2_select_path(const float* S, const int32_t* cand, int B, int steps, int K, int32_t* path, void* stream);

/* Mixed-depth batches (dflash2.ts blockColumns / #block: a block asked to draft `depth` tokens runs
 * over its anchor and min(G - 1, max(1, depth)) mask rows; MAX DFlash2Qwen3_5.supports_zero_draft_rows
 * is False, so no block drafts nothing). In a dense [B, G, ...] batch block b drafts
 * d_b = min(steps, max(1, depths[b])) tokens; its rows past d_b + 1 are padding. The conv and the
 * head need no change for that (the conv only looks one row back, and the head works row by row),
 * so only the walk honours the depths: block b walks slots [0, d_b) and path[b, l] = -1 for later
 * slots.
 *   depths [B] int32 (device). Every value is accepted and clamped to [1, steps] as blockColumns
 *   clamps it. Other arguments as for dflash2_score_edges / dflash2_select_path; path is required.
 *   S (if requested) is computed for every slot. */
DFLASH2_API int dflash2_score_edges_depths(const int32_t* cand, const float* unary, const float* z,
                                           const int32_t* anchors, const void* pred_book, const void* succ_book,
                                           const int32_t* depths, int B, int steps, int K, int R, int V, int dtype,
                                           float* S, int32_t* path, void* stream);
DFLASH2_API int dflash2_select_path_depths(const float* S, const int32_t* cand, const int32_t* depths, int B, int steps,
                                           int K, int32_t* path, void* stream);

/* ------------------------------------------------------------------------------------
 * Ragged batches: only the rows a block drafts go through the head and the selector.
 * (dflash2.ts blockColumns / #block: a block asked to draft `depth` tokens runs over its anchor
 * and d = min(G - 1, max(1, depth)) mask rows, and only those rows reach the head and #select.)
 * In a dense [B, G, ...] batch the conv runs over all G rows of every block (the rows past d + 1
 * are padding that never reaches an earlier row: the conv looks one row back); the head's rows
 * are then packed per block:
 *   row_offsets [B + 1] int32 (device): row_offsets[0] = 0 and row_offsets[b + 1] - row_offsets[b]
 *                  = d_b, the rows block b drafts, in [1, G - 1]; m_rows = row_offsets[B] (host).
 * dflash2_conv_finish_ragged is dflash2_conv_finish with the next norm written only for block b's
 * first d_b rows from next_row0 on, at rows row_offsets[b] .. of next_n [m_rows, H] (next_norm_w
 * and next_n required). dflash2_head_topk then runs over M = m_rows rows as usual, and
 * dflash2_score_edges_ragged reads block b's slots at rows row_offsets[b] .. of cand, unary, z
 * ([m_rows, K], [m_rows, K], [m_rows, R]) and S ([m_rows, K, K] or NULL), and writes path
 * [B, steps] (required) with -1 past d_b. It supports K = 16 with R in {16, 32, 64} (bf16) or
 * {16, 32} (f32). A block whose span is not inside [0, m_rows) or holds outside [1, G - 1]
 * (finish) / [1, steps] (edges) rows records DFLASH2_ERR_INVALID_ARG in the device error word and
 * is skipped (nothing written for it; its path stays -1). */
DFLASH2_API int dflash2_conv_finish_ragged(const void* y, const void* coef1, const float* base, int B, int G, int H,
                                           int group_size, int taps, int dtype, const void* residual, void* out,
                                           const void* next_norm_w, float eps, void* next_n, int next_row0,
                                           const int32_t* row_offsets, int m_rows, void* stream);
DFLASH2_API int dflash2_score_edges_ragged(const int32_t* cand, const float* unary, const float* z,
                                           const int32_t* anchors, const void* pred_book, const void* succ_book,
                                           const int32_t* row_offsets, int B, int steps, int K, int R, int V,
                                           int m_rows, int dtype, float* S, int32_t* path, void* stream);

/* ------------------------------------------------------------------------------------
 * The sublayer projections around a conv site, with the conv fused into them.
 * (dflash2.ts #block: a = #conv(n, coef, 0) feeds q/k/v (attention) or gate/up (MLP); o or down's
 * output goes through #conv(., coef, 1) and is added to the residual in fp32. MAX
 * DFlash2TransformerBlock: h = conv.prepare(norm(r)); h = sublayer(h); r += conv.finish(h).)
 * bf16 only (DFLASH2_BF16; anything else returns DFLASH2_ERR_UNSUPPORTED). fp32 accumulation on the
 * tensor cores; outputs rounded once to bf16.
 *
 * dflash2_conv_coefficients: prepare without the side-0 output. Optional RMSNorm (norm_w given:
 *   n_out [B*G, H] receives n; else n = x and n_out may be NULL), kernel_projection, then
 *   d0 [2, groups, B*G] fp32 = side 0's deltas, d0[tap, g, m] = D[m, 0, tap, g] (tap-and-group
 *   major, the layout the fused input projection loads), and coef1 [B*G, 2, groups] dtype = side
 *   1's (as dflash2_conv_prepare's coef1). Workspace as dflash2_conv_prepare_workspace_bytes.
 *
 * dflash2_proj: out [M, N] = a [M, K] . W^T.
 * dflash2_proj_conv_in: out = Conv_0(n) . W^T, Conv_0(n)[m, k] = (base[0,0,k] + d0[0,k/gs,m]) n[m, k]
 *   + (base[0,1,k] + d0[1,k/gs,m]) n[m-1, k], n[m-1] = 0 at each block's first row (m % G == 0);
 *   the side-0 output is computed in the GEMM's operand producer and never written. K = H;
 *   base [2, 2, K] fp32; d0 16-byte aligned; G divides 128, M % G == 0, group_size 16.
 * dflash2_proj_conv_out: out = residual + Conv_1(a . W^T) (residual may be NULL), Conv_1 with the
 *   side-1 deltas coef1 [M, 2, N/gs] (bf16) and base[1] over the N = H output channels, computed in
 *   the GEMM's epilogue (fp32 add, one rounding). G divides 32, M % G == 0, group_size in {8, 16, 32},
 *   N % 32 == 0. out may not alias residual.
 *
 * Workspace: at least dflash2_proj_workspace_bytes(M, N, K) bytes, 256-byte aligned (0 bytes, and
 * workspace may be NULL, when the shape needs none: up to 128 rows the K range is split over the
 * CTAs of a thread-block cluster and reduced in shared memory; above, a shape whose tiles do not
 * fill the SMs splits K over them and the partial sums go through the workspace to a reduce pass
 * that applies the epilogue; with at least half as many 128 x 256 tiles as SMs every SM takes an
 * equal stream-K share of the tiles' k-blocks and the workspace holds one 128 x 256 fp32 partial
 * tile per CTA, handed to the tile's owner through a flag array inside the library). The flags are
 * per device and process: calls of these three entry points that can run at the same time on one
 * device (on different streams) must not overlap; keep them on one stream. Above 384 rows a 4-bit
 * weight is dequantised once into the workspace (N x K bf16, after the partial tiles) and the
 * projection runs on that copy, and dflash2_proj_conv_in applies side 0 to the rows once (M x K
 * bf16, after that) before its projection; the query, which knows neither the weight format nor the
 * fusion, counts both from 385 rows on. The contents of the workspace need no initialisation.
 *
 * Weights: wbits = 16: w is bf16 [N, K] (out, in). wbits = 4: affine 4-bit weights in groups of 64
 * along K (dflash2.ts quantizedWeight: quantize(w, 64, bits), mode "affine"): w is [N, K/8] uint32,
 * value k of row n in bits 4 (k % 8) .. 4 (k % 8) + 3 of word k / 8 (an unsigned q in [0, 15]);
 * w_scales and w_biases are bf16 [K/64, N] (group-major, so one group's values for a tile of rows
 * are contiguous); W[n, k] = w_scales[k/64, n] * q + w_biases[k/64, n], rounded once to bf16
 * before the MMA. K % 64 == 0, N % 8 == 0, M >= 1; a, w, w_scales, w_biases, out, residual and base
 * 16-byte aligned.
 * ---------------------------------------------------------------------------------- */
DFLASH2_API int dflash2_conv_coefficients(const void* x, const void* norm_w, float eps, const void* w_kp, int B, int G,
                                          int H, int group_size, int taps, int dtype, void* n_out, float* d0,
                                          void* coef1, void* workspace, size_t workspace_bytes, void* stream);
DFLASH2_API size_t dflash2_proj_workspace_bytes(int M, int N, int K);
DFLASH2_API int dflash2_proj(const void* a, int M, int K, const void* w, const void* w_scales, const void* w_biases,
                             int wbits, int N, int dtype, void* out, void* workspace, size_t workspace_bytes,
                             void* stream);
DFLASH2_API int dflash2_proj_conv_in(const void* n, const float* d0, const float* base, int G, int group_size, int M,
                                     int K, const void* w, const void* w_scales, const void* w_biases, int wbits, int N,
                                     int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream);
DFLASH2_API int dflash2_proj_conv_out(const void* a, int M, int K, const void* w, const void* w_scales,
                                      const void* w_biases, int wbits, int N, const void* coef1, const float* base,
                                      int G, int group_size, const void* residual, int dtype, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Self-test of the bounded-wait machinery: launches one block that waits on an mbarrier that
 * nothing completes, with a limit of `limit_us` microseconds (1..1000000). The wait gives up,
 * records DFLASH2_ERR_TIMEOUT in the device error word and the kernel returns; read it with
 * dflash2_poll_error(). Has no counterpart on the pages. */
DFLASH2_API int dflash2_selftest_bounded_wait(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H_ */
