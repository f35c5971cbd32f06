/*
 * spec.h -- C ABI of the batch-invariant speculative-verification library
 * (libspec.so, CUDA sm_103a).
 *
 * Contract.  Greedy speculative decoding returns the same tokens as ordinary
 * one-token-at-a-time decoding only if the target model computes, for every
 * query row, the same logits whether the row is evaluated alone (width 1), in
 * a verify block of width 2-8, or in a ragged batch of several sequences
 * (ramgpt.org, "When Lossless Speculation Stops Being Lossless on Blackwell",
 * sections "The Hidden Contract Behind Lossless Speculation" and "A Better
 * Backend Test Matrix").  Every floating-point entry point below computes each
 * output element with a sequence of operations fixed by the reduction length
 * (K for the matmul, the row's own KV length for attention, H for norms) and
 * by nothing else: not by the number of columns, rows or sequences in the
 * call, nor by where in the call the row sits.  Results are therefore
 * bit-identical across widths and batch compositions.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *    library allocates no device memory and keeps no per-call state; scratch
 *    is caller-supplied workspace sized by the matching *_workspace() call
 *    (spec_qmatmul_static_scratch, below, is the one exception: its scratch
 *    is a fixed array inside the library).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  All calls except spec_qmatmul_static_scratch may be
 *    captured in a CUDA graph.
 *  - The returned status reports errors the host can see: bad shapes, NULL or
 *    misaligned pointers, short workspace, launch failure.  On any status
 *    other than SPEC_OK nothing was launched, and spec_last_error() gives a
 *    one-line reason (thread-local).
 *  - Errors only the device can see (a token id out of range, a NaN logit, a
 *    block-table entry that is negative, a sequence longer than the declared
 *    bound) are OR-ed into the caller's int32 word `dev_err` (may be NULL) as
 *    SPEC_DEVERR_* bits.  Kernels never trap and never wait without a bound.
 *  - bf16 / fp16 values are passed as their 16-bit patterns (uint16_t).
 *  - KV caches are paged: [num_pages][Hkv][16][D], 16 tokens per page; token j
 *    of sequence s lives in page block_table[s * max_blocks + j / 16], slot
 *    j % 16.
 *  - Ragged batches: sequence s owns rows cu_rows[s] .. cu_rows[s+1]-1
 *    (cu_rows has S+1 entries, cu_rows[0] = 0, cu_rows[S] = R); its rows sit
 *    at absolute positions ctx_start[s], ctx_start[s]+1, ...
 */
#ifndef SPEC_H
#define SPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *spec_stream_t; /* a cudaStream_t */

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* bad shape, NULL or misaligned pointer */
    SPEC_ERR_UNSUPPORTED = 2, /* valid request the library does not support */
    SPEC_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than *_workspace() */
    SPEC_ERR_CUDA = 4         /* a CUDA runtime call failed */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_F16 = 1, SPEC_BF16 = 2 } spec_dtype;

/* bits OR-ed into *dev_err by kernels */
#define SPEC_DEVERR_TOKEN_RANGE 0x1 /* a token id outside [0, V) */
#define SPEC_DEVERR_NAN 0x2         /* a NaN logit (it never wins an argmax) */
#define SPEC_DEVERR_BLOCK_TABLE 0x4 /* a needed block-table entry is negative or >= num_pages */
#define SPEC_DEVERR_LENGTH 0x8      /* a sequence exceeds max_kv_len / max_blocks * 16 */
#define SPEC_DEVERR_TIMEOUT 0x10    /* a bounded wait on an mbarrier ran out */
#define SPEC_DEVERR_LAYOUT 0x20     /* cu_rows not non-decreasing or cu_rows[S] != R */

const char *spec_status_string(spec_status st);
const char *spec_last_error(void);

/* ------------------------------------------------------------------------
 * K1  block-4-bit dequantising matmul
 *
 *   y[j][n] (+)= sum_k x[j][k] * d[n][k/32] * (nib(n, k) - 8)
 *
 * ramgpt.org, "When Lossless Speculation Stops Being Lossless on Blackwell",
 * section "Quantized Matrix Multiplication Shows the Same Class of Failure":
 * a batched product must equal the concatenation of single-column products.
 * tokenstrom.com, "'Lossless,' but not quite", section "Why the math checks
 * out and the text still flips": the mat-vec's warp split (and so its partial-
 * sum order) changed with the number of tokens.  Here the K-split, each lane's
 * partial-sum order and the combine order are functions of K alone.
 *
 *   wq   uint8 [N][K/2]: two 4-bit codes per byte, even k in the low nibble,
 *        code = q + 8 for q in [-8, 7].  16-byte aligned.
 *   ws   fp16 bits [N][K/32]: one scale per 32 consecutive k.  16-byte aligned.
 *   x    bf16 bits [n_cols][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned.
 *   y    [n_cols][ldy] of y_dt (SPEC_F32 or SPEC_BF16), ldy >= N.
 *        accumulate != 0 adds into y (SPEC_F32 only): y = fp32(y + result).
 *   workspace  at least spec_qmatmul_workspace(N, K, n_cols) bytes, 16-byte
 *        aligned, zero-filled before its first use (cudaMemset once).  A call
 *        keeps one arrival counter per 128 rows and column group (at most
 *        10 groups, only while they fit in 64 KB) at the workspace's start;
 *        every call that returns SPEC_OK and reports no
 *        SPEC_DEVERR_TIMEOUT leaves the first 64 KB zero again (counters reset,
 *        consumed partial sums cleared), so one workspace serves any sequence
 *        of calls of any shapes on one stream; calls that overlap on the GPU
 *        need separate workspaces.
 *   K % 256 == 0, 1 <= N <= 2097152 (counters fit in 64 KB), n_cols >= 0
 *   (0 launches nothing).
 *   The kernel is launched with programmatic dependent launch: it may start
 *   reading wq and ws while the preceding kernel on the stream is still
 *   running (weights are treated as constant inputs); x, y and the workspace
 *   are touched only after that kernel has finished.
 *
 * Arithmetic of one output element (fixed by K): K is cut into segments of
 * 512 (the last may be 256); within a segment each 32-k block's partial is
 * one chain of two m16n8k16 MMAs, scaled by its fp16 scale into an fp32
 * accumulator in ascending block order; segment partials are added in
 * ascending segment order.
 *
 * Passes: up to 8 columns run as one 8-column pass, up to 16 as one 16-column
 * pass; 17 to 80 columns as the cheapest (by a fitted time estimate) of one
 * 80-column pass and one launch of 16- or 8-column groups; more as 80-column
 * passes.  The plan changes only
 * which CTA computes a column, never its arithmetic.
 * ---------------------------------------------------------------------- */
size_t spec_qmatmul_workspace(int N, int K, int n_cols);
spec_status spec_qmatmul(const uint8_t *wq, const uint16_t *ws, int N, int K,
                         const uint16_t *x, int n_cols, int ldx,
                         void *y, spec_dtype y_dt, int ldy, int accumulate,
                         void *workspace, size_t ws_bytes,
                         int32_t *dev_err, spec_stream_t stream);

/* The 80-column pass of spec_qmatmul with its activations already packed
 * (the same arithmetic, bit for bit): `xpk` holds the packed form of up to 80
 * activation columns (column c = row c of the producer) for every 256-k stage
 * of K, spec_packed_activation_bytes(K) bytes, written by
 * spec_add_rmsnorm_packed or spec_swiglu_packed; the call skips the packing
 * kernel spec_qmatmul launches before such a pass.  17 <= n_cols <= 80 (one
 * pass; columns from n_cols on are neither read for y nor written), K a
 * multiple of 256, xpk 16-byte aligned; y, ldy, accumulate, workspace
 * (spec_qmatmul_workspace(N, K, n_cols)) and dev_err as for spec_qmatmul.
 * Source: ramgpt.org, "When Lossless Speculation Stops Being Lossless on
 * Blackwell", section "Quantized Matrix Multiplication Shows the Same Class of
 * Failure" (only the delivery of the activations changes). */
size_t spec_packed_activation_bytes(int K);

/* Gate/up matmul with the SwiGLU applied as each output is written:
 *   act[j][f] = bf16(silu(g) * u),  silu(g) = g / (1 + e^-g) in fp32,
 * g and u the invariant K1 products (spec_qmatmul's arithmetic) of column j with
 * feature f's gate and up weight rows.  wq / ws hold the 2F rows of the gate/up
 * matrix interleaved: rows 16i .. 16i+7 are the gate rows of features
 * 8i .. 8i+7, rows 16i+8 .. 16i+15 their up rows (a row's result does not
 * depend on where it sits, so act equals spec_swiglu of spec_qmatmul's [gate;
 * up] output bit for bit).  F a positive multiple of 8; act bf16
 * [n_cols][ld_act], ld_act >= F; x, ldx, K, workspace
 * (spec_qmatmul_workspace(2F, K, n_cols)) and dev_err as for spec_qmatmul.
 * xpk (optional, 16-byte aligned): the same activations packed as for
 * spec_qmatmul_packed (17 <= n_cols <= 80); the call then plans as for a
 * caller with packed activations and an 80-column pass reads them.
 * The fp32 gate/up product is never written.  Source: the decoder's SwiGLU
 * feed-forward of ramgpt.org, "When Lossless Speculation Stops Being Lossless
 * on Blackwell" (the target model whose per-row results must not depend on
 * the batch). */
spec_status spec_qmatmul_swiglu(const uint8_t *wq, const uint16_t *ws, int F, int K,
                                const uint16_t *x, const void *xpk, int n_cols, int ldx,
                                uint16_t *act, int ld_act,
                                void *workspace, size_t ws_bytes,
                                int32_t *dev_err, spec_stream_t stream);

/* The pass width spec_qmatmul would take for n_cols columns of an N x K
 * matrix: 8, 16 (column groups of that width in one launch) or 80 (the
 * 80-column pass).  packed_input != 0 asks as for a caller that holds the
 * packed activations of spec_qmatmul_packed (the 80-column pass then needs no
 * packing launch): 80 means that entry point is the faster call, anything else
 * that spec_qmatmul is.  0 for an empty or invalid shape.  Host only. */
int spec_qmatmul_plan(int N, int K, int n_cols, int packed_input);
spec_status spec_qmatmul_packed(const uint8_t *wq, const uint16_t *ws, int N, int K, const void *xpk,
                                int n_cols, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream);

/* The same product for a column count known only on the device: the first
 * c = min(n_cols, *dev_cols) columns of x when *dev_cols >= min_cols, else
 * nothing (y untouched).  dev_cols (device int32) is read after the preceding
 * kernel on the stream has finished, so a kernel just before may write it; the
 * call launches the same kernels whatever the count, which lets a captured CUDA
 * graph re-evaluate a data-dependent number of rows.  n_cols is the most the
 * call may compute (it sizes the workspace and the passes); every other
 * argument and the arithmetic are those of spec_qmatmul, so a column's bits do
 * not depend on the count. */
spec_status spec_qmatmul_devcols(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                 const uint16_t *x, int n_cols, int ldx,
                                 void *y, spec_dtype y_dt, int ldy, int accumulate,
                                 const int32_t *dev_cols, int min_cols,
                                 void *workspace, size_t ws_bytes,
                                 int32_t *dev_err, spec_stream_t stream);

/* The same product with two-level (super-block) scales.  The pages name
 * two-level formats -- tokenstrom.com, "'Lossless,' but not quite", section
 * "Why the math checks out and the text still flips" (Q4_K / Q6_K); ramgpt.org,
 * "When Lossless Speculation Stops Being Lossless on Blackwell", section
 * "Quantized Matrix Multiplication Shows the Same Class of Failure" (IQ3_S /
 * IQ4_XS) -- but define none, so this one is the library's own:
 *
 *   y[j][n] (+)= sum_k x[j][k] * D[n][k/256] * s[n][k/32] * (nib(n, k) - 8)
 *
 *   wq   as for spec_qmatmul.
 *   sbr  uint8 [N][ceil(K/512) * 16], 16-byte aligned: per row and per 256-k
 *        super-block one 8-byte record, read as a little-endian 64-bit word:
 *        bits 6j .. 6j+5 = s_j in 0 .. 63, the scale of the super-block's
 *        32-k block j; bits 48 .. 63 = D, an fp16 super-scale.  When K/256 is
 *        odd each row's last record is padding (ignored).
 * Block b's scale is D * s_(b mod 8) formed exactly in fp32; every other
 * argument, the workspace (spec_qmatmul_workspace), the arithmetic and the
 * batch invariance are those of spec_qmatmul. */
spec_status spec_qmatmul_sb(const uint8_t *wq, const uint8_t *sbr, int N, int K,
                            const uint16_t *x, int n_cols, int ldx,
                            void *y, spec_dtype y_dt, int ldy, int accumulate,
                            void *workspace, size_t ws_bytes,
                            int32_t *dev_err, spec_stream_t stream);

/* The same product with a K-segment length of seg_stages x 512 chosen per
 * call (seg_stages = 0: picked from the problem size and the GPU for speed),
 * so its reduction order depends on the call: NOT batch invariant.  It exists
 * to measure what width-1 speed the invariant kernel gives up (the pages'
 * prior-art kernels pick geometry by width; tokenstrom.com, "'Lossless,' but
 * not quite", section "Why the math checks out and the text still flips").
 * Same argument rules as spec_qmatmul; y is fp32, no accumulate. */
spec_status spec_qmatmul_noninvariant(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                      const uint16_t *x, int n_cols, int ldx,
                                      float *y, int ldy, int seg_stages,
                                      void *workspace, size_t ws_bytes, spec_stream_t stream);

/* spec_qmatmul without a workspace argument; the source pages describe no
 * such call, it is a convenience of this library.  Its scratch is a fixed
 * 8 MiB array in the library's own device memory (one per device), so the
 * call allocates nothing.  It is meant for callers that cannot hand over a
 * buffer: a plain C host loop that owns no device allocator, a caller whose
 * device memory is all reserved by another framework's caching allocator, or
 * one that must not call cudaMalloc / cudaFree because those calls may
 * synchronise the device and stall the streams it is feeding.
 *
 * Arguments, arithmetic and results are those of spec_qmatmul with the same
 * inputs (bit for bit).  Shapes whose scratch would exceed 8 MiB, i.e.
 * ceil(N/128) * (1 + ceil(K/512)) * 4096 * nt bytes plus 256-byte-rounded
 * ceil(N/128) ints, with nt = 1 for n_cols <= 8, 2 for <= 16 and 10 above,
 * are rejected with SPEC_ERR_WORKSPACE and a message (for example N = 17408,
 * K = 5120 fits at up to 8 columns).  The scratch's leading counters must be
 * zero when the kernel starts: the call clears them on `stream` itself before
 * each launch, so nothing has to be zeroed by the caller.
 * There is one scratch per device: two calls whose work can overlap on the
 * GPU (different streams without an ordering between them) race on it and
 * give wrong results.  Order such calls, for example by issuing them on one
 * stream.  The first call on a device, made with that device current, looks
 * up the scratch address (cudaGetSymbolAddress); make that first call before
 * any stream capture begins. */
spec_status spec_qmatmul_static_scratch(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                        const uint16_t *x, int n_cols, int ldx,
                                        void *y, spec_dtype y_dt, int ldy, int accumulate,
                                        int32_t *dev_err, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * K2 + K3  split-KV causal attention for verify blocks (paged KV cache)
 *
 * ramgpt.org, section "Flash Attention Changes Geometry With Batch Width":
 * the tile geometry chosen by query width changed the KV traversal and the
 * combine order.  Here the KV sequence is cut into chunks of a constant 256
 * keys; row r (position p) gets one partial (max, sum, weighted values) per
 * chunk c <= p / 256 over keys [256c, min(256c + 255, p)]: each 64-key
 * sub-tile of the chunk whose first key is <= p yields its own (max, sum,
 * values) and the sub-tiles are merged in ascending order; the chunk
 * partials are then combined in ascending c.  Nothing depends on the other
 * rows of the call.
 *
 *   q        [R][Hq][D] of qkv_dt (SPEC_F16 or SPEC_BF16), 16-byte aligned
 *   k_cache, v_cache  [num_pages][Hkv][16][D] of qkv_dt, 16-byte aligned
 *   block_table int32 [S][max_blocks]
 *   ctx_start int32 [S]: tokens already cached before the block; the block's
 *            own K/V must already be in the cache (positions ctx_start[s] ..
 *            ctx_start[s] + rows - 1).  Row i attends to keys 0 .. ctx_start+i.
 *   cu_rows  int32 [S+1]
 *   max_kv_len  host bound on ctx_start[s] + rows of s: it sizes the
 *            workspace and the item count; the kernel itself stops at the
 *            chunks the sequences reach, so a loose bound (a graph captured
 *            once for a whole generation) costs next to nothing.  A sequence
 *            longer than the bound or than max_blocks * 16 keys is reported
 *            (SPEC_DEVERR_LENGTH), one whose rows fall outside [0, R) as
 *            SPEC_DEVERR_LAYOUT; the rows of such a sequence, and of one with
 *            a negative ctx_start, are written as zeros.
 *   out      [R][Hq][D] of out_dt (SPEC_F32 or SPEC_BF16)
 *   scale    multiplies q.k before the softmax
 *   D in {64, 128}; Hq % Hkv == 0; Hq / Hkv <= 16.
 * ---------------------------------------------------------------------- */
size_t spec_flash_decode_workspace(int R, int Hq, int D, int max_kv_len);
spec_status spec_flash_decode(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, float scale,
                              const void *k_cache, const void *v_cache, int num_pages,
                              const int32_t *block_table, int max_blocks,
                              const int32_t *ctx_start, const int32_t *cu_rows, int S, int R,
                              int max_kv_len, void *out, spec_dtype out_dt,
                              void *workspace, size_t ws_bytes, int32_t *dev_err,
                              spec_stream_t stream);

/* spec_flash_decode with bf16 output that also writes each output row r
 * (Hq * D values), as column r of an 80-column K1 pass, in the packed form
 * spec_qmatmul_packed reads (the o projection's input): xpk of
 * spec_packed_activation_bytes(Hq * D) bytes, 16-byte aligned; R <= 80,
 * Hq * D a multiple of 256.  out is written as by spec_flash_decode. */
spec_status spec_flash_decode_packed(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, float scale,
                                     const void *k_cache, const void *v_cache, int num_pages,
                                     const int32_t *block_table, int max_blocks,
                                     const int32_t *ctx_start, const int32_t *cu_rows, int S, int R,
                                     int max_kv_len, void *out, void *workspace, size_t ws_bytes,
                                     void *xpk, int32_t *dev_err, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * K4  ragged greedy verification
 *
 * proofoftech.org, "'Lossless' speculative decoding isn't free", opening
 * section: the target checks the drafts in one pass, accepts the prefix it
 * agrees with and corrects the first token it does not.  ramgpt.org, section
 * "The Hidden Contract Behind Lossless Speculation": greedy choice = the
 * maximum-logit token.
 *
 *   logits  [R][V] of dt (SPEC_F32 or SPEC_BF16), 16-byte aligned, V % 8 == 0
 *   drafts  int32 [R - S]: sequence s's L_s = rows_s - 1 drafts start at
 *           drafts[cu_rows[s] - s]
 *   argmax_out int32 [R]: lowest index of each row's maximum
 *   accepted   int32 [S]: first i < L_s with draft_i != argmax[r0 + i], else L_s
 *   correction int32 [S]: argmax[r0 + accepted[s]]
 *   ctx_new    int32 [S]: ctx_start[s] + accepted[s] + 1
 *   Integer results are exact; NaN logits never win and set SPEC_DEVERR_NAN.
 * ---------------------------------------------------------------------- */
size_t spec_verify_greedy_workspace(int R, int V);
spec_status spec_verify_greedy(const void *logits, spec_dtype dt, int V,
                               const int32_t *cu_rows, int S, int R,
                               const int32_t *drafts, const int32_t *ctx_start,
                               int32_t *argmax_out, int32_t *accepted, int32_t *correction,
                               int32_t *ctx_new, void *workspace, size_t ws_bytes,
                               int32_t *dev_err, spec_stream_t stream);

/* K4 with temperature sampling.  The pages state the byte-identity contract
 * for greedy decoding; extending it to sampling by tying every random draw to
 * the sequence and the position (never to the batch) is this library's
 * reading of ramgpt.org, section "A Better Backend Test Matrix".
 * Row r of sequence s at position p = ctx_start[s] + (r - cu_rows[s]) draws
 *     token[r] = argmax_v fma(logit[r][v], inv_temperature, -log(-log(u)))
 * (ties: lowest v; a Gumbel-max draw, i.e. an exact sample of
 * softmax(logit / T)), where u = (w >> 9) * 2^-23 + 2^-24 and w is word v % 4 of
 * Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3")
 * with counter (v / 4, p, id_s, 0x53504543) and key (seed low, seed high 32
 * bits); id_s = seq_id[s], or s when seq_id is NULL.  Acceptance, correction
 * and ctx_new are then those of spec_verify_greedy with token[] in place of
 * argmax[]: a width-1 decode that samples with the same seed and sequence ids
 * produces the same tokens, so speculative sampling reproduces it byte for
 * byte.  inv_temperature = 1 / T > 0 and finite.  Other arguments, the
 * workspace (spec_verify_greedy_workspace) and errors as in
 * spec_verify_greedy. */
spec_status spec_verify_sample(const void *logits, spec_dtype dt, int V,
                               const int32_t *cu_rows, int S, int R,
                               const int32_t *drafts, const int32_t *ctx_start,
                               const int32_t *seq_id, float inv_temperature, uint64_t seed,
                               int32_t *token_out, int32_t *accepted, int32_t *correction,
                               int32_t *ctx_new, void *workspace, size_t ws_bytes,
                               int32_t *dev_err, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * K5  KV-cache realignment after ragged acceptance
 *
 * proofoftech.org, section "Batching breaks the implementation": after
 * sequences accept different numbers of drafts their positions and KV state
 * must be realigned exactly.  Rows 0 .. accepted[s] of sequence s are kept:
 * staged row cu_rows[s] + i is written to the cache slot of position
 * ctx_start[s] + i.  Rejected rows never reach the cache.
 *
 *   k_stage, v_stage  [R][Hkv][D] 16-bit elements, or both NULL when the block
 *            was already written into the cache in place (then only the index
 *            outputs are produced and the cache is not touched)
 *   cu_kept  int32 [S+1]: exclusive prefix sum of accepted[s] + 1
 *   kept_src int32 [R], dst_slot int64 [R]: for kept token j (j < cu_kept[S])
 *            its staging row and its cache slot page * 16 + slot
 *   D % 8 == 0.
 * ---------------------------------------------------------------------- */
spec_status spec_kv_compact(const void *k_stage, const void *v_stage, void *k_cache, void *v_cache,
                            int Hkv, int D, int num_pages, const int32_t *block_table, int max_blocks,
                            const int32_t *ctx_start, const int32_t *accepted,
                            const int32_t *cu_rows, int S, int R,
                            int32_t *cu_kept, int32_t *kept_src, int64_t *dst_slot,
                            int32_t *dev_err, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * Decoder glue for the end-to-end generation workload.  Each is a per-row
 * operation with a fixed reduction order over the row, hence width-invariant.
 * The pages run real decoders but name none of these steps; they are the
 * textbook definitions (RMSNorm, rotate-half RoPE, SwiGLU).
 * ---------------------------------------------------------------------- */

/* h[r][:] = float(emb[tokens[r]][:]); emb bf16 [V][H]; h fp32 [R][H]. */
spec_status spec_embed(const uint16_t *emb, int V, int H, const int32_t *tokens, int R,
                       float *h, int32_t *dev_err, spec_stream_t stream);

/* If delta != NULL first h += delta (fp32, in place).  Then
 * out[r][:] = bf16(h[r][:] / sqrt(mean(h[r]^2) + eps) * w[:]).
 * h, delta fp32 [R][H]; w fp32 [H]; out bf16 [R][H]; H % 4 == 0. */
spec_status spec_add_rmsnorm(float *h, const float *delta, const float *w, int R, int H, float eps,
                             uint16_t *out, spec_stream_t stream);

/* Fill tab[p][i] = (cos, sin)(p * theta^(-2i/D)) for p < max_pos, i < D/2,
 * fp32 [max_pos][D/2][2]; angles evaluated in double. */
spec_status spec_rope_table(float *tab, int max_pos, int D, float theta, spec_stream_t stream);

/* Split qkv rows fp32 [R][(Hq + 2 Hkv) D] = [q | k | v]; rotate q and k
 * (rotate-half) at each row's position; write q bf16 [R][Hq][D] and write k, v
 * (bf16) either into the paged cache at the row's position (k_stage == NULL) or
 * into staging rows k_stage/v_stage [R][Hkv][D]. */
spec_status spec_rope_append(const float *qkv, int R, int Hq, int Hkv, int D,
                             const float *rope_tab, int max_pos,
                             const int32_t *cu_rows, const int32_t *ctx_start, int S,
                             uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache, int num_pages,
                             const int32_t *block_table, int max_blocks,
                             uint16_t *k_stage, uint16_t *v_stage,
                             int32_t *dev_err, spec_stream_t stream);

/* out[r][i] = bf16(silu(gu[r][i]) * gu[r][F + i]); gu fp32 [R][2F]; out bf16 [R][F]. */
spec_status spec_swiglu(const float *gu, int R, int F, uint16_t *out, spec_stream_t stream);

/* spec_add_rmsnorm and spec_swiglu that also write their rows, as columns of
 * an 80-column K1 pass, in the packed form spec_qmatmul_packed reads: xpk of
 * spec_packed_activation_bytes(H or F) bytes, 16-byte aligned; R <= 80, H or F
 * a multiple of 256.  out is written as by the plain calls. */
spec_status spec_add_rmsnorm_packed(float *h, const float *delta, const float *w, int R, int H, float eps,
                                    uint16_t *out, void *xpk, spec_stream_t stream);
spec_status spec_swiglu_packed(const float *gu, int R, int F, uint16_t *out, void *xpk, spec_stream_t stream);

/* out[i] = bf16(in[i]) for i < n (round to nearest even). */
spec_status spec_cast_bf16(const float *in, size_t n, uint16_t *out, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * n-gram drafting on the device (tokenstrom.com, section "Why the math
 * checks out and the text still flips", and ramgpt.org, section "Flash
 * Attention Changes Geometry With Batch Width", both run n-gram speculation;
 * neither gives the rule, so this is a reading).  For each sequence s with
 * history hist[s][0 .. hist_len[s]-1] (row stride hist_cap): find the most
 * recent earlier occurrence of the last n tokens (n = 3, then 2, then 1),
 * propose the up to W tokens that followed it (never past the end of the
 * history) and fill the remaining slots from pad[s][slot].
 *   drafts        int32 [S][W]
 *   matched_n     int32 [S] or NULL: the n that matched (0: none)
 *   block_tokens  int32 [S][W + 1] or NULL: the next verify block, i.e. the
 *                 last history token followed by the W drafts
 * ---------------------------------------------------------------------- */
spec_status spec_ngram_draft(const int32_t *hist, int hist_cap, const int32_t *hist_len, int S, int W,
                             const int32_t *pad, int32_t *drafts, int32_t *matched_n,
                             int32_t *block_tokens, spec_stream_t stream);

/* Commit one verify step to the device-side histories: append drafts[s][0 ..
 * accepted[s]-1] and correction[s] to hist[s], advance hist_len[s] by
 * accepted[s] + 1 and copy ctx[s] = ctx_new[s].  A history that would overflow
 * hist_cap is left unchanged and sets SPEC_DEVERR_LENGTH. */
spec_status spec_commit_accepted(int32_t *hist, int hist_cap, int32_t *hist_len, const int32_t *drafts, int W,
                                 const int32_t *accepted, const int32_t *correction, const int32_t *ctx_new,
                                 int32_t *ctx, int S, int32_t *dev_err, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * Test hook: spec_qmatmul with an explicit column-tile width nt in {1, 2, 10,
 * 11} (columns per pass = 8 nt, 80 for 11; nt = 10 runs the 80-column pass on
 * the mma.sync kernel, nt = 11 on the tcgen05 kernel; the workspace must hold
 * T * (1 + ceil(K/512)) * 128 * 8 nt' floats after 256-byte-rounded T int
 * counters, T = ceil(N/128), nt' = min(nt, 10), and for nt >= 10 another
 * K/256 * 43520 bytes of packed activations).  The result of every column must
 * not depend on nt; the tests use this to show it.  y_dt is SPEC_F32.
 * ---------------------------------------------------------------------- */
spec_status spec_qmatmul_debug_nt(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                  int n_cols, int ldx, float *y, int ldy, int nt,
                                  void *workspace, size_t ws_bytes, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * Margin-gated re-check of the LM head
 *
 * tokenstrom.com, "'Lossless,' but not quite", section "Why the math checks
 * out and the text still flips" (only steps whose top-2 margin is small can
 * flip) and section "What the big servers offer and what it costs" (re-check
 * only the uncertain steps).  `logits` [R][V] fp32 come from a fast evaluation
 * (e.g. spec_qmatmul_noninvariant) of y = W x_r whose entries differ from the
 * invariant evaluation's (spec_qmatmul) by at most err_r = err_coef *
 * ||x_r||_1 (x_r: the bf16 row of `x` [R][ldx], H entries; err_coef is the
 * caller's summation-order bound for its matrix).  For each row:
 *   top[r]   = argmax of logits[r] (lowest index on ties; NaN never wins and
 *              sets SPEC_DEVERR_NAN);
 *   flagged  unless top-2 margin > 2 err_r (a tie is always flagged).
 * A row not flagged has the invariant evaluation's argmax.  The flagged rows
 * are listed in row order: rows[0 .. min(count, capacity)) (device int32),
 * their activations copied to x_gathered [capacity][H] bf16; *count = the
 * number flagged, *overflow = R when it exceeds capacity, else 0 (device
 * int32 each).  Re-evaluate with spec_qmatmul_devcols(x_gathered, n_cols =
 * capacity, dev_cols = count) into y_gathered [capacity][V], copy those rows
 * back with spec_gate_scatter, and (for overflow) spec_qmatmul_devcols over all
 * R rows with dev_cols = overflow, min_cols = 1.  The result: every row's
 * argmax equals the invariant argmax, with a fixed launch sequence.
 *   V % 4 == 0, H % 8 == 0, ldx % 8 == 0; logits, x, x_gathered, workspace
 *   16-byte aligned; workspace >= spec_margin_gate_workspace(R, V) bytes.
 * ---------------------------------------------------------------------- */
size_t spec_margin_gate_workspace(int R, int V);
spec_status spec_margin_gate(const float *logits, int V, int R, const uint16_t *x, int H, int ldx, float err_coef,
                             int32_t *top, int32_t *rows, int32_t *count, int32_t *overflow, int capacity,
                             uint16_t *x_gathered, void *workspace, size_t ws_bytes, int32_t *dev_err,
                             spec_stream_t stream);

/* Copies y_gathered[s] ([capacity][V] fp32) into logits[rows[s]] for s <
 * min(*count, capacity) (count, rows: device int32 from spec_margin_gate). */
spec_status spec_gate_scatter(const float *y_gathered, int V, const int32_t *rows, const int32_t *count,
                              int capacity, float *logits, spec_stream_t stream);

/* ------------------------------------------------------------------------
 * Test hook for the bounded-wait error path (the pages have no counterpart:
 * this exercises the library's own failure handling).  Launches one thread
 * that arms an mbarrier for 16 transaction bytes, issues no copy (so nothing
 * is in flight and the phase can never complete), and waits for it through
 * the same bounded wait every kernel uses, limited to `polls` polls.  When the
 * wait runs out the kernel ORs SPEC_DEVERR_TIMEOUT into *dev_err (device
 * memory) and returns normally; the context stays usable and later calls on
 * the stream run as usual.  polls must be in [1, 2^20]; dev_err non-NULL.
 * ---------------------------------------------------------------------- */
spec_status spec_debug_wait_timeout(uint32_t polls, int32_t *dev_err, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_H */
