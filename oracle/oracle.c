/*
 * CPU oracle for batch-invariant greedy speculative verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * definition of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library never
 * does.  It shares no code, header, table or helper with the CUDA sources.
 *
 * Every floating-point accumulation is in double precision and in plain index
 * order.  Storage formats decoded here (bf16, fp16, int4 nibbles) are decoded
 * from their definitions, not with any GPU intrinsic.
 *
 * Sources (titles of the pages the method is taken from):
 *  [T] tokenstrom.com, "'Lossless,' but not quite: why speculative decoding
 *      changes your LLM's answers"
 *  [R] ramgpt.org, "When Lossless Speculation Stops Being Lossless on Blackwell"
 *  [P] proofoftech.org, "'Lossless' speculative decoding isn't free"
 *
 * The pages define the method in words; where they are silent the plainest
 * reading is taken and named at the function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2
#define OR_PAGE 16

/* ---------------------------------------------------------------------------
 * storage formats
 * ------------------------------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double or_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double or_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Round to bfloat16, nearest with ties to even (8 significant bits). */
uint16_t or_double_to_bf16(double x)
{
    float f;
    uint32_t u;
    if (isnan(x))
        return 0x7fc0;
    if (x == 0.0) {
        f = (float)x;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    int e;
    double m = frexp(fabs(x), &e);           /* |x| = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 8));       /* 8 significant bits, ties to even */
    double y = ldexp(r, e - 8);
    f = (float)(x < 0 ? -y : y);             /* exact: y has 8 significant bits */
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double or_elem(const void *p, int dt, size_t i)
{
    switch (dt) {
    case OR_F32: return (double)((const float *)p)[i];
    case OR_F16: return or_f16_to_double(((const uint16_t *)p)[i]);
    default: return or_bf16_to_double(((const uint16_t *)p)[i]);
    }
}

/* ---------------------------------------------------------------------------
 * 1. block-quantised matrix multiplication
 *
 * [R] "Quantized Matrix Multiplication Shows the Same Class of Failure": the
 * operation whose batched result must equal the concatenation of single-column
 * results.  [T] "Why the math checks out and the text still flips": Q4_K-style
 * quantised weights in the matrix-vector product.  The pages define no format;
 * the stand-in is int4 in blocks of 32 along K with one fp16 scale per block:
 *
 *   y[j][n] = sum_k x[j][k] * d[n][k/32] * (nibble(n, k) - 8)
 *
 * nibble(n, k) is the low nibble of byte wq[n][k/2] for even k, the high
 * nibble for odd k.  x is bf16 [n_cols][ldx]; y is [n_cols][N].
 * ------------------------------------------------------------------------- */
void oracle_qmatmul(const uint8_t *wq, const uint16_t *ws, int N, int K,
                    const uint16_t *x, int n_cols, int ldx, double *y)
{
    for (int j = 0; j < n_cols; ++j) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < K / 32; ++b) {
                double d = or_f16_to_double(ws[(size_t)n * (K / 32) + b]);
                for (int k = 32 * b; k < 32 * b + 32; ++k) {
                    uint8_t byte = wq[(size_t)n * (K / 2) + k / 2];
                    int nib = (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
                    double q = (double)(nib - 8);
                    double xv = or_bf16_to_double(x[(size_t)j * ldx + k]);
                    acc += xv * d * q;   /* the product is exact in double */
                }
            }
            y[(size_t)j * N + n] = acc;
        }
    }
}

/* ---------------------------------------------------------------------------
 * 1b. the same product with two-level (super-block) scales
 *
 * [T] "Why the math checks out and the text still flips" names Q4_K / Q6_K
 * (llama.cpp K-quants, scales in two levels) and [R] "Quantized Matrix
 * Multiplication Shows the Same Class of Failure" names IQ3_S / IQ4_XS; the
 * pages define none of them, so this format is self-defined in their spirit:
 * the same 4-bit codes, and per row and per 256-k super-block one 8-byte record
 * (read as a little-endian 64-bit word):
 *
 *   bits 6j .. 6j+5   s_j in 0 .. 63, the scale of 32-k block j of the super-block
 *   bits 48 .. 63     D, an fp16 super-scale
 *
 * Block b's scale is D * s_(b mod 8).  A row holds ceil(K/512) pairs of records
 * (16 bytes each; when K/256 is odd the last record is padding):
 *
 *   y[j][n] = sum_k x[j][k] * D[n][k/256] * s[n][k/32] * (nibble(n, k) - 8)
 * ------------------------------------------------------------------------- */
void oracle_sb_record(const uint8_t *rec, int32_t *s, double *D)
{
    uint64_t w = 0;
    for (int i = 7; i >= 0; --i) w = (w << 8) | rec[i];   /* little-endian */
    for (int j = 0; j < 8; ++j) s[j] = (int32_t)((w >> (6 * j)) & 63u);
    *D = or_f16_to_double((uint16_t)(w >> 48));
}

void oracle_qmatmul_sb(const uint8_t *wq, const uint8_t *sbr, int N, int K,
                       const uint16_t *x, int n_cols, int ldx, double *y)
{
    const int pitch = (K + 511) / 512 * 16;   /* bytes of records per row */
    for (int j = 0; j < n_cols; ++j) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int sb = 0; sb < K / 256; ++sb) {
                int32_t s[8];
                double D;
                oracle_sb_record(sbr + (size_t)n * pitch + 8 * sb, s, &D);
                for (int k = 256 * sb; k < 256 * sb + 256; ++k) {
                    uint8_t byte = wq[(size_t)n * (K / 2) + k / 2];
                    int nib = (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
                    double d = D * (double)s[(k / 32) % 8];
                    double xv = or_bf16_to_double(x[(size_t)j * ldx + k]);
                    acc += xv * d * (double)(nib - 8);   /* exact in double */
                }
            }
            y[(size_t)j * N + n] = acc;
        }
    }
}

/* ---------------------------------------------------------------------------
 * 2. causal softmax attention over a paged KV cache
 *
 * [R] "Flash Attention Changes Geometry With Batch Width": attention for the
 * rows of a verify block.  [R] "The Hidden Contract Behind Lossless
 * Speculation": the block's rows are the positions ordinary decoding would
 * have evaluated one at a time, so row i of sequence s, at absolute position
 * p = ctx_start[s] + i, attends to keys 0 .. p and to nothing after it.
 *
 *   s_j  = scale * sum_d q[d] k_j[d]          j = 0 .. p
 *   out  = sum_j exp(s_j - max s) v_j / sum_j exp(s_j - max s)
 *
 * Query head h reads KV head h / (Hq / Hkv) (grouped heads, contiguous groups).
 * Key j of sequence s lives in page block_table[s][j / 16], slot j % 16; the
 * cache is [pages][Hkv][16][D].  q is [R][Hq][D]; out is [R][Hq][D].  When
 * want is not NULL only the (row, head) pairs with want[r * Hq + h] != 0 are
 * computed (rows and heads are independent of one another).
 * ------------------------------------------------------------------------- */
void oracle_attention(const void *q, int dt, int Hq, int Hkv, int D, double scale,
                      const void *k_cache, const void *v_cache,
                      const int32_t *block_table, int max_blocks,
                      const int32_t *ctx_start, const int32_t *cu_rows, int S,
                      const uint8_t *want, double *out)
{
    int group = Hq / Hkv;
    for (int s = 0; s < S; ++s) {
        int rows = cu_rows[s + 1] - cu_rows[s];
        int len = ctx_start[s] + rows;
        double *score = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
        for (int i = 0; i < rows; ++i) {
            int r = cu_rows[s] + i;
            int p = ctx_start[s] + i;
            for (int h = 0; h < Hq; ++h) {
                if (want && !want[(size_t)r * Hq + h])
                    continue;
                int kvh = h / group;
                double smax = -INFINITY;
                for (int j = 0; j <= p; ++j) {
                    int page = block_table[(size_t)s * max_blocks + j / OR_PAGE];
                    size_t kb = (((size_t)page * Hkv + kvh) * OR_PAGE + j % OR_PAGE) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += or_elem(q, dt, ((size_t)r * Hq + h) * D + d) * or_elem(k_cache, dt, kb + d);
                    score[j] = scale * dot;
                    if (score[j] > smax)
                        smax = score[j];
                }
                double denom = 0.0;
                for (int j = 0; j <= p; ++j)
                    denom += exp(score[j] - smax);
                /* score[j] now becomes the softmax weight of key j */
                for (int j = 0; j <= p; ++j)
                    score[j] = exp(score[j] - smax) / denom;
                for (int d = 0; d < D; ++d)
                    out[((size_t)r * Hq + h) * D + d] = 0.0;
                for (int j = 0; j <= p; ++j) {
                    int page = block_table[(size_t)s * max_blocks + j / OR_PAGE];
                    size_t vb = (((size_t)page * Hkv + kvh) * OR_PAGE + j % OR_PAGE) * D;
                    for (int d = 0; d < D; ++d)
                        out[((size_t)r * Hq + h) * D + d] += score[j] * or_elem(v_cache, dt, vb + d);
                }
            }
        }
        free(score);
    }
}

/* ---------------------------------------------------------------------------
 * 3. greedy verification
 *
 * [P] "Lossless is a theorem, and theorems have hypotheses" / first section:
 * the target verifies the drafted tokens in one pass, accepts the prefix it
 * agrees with and corrects the first token it does not.  [R] "The Hidden
 * Contract Behind Lossless Speculation": under greedy decoding the target's
 * choice at each position is the maximum-logit token.
 *
 * Sequence s owns verify rows r0 = cu_rows[s] .. cu_rows[s+1]-1, i.e. L + 1
 * rows for L drafts; drafts[r0 - s + i] is the token proposed for the position
 * that row r0 + i predicts.
 *   argmax[r]      = smallest index of the row maximum (reading: ties go to
 *                    the lowest index; the pages do not say)
 *   accepted[s]    = first i < L with drafts[i] != argmax[r0 + i], else L
 *   correction[s]  = argmax[r0 + accepted[s]]
 *   ctx_new[s]     = ctx_start[s] + accepted[s] + 1
 * Returns the number of NaN logits seen (inputs are expected to be finite).
 * ------------------------------------------------------------------------- */
int oracle_verify_greedy(const void *logits, int dt, int V, const int32_t *cu_rows, int S,
                         const int32_t *drafts, const int32_t *ctx_start,
                         int32_t *argmax, int32_t *accepted, int32_t *correction,
                         int32_t *ctx_new)
{
    int nans = 0;
    int R = cu_rows[S];
    for (int r = 0; r < R; ++r) {
        int best = 0;
        double bv = or_elem(logits, dt, (size_t)r * V);
        if (isnan(bv))
            ++nans;
        for (int v = 1; v < V; ++v) {
            double x = or_elem(logits, dt, (size_t)r * V + v);
            if (isnan(x))
                ++nans;
            if (x > bv || (isnan(bv) && !isnan(x))) {
                bv = x;
                best = v;
            }
        }
        argmax[r] = best;
    }
    for (int s = 0; s < S; ++s) {
        int r0 = cu_rows[s];
        int L = cu_rows[s + 1] - r0 - 1;
        int a = 0;
        while (a < L && drafts[r0 - s + a] == argmax[r0 + a])
            ++a;
        accepted[s] = a;
        correction[s] = argmax[r0 + a];
        ctx_new[s] = ctx_start[s] + a + 1;
    }
    return nans;
}

/* ---------------------------------------------------------------------------
 * 3b. Speculative verification with temperature sampling
 *
 * ramgpt.org, "When Lossless Speculation Stops Being Lossless on Blackwell",
 * section "A Better Backend Test Matrix": the byte-identity requirement is
 * stated for greedy decoding; the method's extension to sampling (keep the
 * random draws tied to the sequence and the position, not to the batch) is
 * our reading.  Each verify row r of sequence s at absolute position p draws
 * its token as
 *     t_r = argmax_v  fma(logit[r][v], inv_temp, g(id_s, p, v))    (ties: lower v)
 * where id_s is the sequence's identity (seq_id[s], or s when seq_id is NULL)
 * with a Gumbel variate g = -log(-log(u)), u = (b >> 9) * 2^-23 + 2^-24 and
 * b = word (v mod 4) of Philox4x32-10(counter = (v / 4, p, s, 0x53504543),
 * key = (seed_lo, seed_hi)).  Gumbel-max makes t_r an exact sample of
 * softmax(logit / T).  Drafts are accepted while draft_i == t_{r0+i}; the
 * correction is t at the first mismatch (or of the last row).  A width-1
 * decode with the same seed draws the same tokens at the same positions, so
 * speculative sampling reproduces it byte for byte.  Scores are computed in
 * fp32 with a fused multiply-add, as a kernel computes them.
 *
 * Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of
 * two 32x32->64-bit products with multipliers 0xD2511F53 and 0xCD9E8D57 and
 * a key advanced by the Weyl constants 0x9E3779B9 and 0xBB67AE85 between
 * rounds.
 * ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0, c1 = n1, c2 = n2, c3 = n3;
    }
    out[0] = c0, out[1] = c1, out[2] = c2, out[3] = c3;
}

static float or_sample_score(float x, float inv_temp, uint32_t seed_lo, uint32_t seed_hi, int s, int p, int v)
{
    const uint32_t ctr[4] = {(uint32_t)v / 4u, (uint32_t)p, (uint32_t)s, 0x53504543u};
    const uint32_t key[2] = {seed_lo, seed_hi};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    const float u = (float)(w[v % 4] >> 9) * (1.0f / 8388608.0f) + (1.0f / 16777216.0f);
    const float g = -logf(-logf(u));
    return fmaf(x, inv_temp, g);
}

int oracle_verify_sample(const void *logits, int dt, int V, const int32_t *cu_rows, int S,
                         const int32_t *drafts, const int32_t *ctx_start, const int32_t *seq_id, float inv_temp,
                         uint32_t seed_lo, uint32_t seed_hi,
                         int32_t *token, int32_t *accepted, int32_t *correction, int32_t *ctx_new,
                         float *top2_gap)
{
    int nans = 0;
    for (int s = 0; s < S; ++s) {
        for (int r = cu_rows[s]; r < cu_rows[s + 1]; ++r) {
            const int p = ctx_start[s] + (r - cu_rows[s]);
            int best = -1;
            float bv = 0.f, second = -INFINITY;
            for (int v = 0; v < V; ++v) {
                const float x = (float)or_elem(logits, dt, (size_t)r * V + v);
                if (isnan(x)) {
                    ++nans;
                    continue;
                }
                const float sc = or_sample_score(x, inv_temp, seed_lo, seed_hi, seq_id ? seq_id[s] : s, p, v);
                if (best < 0 || sc > bv) {
                    if (best >= 0) second = bv;
                    bv = sc;
                    best = v;
                } else if (sc > second) {
                    second = sc;
                }
            }
            token[r] = best < 0 ? 0 : best;
            if (top2_gap) top2_gap[r] = bv - second;
        }
    }
    for (int s = 0; s < S; ++s) {
        int r0 = cu_rows[s];
        int L = cu_rows[s + 1] - r0 - 1;
        int a = 0;
        while (a < L && drafts[r0 - s + a] == token[r0 + a])
            ++a;
        accepted[s] = a;
        correction[s] = token[r0 + a];
        ctx_new[s] = ctx_start[s] + a + 1;
    }
    return nans;
}

/* ---------------------------------------------------------------------------
 * 4. KV-cache realignment after ragged acceptance
 *
 * [P] "Batching breaks the implementation": sequences in a batch accept
 * different numbers of drafts, after which positions and per-sequence KV state
 * must be realigned exactly.  Reading: the block's K/V rows were computed into
 * a staging buffer; rows 0 .. accepted[s] of sequence s (the last emitted
 * token and the accepted drafts) are kept and written to the cache slots of
 * positions ctx_start[s] .. ctx_start[s] + accepted[s]; rejected rows never
 * reach the cache.  With k_stage == NULL the rows were written to the cache
 * in place and only the index outputs are produced.
 *   cu_kept[s]  = sum_{t < s} (accepted[t] + 1)
 *   kept_src[j] = staging row of kept token j
 *   dst_slot[j] = page * 16 + slot of kept token j
 * Elements are copied as opaque 16-bit values; stage is [R][Hkv][D].
 * ------------------------------------------------------------------------- */
void oracle_kv_compact(const uint16_t *k_stage, const uint16_t *v_stage,
                       uint16_t *k_cache, uint16_t *v_cache, int Hkv, int D,
                       const int32_t *block_table, int max_blocks,
                       const int32_t *ctx_start, const int32_t *accepted,
                       const int32_t *cu_rows, int S,
                       int32_t *cu_kept, int32_t *kept_src, int64_t *dst_slot)
{
    cu_kept[0] = 0;
    for (int s = 0; s < S; ++s)
        cu_kept[s + 1] = cu_kept[s] + accepted[s] + 1;
    for (int s = 0; s < S; ++s) {
        for (int i = 0; i <= accepted[s]; ++i) {
            int j = cu_kept[s] + i;
            int pos = ctx_start[s] + i;
            int page = block_table[(size_t)s * max_blocks + pos / OR_PAGE];
            int slot = pos % OR_PAGE;
            int src = cu_rows[s] + i;
            kept_src[j] = src;
            dst_slot[j] = (int64_t)page * OR_PAGE + slot;
            if (k_stage) {
                for (int h = 0; h < Hkv; ++h) {
                    for (int d = 0; d < D; ++d) {
                        size_t dst = (((size_t)page * Hkv + h) * OR_PAGE + slot) * D + d;
                        size_t from = ((size_t)src * Hkv + h) * D + d;
                        k_cache[dst] = k_stage[from];
                        v_cache[dst] = v_stage[from];
                    }
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * 5. decoder pieces for the end-to-end greedy generation workload
 *
 * The pages run real decoders; the workload here is a random-init decoder
 * whose parts are plain textbook definitions (readings, the pages name none):
 * RMSNorm with eps, rotate-half rotary embedding with base theta, a SwiGLU
 * feed-forward, int4 block-32 linear layers without bias, bf16 activations
 * entering every matmul, an fp32 residual stream and fp32 logits.
 * ------------------------------------------------------------------------- */

/* y = x / sqrt(mean(x^2) + eps) * w */
void oracle_rmsnorm(const double *x, int H, const float *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < H; ++i)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; ++i)
        y[i] = x[i] * inv * (double)w[i];
}

/* rotate-half: pair (i, i + D/2) rotated by angle pos * theta^(-2i/D) */
void oracle_rope(double *v, int D, int pos, double theta)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double a = (double)pos * pow(theta, -2.0 * i / D);
        double x1 = v[i], x2 = v[i + half];
        v[i] = x1 * cos(a) - x2 * sin(a);
        v[i + half] = x2 * cos(a) + x1 * sin(a);
    }
}

/* silu(g) * u with silu(g) = g / (1 + e^-g) */
double oracle_silu_mul(double g, double u)
{
    return g / (1.0 + exp(-g)) * u;
}

/* One int4 linear layer applied to one bf16 activation row: y[n] = sum_k ... */
static void or_linear_row(const uint8_t *wq, const uint16_t *ws, int N, int K,
                          const uint16_t *x_bf16, double *y)
{
    oracle_qmatmul(wq, ws, N, K, x_bf16, 1, K, y);
}

/*
 * One decoder layer over a verify batch, in place on the residual stream h
 * ([R][H], float32).  Sequence s's rows sit at positions ctx_start[s] + i.
 * The layer writes the block rows' K and V (bf16) into the paged cache before
 * attending, so each row sees the cached prefix plus the block rows up to and
 * including itself.
 *   a    = bf16(rmsnorm(h, norm1))
 *   qkv  = Wqkv a                       rows [q | k | v]
 *   q, k = rope(q), rope(k) at the row's position; q, k, v rounded to bf16
 *   o    = bf16(attention(q, cache))    scale 1/sqrt(head_dim)
 *   h    = fp32(h + Wo o)
 *   a    = bf16(rmsnorm(h, norm2))
 *   h    = fp32(h + Wdown bf16(silu(gate) * up))   gate/up rows [gate | up]
 */
void oracle_decoder_layer(float *h, int R, int H, int Hq, int Hkv, int D, int F,
                          double eps, double theta,
                          const uint8_t *qkv_q, const uint16_t *qkv_s,
                          const uint8_t *o_q, const uint16_t *o_s,
                          const uint8_t *gu_q, const uint16_t *gu_s,
                          const uint8_t *dn_q, const uint16_t *dn_s,
                          const float *norm1, const float *norm2,
                          uint16_t *k_cache, uint16_t *v_cache,
                          const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_start, const int32_t *cu_rows, int S)
{
    int nqkv = (Hq + 2 * Hkv) * D;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(H > F ? H : F));
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(nqkv > 2 * F ? nqkv : 2 * F));
    uint16_t *a = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(H > F ? H : F));
    uint16_t *qb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)R * Hq * D);
    double *att = (double *)malloc(sizeof(double) * (size_t)R * Hq * D);
    uint16_t *attb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hq * D);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);

    /* attention sub-block: q/k/v per row, K/V into the cache */
    for (int s = 0; s < S; ++s) {
        for (int r = cu_rows[s]; r < cu_rows[s + 1]; ++r) {
            int pos = ctx_start[s] + (r - cu_rows[s]);
            for (int i = 0; i < H; ++i)
                xd[i] = h[(size_t)r * H + i];
            oracle_rmsnorm(xd, H, norm1, eps, tmp);
            for (int i = 0; i < H; ++i)
                a[i] = or_double_to_bf16(tmp[i]);
            or_linear_row(qkv_q, qkv_s, nqkv, H, a, tmp);
            for (int hh = 0; hh < Hq; ++hh) {
                oracle_rope(tmp + (size_t)hh * D, D, pos, theta);
                for (int d = 0; d < D; ++d)
                    qb[((size_t)r * Hq + hh) * D + d] = or_double_to_bf16(tmp[(size_t)hh * D + d]);
            }
            int page = block_table[(size_t)s * max_blocks + pos / OR_PAGE];
            for (int kh = 0; kh < Hkv; ++kh) {
                double *kv = tmp + (size_t)(Hq + kh) * D;
                double *vv = tmp + (size_t)(Hq + Hkv + kh) * D;
                oracle_rope(kv, D, pos, theta);
                size_t dst = (((size_t)page * Hkv + kh) * OR_PAGE + pos % OR_PAGE) * D;
                for (int d = 0; d < D; ++d) {
                    k_cache[dst + d] = or_double_to_bf16(kv[d]);
                    v_cache[dst + d] = or_double_to_bf16(vv[d]);
                }
            }
        }
    }
    oracle_attention(qb, OR_BF16, Hq, Hkv, D, 1.0 / sqrt((double)D), k_cache, v_cache,
                     block_table, max_blocks, ctx_start, cu_rows, S, NULL, att);

    int Rtot = cu_rows[S];
    for (int r = 0; r < Rtot; ++r) {
        for (int i = 0; i < Hq * D; ++i)
            attb[i] = or_double_to_bf16(att[(size_t)r * Hq * D + i]);
        or_linear_row(o_q, o_s, H, Hq * D, attb, y);
        for (int i = 0; i < H; ++i)
            h[(size_t)r * H + i] = (float)((double)h[(size_t)r * H + i] + y[i]);

        for (int i = 0; i < H; ++i)
            xd[i] = h[(size_t)r * H + i];
        oracle_rmsnorm(xd, H, norm2, eps, tmp);
        for (int i = 0; i < H; ++i)
            a[i] = or_double_to_bf16(tmp[i]);
        or_linear_row(gu_q, gu_s, 2 * F, H, a, tmp);
        for (int i = 0; i < F; ++i)
            a[i] = or_double_to_bf16(oracle_silu_mul(tmp[i], tmp[F + i]));
        or_linear_row(dn_q, dn_s, H, F, a, y);
        for (int i = 0; i < H; ++i)
            h[(size_t)r * H + i] = (float)((double)h[(size_t)r * H + i] + y[i]);
    }
    free(xd); free(tmp); free(a); free(qb); free(att); free(attb); free(y);
}

/* Embedding lookup into the fp32 residual stream. */
void oracle_embed(const uint16_t *emb, int H, const int32_t *tokens, int R, float *h)
{
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < H; ++i)
            h[(size_t)r * H + i] = (float)or_bf16_to_double(emb[(size_t)tokens[r] * H + i]);
}

/* Final norm and LM head: logits[r][v] (fp32) = Wlm bf16(rmsnorm(h)). */
void oracle_lm_head(const float *h, int R, int H, const float *norm, double eps,
                    const uint8_t *lm_q, const uint16_t *lm_s, int V, float *logits)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    double *t = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)V);
    uint16_t *a = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
    for (int r = 0; r < R; ++r) {
        for (int i = 0; i < H; ++i)
            xd[i] = h[(size_t)r * H + i];
        oracle_rmsnorm(xd, H, norm, eps, t);
        for (int i = 0; i < H; ++i)
            a[i] = or_double_to_bf16(t[i]);
        or_linear_row(lm_q, lm_s, V, H, a, y);
        for (int v = 0; v < V; ++v)
            logits[(size_t)r * V + v] = (float)y[v];
    }
    free(xd); free(t); free(y); free(a);
}

/* ---------------------------------------------------------------------------
 * 6. n-gram drafting
 *
 * [T] "Why the math checks out and the text still flips" and [R] "Flash
 * Attention Changes Geometry With Batch Width" run n-gram speculation, which
 * proposes tokens from the sequence's own history.  Reading (the pages give no
 * rule): take the most recent earlier occurrence of the last n tokens, n = 3,
 * then 2, then 1; propose the up to W tokens that followed it (never past the
 * end of the history); fill the remaining slots from pad[].
 * Returns the n that matched, 0 when none did.
 * ------------------------------------------------------------------------- */
int oracle_ngram_draft(const int32_t *hist, int len, int W, const int32_t *pad, int32_t *out)
{
    for (int n = 3; n >= 1; --n) {
        if (len < n + 1)
            continue;
        for (int j = len - n - 1; j >= 0; --j) {
            int match = 1;
            for (int t = 0; t < n; ++t) {
                if (hist[j + t] != hist[len - n + t]) {
                    match = 0;
                    break;
                }
            }
            if (!match)
                continue;
            int c = 0;
            while (c < W && j + n + c < len) {
                out[c] = hist[j + n + c];
                ++c;
            }
            for (; c < W; ++c)
                out[c] = pad[c];
            return n;
        }
    }
    for (int c = 0; c < W; ++c)
        out[c] = pad[c];
    return 0;
}

/* ---------------------------------------------------------------------------
 * 7. margin-gated re-check
 *
 * [T] "Why the math checks out and the text still flips" (MarginGate: only the
 * steps whose top-2 margin is small can flip) and "What the big servers offer
 * and what it costs" (re-check only the uncertain steps).  The pages give the
 * idea, not a rule.  Reading: a row's logits come from a fast evaluation whose
 * every entry lies within err[r] of the invariant evaluation's; the row is
 * re-checked unless its top-2 margin exceeds 2 err[r] -- then no other entry can
 * reach the top one in the invariant logits, so both argmaxes agree.
 *
 * For each row r of logits [R][V] (fp32): top = the largest entry (lowest index
 * on ties), margin = top value - the largest value at any other index (0 on a
 * tie), recheck = (margin <= 2 err[r]).  Returns the number of rows flagged.
 * ------------------------------------------------------------------------- */
int oracle_margin_gate(const float *logits, int R, int V, const double *err, int32_t *top, double *margin,
                       uint8_t *recheck)
{
    int n = 0;
    for (int r = 0; r < R; ++r) {
        const float *row = logits + (size_t)r * V;
        int best = 0;
        for (int v = 1; v < V; ++v)
            if (row[v] > row[best])
                best = v;
        double second = -INFINITY;
        for (int v = 0; v < V; ++v)
            if (v != best && (double)row[v] > second)
                second = (double)row[v];
        top[r] = best;
        margin[r] = V > 1 ? (double)row[best] - second : INFINITY;
        recheck[r] = margin[r] <= 2.0 * err[r] ? 1 : 0;
        n += recheck[r];
    }
    return n;
}
