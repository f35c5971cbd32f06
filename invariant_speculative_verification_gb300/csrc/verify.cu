// K4: ragged greedy verification and K5: KV-cache realignment.
//
// proofoftech.org, "'Lossless' speculative decoding isn't free": the target
// accepts the prefix of drafts it agrees with and corrects the first token it
// does not (opening section); sequences that accept different counts must
// have positions and KV state realigned exactly (section "Batching breaks the
// implementation").  ramgpt.org, "When Lossless Speculation Stops Being
// Lossless on Blackwell", section "The Hidden Contract Behind Lossless
// Speculation": greedy choice is the maximum-logit token.
//
// Every output here is an integer decided by exact comparisons (argmax over
// values compared in fp32, which holds bf16 and fp32 logits exactly), so the
// result cannot depend on the batch composition or the split of the scan.
#include <climits>

#include "common.cuh"

namespace {

constexpr int VT = 256;  // threads of the argmax scan

struct Best {
    float v;
    int i;
};

// larger value wins; equal values: lower index wins; NaN never wins
__device__ __forceinline__ Best better(Best a, Best b) {
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

// Temperature sampling (spec_verify_sample): the row's token is the argmax of
// fma(logit, inv_temp, g) with g = -log(-log(u)) a Gumbel variate; u comes from
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11) with counter (v / 4, position, sequence id, 0x53504543)
// and key (seed_lo, seed_hi), word v % 4: u = (w >> 9) 2^-23 + 2^-24.
struct SampleArgs {
    float inv_temp;
    uint32_t seed_lo, seed_hi;
    const int32_t *cu_rows, *ctx_start, *seq_id;
    int S;
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0, c1 = lo1, c2 = n2, c3 = lo0;
    }
    return make_uint4(c0, c1, c2, c3);
}

__device__ __forceinline__ float gumbel(uint32_t w) {
    const float u = __uint2float_rn(w >> 9) * (1.0f / 8388608.0f) + (1.0f / 16777216.0f);
    return -logf(-logf(u));
}

template <bool BF16, bool SAMPLE>
__global__ void __launch_bounds__(VT)
argmax_partial_kernel(const void *__restrict__ logits, int V, int split, int R, Best *__restrict__ part,
                      int32_t *dev_err, SampleArgs sa) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.y, sp = blockIdx.x;
    if (r >= R) return;
    constexpr int VEC = BF16 ? 8 : 4;
    const int nvec = V / VEC;
    const int v0 = (int)((long long)nvec * sp / split), v1 = (int)((long long)nvec * (sp + 1) / split);
    const uint4 *row = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(logits) +
                                                      (size_t)r * V * (BF16 ? 2 : 4));
    Best b{-INFINITY, INT_MAX};
    bool nan = false;
    // sampling: this row's sequence (the last s with cu_rows[s] <= r), position and identity
    uint32_t pos = 0, sid = 0;
    if (SAMPLE) {
        int lo = 0, hi = sa.S;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sa.cu_rows[mid] <= r) lo = mid; else hi = mid;
        }
        pos = (uint32_t)(sa.ctx_start[lo] + (r - sa.cu_rows[lo]));
        sid = (uint32_t)(sa.seq_id ? sa.seq_id[lo] : lo);
    }
    auto scan = [&](const uint4 &w, int v) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t rnd[8];
        if (SAMPLE) {
            // the 16-byte vector holds elements v*VEC .. v*VEC+VEC-1: counters (v*VEC)/4 ..
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const uint4 ph = philox4x32_10((uint32_t)((v * VEC) / 4 + q), pos, sid, 0x53504543u, sa.seed_lo,
                                               sa.seed_hi);
                rnd[4 * q] = ph.x, rnd[4 * q + 1] = ph.y, rnd[4 * q + 2] = ph.z, rnd[4 * q + 3] = ph.w;
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float x;
            if (BF16)
                x = __uint_as_float((e & 1) ? (u[e >> 1] & 0xFFFF0000u) : (u[e >> 1] << 16));
            else
                x = __uint_as_float(u[e]);
            nan |= (x != x);
            if (SAMPLE) x = fmaf(x, sa.inv_temp, gumbel(rnd[e]));
            const int idx = v * VEC + e;
            if (x > b.v || (x == b.v && idx < b.i)) {
                b.v = x;
                b.i = idx;
            }
        }
    };
    // four 16-byte loads in flight per thread; every comparison is exact, so the
    // order in which a thread visits its elements does not change the result
    constexpr int U = 4;
    int v = v0 + threadIdx.x;
    for (; v + (U - 1) * VT < v1; v += U * VT) {
        uint4 w[U];
#pragma unroll
        for (int j = 0; j < U; ++j) w[j] = __ldcs(row + v + j * VT);
#pragma unroll
        for (int j = 0; j < U; ++j) scan(w[j], v + j * VT);
    }
    for (; v < v1; v += VT) scan(__ldcs(row + v), v);
    if (nan) dev::report(dev_err, SPEC_DEVERR_NAN);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best other{__shfl_xor_sync(0xffffffffu, b.v, o), __shfl_xor_sync(0xffffffffu, b.i, o)};
        b = better(b, other);
    }
    __shared__ Best wb[VT / 32];
    if ((threadIdx.x & 31) == 0) wb[threadIdx.x >> 5] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best t = wb[0];
        for (int w = 1; w < VT / 32; ++w) t = better(t, wb[w]);
        part[(size_t)r * split + sp] = t;
    }
}

// one warp per sequence: finish the argmax of its rows, then accept / correct
__global__ void __launch_bounds__(128)
verify_finalize_kernel(const Best *__restrict__ part, int split, const int32_t *__restrict__ cu_rows, int S, int R,
                       int V, const int32_t *__restrict__ drafts, const int32_t *__restrict__ ctx_start,
                       int32_t *__restrict__ argmax_out, int32_t *__restrict__ accepted,
                       int32_t *__restrict__ correction, int32_t *__restrict__ ctx_new, int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int s = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= S) return;
    if (s == 0 && lane == 0 && cu_rows[S] != R) dev::report(dev_err, SPEC_DEVERR_LAYOUT);
    const int r0 = cu_rows[s], r1 = cu_rows[s + 1];
    if (r1 <= r0 || r0 < 0 || r1 > R) {
        if (lane == 0) dev::report(dev_err, SPEC_DEVERR_LAYOUT);
        return;
    }
    const int L = r1 - r0 - 1;
    int a = L;
    for (int base = 0; base <= L; base += 32) {
        const int i = base + lane;
        int am = 0;
        bool mismatch = false;
        if (i <= L) {
            const Best *p = part + (size_t)(r0 + i) * split;
            Best b = p[0];
            for (int q = 1; q < split; ++q) b = better(b, p[q]);
            am = (b.i == INT_MAX) ? 0 : b.i;  // an all-NaN row: index 0
            argmax_out[r0 + i] = am;
            if (i < L) {
                const int di = r0 - s + i;
                if (di >= R - S) {  // later sequences with no rows: drafts would overrun
                    dev::report(dev_err, SPEC_DEVERR_LAYOUT);
                    mismatch = true;
                } else {
                    const int d = drafts[di];
                    if (d < 0 || d >= V) dev::report(dev_err, SPEC_DEVERR_TOKEN_RANGE);
                    mismatch = (d != am);
                }
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, mismatch);
        if (m && a == L) a = min(a, base + __ffs(m) - 1);
    }
    __syncwarp();
    if (lane == 0) {
        accepted[s] = a;
        correction[s] = argmax_out[r0 + a];
        ctx_new[s] = ctx_start[s] + a + 1;
    }
}

int argmax_split(int R, int V) {
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    // as many splits as fit in one wave of eight CTAs per SM: rounding up left
    // a partial second wave (1312 CTAs for 1216 slots at 328 rows, 24.9 us
    // against 22.1 us for three splits; every split gives the same argmax)
    int sp = (8 * sms) / R;
    const int max_sp = V / 4096 > 0 ? V / 4096 : 1;  // at least 4096 logits per CTA
    if (sp > max_sp) sp = max_sp;
    if (sp < 1) sp = 1;
    return sp;
}

// ---------------------------------------------------------------------------
// K5
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
kv_compact_kernel(const uint16_t *__restrict__ k_stage, const uint16_t *__restrict__ v_stage,
                  uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache, int Hkv, int D, int num_pages,
                  const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_start,
                  const int32_t *__restrict__ accepted, const int32_t *__restrict__ cu_rows, int S, int R,
                  int32_t *__restrict__ cu_kept, int32_t *__restrict__ kept_src, int64_t *__restrict__ dst_slot,
                  int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ int sh_base;
    if (r == 0 && warp == 0) {
        // cu_kept = exclusive prefix sum of accepted + 1 (warp scan, chunks of 32)
        int run = 0;
        if (lane == 0) cu_kept[0] = 0;
        for (int b = 0; b < S; b += 32) {
            const int s = b + lane;
            int v = (s < S) ? accepted[s] + 1 : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += n;
            }
            if (s < S) cu_kept[s + 1] = run + v;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    // sequence of staged row r
    int lo = 0, hi = S;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu_rows[mid] <= r) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int i = r - cu_rows[s];
    const int a = accepted[s];
    if (i < 0 || i > a || r >= cu_rows[s + 1]) return;  // rejected rows never reach the cache
    if (warp == 0) {
        int sum = 0;
        for (int q = lane; q < s; q += 32) sum += accepted[q] + 1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) sh_base = sum;
    }
    __syncthreads();
    const int j = sh_base + i;
    if (j >= R) {  // accepted counts larger than the drafts: would overrun the index outputs
        if (threadIdx.x == 0) dev::report(dev_err, SPEC_DEVERR_LAYOUT);
        return;
    }
    const int pos = ctx_start[s] + i;
    const int blk = pos / 16, slot = pos % 16;
    int phys = -1;
    if (pos < 0 || blk >= max_blocks) {
        if (threadIdx.x == 0) dev::report(dev_err, SPEC_DEVERR_LENGTH);
    } else {
        phys = block_table[(size_t)s * max_blocks + blk];
        if (phys < 0 || phys >= num_pages) {
            if (threadIdx.x == 0) dev::report(dev_err, SPEC_DEVERR_BLOCK_TABLE);
            phys = -1;
        }
    }
    if (threadIdx.x == 0) {
        kept_src[j] = r;
        dst_slot[j] = phys < 0 ? -1 : (int64_t)phys * 16 + slot;
    }
    if (!k_stage || phys < 0) return;
    // copy Hkv rows of D 16-bit values for K and V (16 bytes per thread-step)
    const int vecs_per_head = D / 8;
    const int total = Hkv * vecs_per_head;
    for (int e = threadIdx.x; e < 2 * total; e += blockDim.x) {
        const bool isv = e >= total;
        const int ee = isv ? e - total : e;
        const int h = ee / vecs_per_head, c = ee % vecs_per_head;
        const uint4 *src = reinterpret_cast<const uint4 *>((isv ? v_stage : k_stage) + ((size_t)r * Hkv + h) * D) + c;
        uint4 *dst = reinterpret_cast<uint4 *>((isv ? v_cache : k_cache) + (((size_t)phys * Hkv + h) * 16 + slot) * D) + c;
        *dst = __ldg(src);
    }
}

}  // namespace

extern "C" size_t spec_verify_greedy_workspace(int R, int V) {
    if (R <= 0 || V <= 0) return 0;
    return (size_t)R * argmax_split(R, V) * sizeof(Best);
}

extern "C" spec_status spec_verify_greedy(const void *logits, spec_dtype dt, int V, const int32_t *cu_rows, int S,
                                          int R, const int32_t *drafts, const int32_t *ctx_start, int32_t *argmax_out,
                                          int32_t *accepted, int32_t *correction, int32_t *ctx_new, void *workspace,
                                          size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(dt == SPEC_F32 || dt == SPEC_BF16, "verify_greedy: dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(V >= 8 && V % 8 == 0, "verify_greedy: V must be a positive multiple of 8 (V=%d)", V);
    SPEC_CHECK_ARG(S >= 0 && R >= S && R <= 65535, "verify_greedy: need S <= R <= 65535 (S=%d R=%d)", S, R);
    SPEC_CHECK_ARG(cu_rows && ctx_start && argmax_out && accepted && correction && ctx_new &&
                       (logits || R == 0) && (drafts || R == S),
                   "verify_greedy: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(logits), "verify_greedy: logits must be 16-byte aligned");
    if (S == 0) return SPEC_OK;
    const int split = argmax_split(R, V);
    const size_t need = (size_t)R * split * sizeof(Best);
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "verify_greedy: workspace needs %zu bytes, got %zu", need, ws_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    Best *part = reinterpret_cast<Best *>(workspace);
    dim3 grid(split, R);
    const SampleArgs none{};
    cudaError_t le = (dt == SPEC_BF16)
                         ? spec::launch_pdl(argmax_partial_kernel<true, false>, grid, dim3(VT), 0, st, logits, V, split,
                                            R, part, dev_err, none)
                         : spec::launch_pdl(argmax_partial_kernel<false, false>, grid, dim3(VT), 0, st, logits, V,
                                            split, R, part, dev_err, none);
    if (le != cudaSuccess) return spec::cuda_status(le, "argmax launch");
    le = spec::launch_pdl(verify_finalize_kernel, dim3((S + 3) / 4), dim3(128), 0, st, (const Best *)part, split, cu_rows,
                          S, R, V, drafts, ctx_start, argmax_out, accepted, correction, ctx_new, dev_err);
    return spec::cuda_status(le, "verify finalize launch");
}

extern "C" spec_status spec_verify_sample(const void *logits, spec_dtype dt, int V, const int32_t *cu_rows, int S,
                                          int R, const int32_t *drafts, const int32_t *ctx_start,
                                          const int32_t *seq_id, float inv_temperature, uint64_t seed,
                                          int32_t *token_out, int32_t *accepted, int32_t *correction,
                                          int32_t *ctx_new, void *workspace, size_t ws_bytes, int32_t *dev_err,
                                          spec_stream_t stream) {
    SPEC_CHECK_ARG(dt == SPEC_F32 || dt == SPEC_BF16, "verify_sample: dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(V >= 8 && V % 8 == 0, "verify_sample: V must be a positive multiple of 8 (V=%d)", V);
    SPEC_CHECK_ARG(S >= 0 && R >= S && R <= 65535, "verify_sample: need S <= R <= 65535 (S=%d R=%d)", S, R);
    SPEC_CHECK_ARG(inv_temperature > 0.f && inv_temperature < INFINITY,
                   "verify_sample: inv_temperature must be positive and finite");
    SPEC_CHECK_ARG(cu_rows && ctx_start && token_out && accepted && correction && ctx_new &&
                       (logits || R == 0) && (drafts || R == S),
                   "verify_sample: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(logits), "verify_sample: logits must be 16-byte aligned");
    if (S == 0) return SPEC_OK;
    const int split = argmax_split(R, V);
    const size_t need = (size_t)R * split * sizeof(Best);
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "verify_sample: workspace needs %zu bytes, got %zu", need, ws_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    Best *part = reinterpret_cast<Best *>(workspace);
    const SampleArgs sa{inv_temperature, (uint32_t)seed, (uint32_t)(seed >> 32), cu_rows, ctx_start, seq_id, S};
    dim3 grid(split, R);
    cudaError_t le = (dt == SPEC_BF16)
                         ? spec::launch_pdl(argmax_partial_kernel<true, true>, grid, dim3(VT), 0, st, logits, V, split,
                                            R, part, dev_err, sa)
                         : spec::launch_pdl(argmax_partial_kernel<false, true>, grid, dim3(VT), 0, st, logits, V,
                                            split, R, part, dev_err, sa);
    if (le != cudaSuccess) return spec::cuda_status(le, "sample launch");
    le = spec::launch_pdl(verify_finalize_kernel, dim3((S + 3) / 4), dim3(128), 0, st, (const Best *)part, split, cu_rows,
                          S, R, V, drafts, ctx_start, token_out, accepted, correction, ctx_new, dev_err);
    return spec::cuda_status(le, "verify finalize launch");
}

extern "C" spec_status spec_kv_compact(const void *k_stage, const void *v_stage, void *k_cache, void *v_cache,
                                       int Hkv, int D, int num_pages, const int32_t *block_table, int max_blocks,
                                       const int32_t *ctx_start, const int32_t *accepted, const int32_t *cu_rows,
                                       int S, int R, int32_t *cu_kept, int32_t *kept_src, int64_t *dst_slot,
                                       int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(Hkv >= 1 && D >= 8 && D % 8 == 0, "kv_compact: need Hkv >= 1 and D %% 8 == 0 (Hkv=%d D=%d)", Hkv,
                   D);
    SPEC_CHECK_ARG(S >= 0 && R >= S && num_pages >= 1 && max_blocks >= 1,
                   "kv_compact: bad sizes (S=%d R=%d num_pages=%d max_blocks=%d)", S, R, num_pages, max_blocks);
    SPEC_CHECK_ARG((k_stage == nullptr) == (v_stage == nullptr), "kv_compact: k_stage and v_stage both or neither");
    SPEC_CHECK_ARG(block_table && ctx_start && accepted && cu_rows && cu_kept && kept_src && dst_slot,
                   "kv_compact: NULL pointer");
    SPEC_CHECK_ARG(!k_stage || (k_cache && v_cache && spec::aligned16(k_stage) && spec::aligned16(v_stage) &&
                                spec::aligned16(k_cache) && spec::aligned16(v_cache)),
                   "kv_compact: stage and cache pointers must be non-NULL and 16-byte aligned");
    if (S == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(
        kv_compact_kernel, dim3(R), dim3(256), 0, (cudaStream_t)stream, reinterpret_cast<const uint16_t *>(k_stage),
        reinterpret_cast<const uint16_t *>(v_stage), reinterpret_cast<uint16_t *>(k_cache),
        reinterpret_cast<uint16_t *>(v_cache), Hkv, D, num_pages, block_table, max_blocks, ctx_start, accepted, cu_rows,
        S, R, cu_kept, kept_src, dst_slot, dev_err);
    return spec::cuda_status(le, "kv_compact launch");
}
