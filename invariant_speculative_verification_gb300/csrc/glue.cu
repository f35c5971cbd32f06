// Decoder glue and n-gram drafting for the end-to-end greedy generation
// workload.  Every floating-point kernel here works on one row at a time with a
// reduction order fixed by the row length, so it is width-invariant.
#include "qmm_shared.cuh"

namespace {

__global__ void embed_kernel(const uint16_t *__restrict__ emb, int V, int H, const int32_t *__restrict__ tokens,
                             float *__restrict__ h, int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.x;
    int tok = tokens[r];
    const bool bad = tok < 0 || tok >= V;
    if (bad && threadIdx.x == 0) dev::report(dev_err, SPEC_DEVERR_TOKEN_RANGE);
    for (int i = threadIdx.x; i < H; i += blockDim.x)
        h[(size_t)r * H + i] = bad ? 0.f : __uint_as_float((uint32_t)emb[(size_t)tok * H + i] << 16);
}

// fixed-order row reduction: each thread sums its own elements in index order,
// then a fixed xor tree inside the warp, then warps in ascending order
constexpr int NT_NORM = 256;
__global__ void __launch_bounds__(NT_NORM)
add_rmsnorm_kernel(float *__restrict__ h, const float *__restrict__ delta, const float *__restrict__ w, int H,
                   float eps, uint16_t *__restrict__ out, uint8_t *__restrict__ xpk) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.x;
    float4 *hr = reinterpret_cast<float4 *>(h + (size_t)r * H);
    const float4 *dr = delta ? reinterpret_cast<const float4 *>(delta + (size_t)r * H) : nullptr;
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    const int n4 = H / 4;
    // up to NKEEP float4 of the row (and of w) stay in registers between the two
    // passes, their loads all issued at once; a longer row reloads the rest
    constexpr int NKEEP = 4;
    float4 keep[NKEEP], wkeep[NKEEP];
#pragma unroll
    for (int k = 0; k < NKEEP; ++k) {
        const int i = threadIdx.x + k * NT_NORM;
        if (i < n4) {
            keep[k] = hr[i];
            wkeep[k] = w4[i];
        }
    }
    // each thread's elements in index order: the kept ones, then the rest
    auto add_sq = [&](float4 &v, int i, float &acc) {
        if (dr) {
            const float4 d = dr[i];
            v.x += d.x; v.y += d.y; v.z += d.z; v.w += d.w;
            hr[i] = v;
        }
        acc += v.x * v.x;
        acc += v.y * v.y;
        acc += v.z * v.z;
        acc += v.w * v.w;
    };
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NKEEP; ++k) {
        const int i = threadIdx.x + k * NT_NORM;
        if (i < n4) add_sq(keep[k], i, ss);
    }
    for (int i = threadIdx.x + NKEEP * NT_NORM; i < n4; i += NT_NORM) {
        float4 v = hr[i];
        add_sq(v, i, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float wsum[NT_NORM / 32];
    __shared__ float inv_s;
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < NT_NORM / 32; ++i) t += wsum[i];
        inv_s = rsqrtf(t / (float)H + eps);
    }
    __syncthreads();
    const float inv = inv_s;
    uint2 *o2 = reinterpret_cast<uint2 *>(out + (size_t)r * H);
    auto emit = [&](const float4 &v, const float4 &ww, int i) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x * inv * ww.x, v.y * inv * ww.y);
        __nv_bfloat162 b = __floats2bfloat162_rn(v.z * inv * ww.z, v.w * inv * ww.w);
        o2[i] = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
    };
#pragma unroll
    for (int k = 0; k < NKEEP; ++k) {
        const int i = threadIdx.x + k * NT_NORM;
        if (i < n4) emit(keep[k], wkeep[k], i);
    }
    for (int i = threadIdx.x + NKEEP * NT_NORM; i < n4; i += NT_NORM) emit(hr[i], w4[i], i);
    if (xpk) {
        // the row is column r of an 80-column K1 pass: write its packed blocks too
        __syncthreads();   // the row's bf16 values, stored above by every thread, are visible to the block
        for (int b = threadIdx.x; b < H / 32; b += NT_NORM) qmm::pack_wide_block(out + (size_t)r * H + 32 * b, 32 * b, r, xpk);
    }
}

__global__ void rope_table_kernel(float *tab, int max_pos, int D, double theta) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int half = D / 2;
    const long long n = (long long)max_pos * half;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(e / half), i = (int)(e % half);
        const double a = (double)p * pow(theta, -2.0 * i / D);
        tab[2 * e] = (float)cos(a);
        tab[2 * e + 1] = (float)sin(a);
    }
}

__global__ void rope_append_kernel(const float *__restrict__ qkv, int Hq, int Hkv, int D,
                                   const float *__restrict__ tab, int max_pos, const int32_t *__restrict__ cu_rows,
                                   const int32_t *__restrict__ ctx_start, int S, uint16_t *__restrict__ q_out,
                                   uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache, int num_pages,
                                   const int32_t *__restrict__ block_table, int max_blocks, uint16_t *__restrict__ k_stage,
                                   uint16_t *__restrict__ v_stage, int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.x;
    const int s = dev::warp_seq_of_row(cu_rows, S, r);
    const int pos = ctx_start[s] + (r - cu_rows[s]);
    const int half = D / 2;
    const float *row = qkv + (size_t)r * (Hq + 2 * Hkv) * D;
    bool pos_ok = pos >= 0 && pos < max_pos;
    int phys = -1;
    if (!k_stage) {
        if (pos_ok && pos / 16 < max_blocks) {
            phys = block_table[(size_t)s * max_blocks + pos / 16];
            if (phys < 0 || phys >= num_pages) {
                if (threadIdx.x == 0) dev::report(dev_err, SPEC_DEVERR_BLOCK_TABLE);
                phys = -1;
            }
        } else if (threadIdx.x == 0) {
            dev::report(dev_err, SPEC_DEVERR_LENGTH);
        }
    } else if (!pos_ok && threadIdx.x == 0) {
        dev::report(dev_err, SPEC_DEVERR_LENGTH);
    }
    const int slot = pos & 15;
    // rotated pairs: q heads then k heads
    for (int e = threadIdx.x; e < (Hq + Hkv) * half; e += blockDim.x) {
        const int hh = e / half, i = e % half;
        const float x1 = row[hh * D + i], x2 = row[hh * D + i + half];
        float c = 1.f, sn = 0.f;
        if (pos_ok) {
            const float2 cs = reinterpret_cast<const float2 *>(tab)[(size_t)pos * half + i];
            c = cs.x;
            sn = cs.y;
        }
        const float y1 = x1 * c - x2 * sn;
        const float y2 = x2 * c + x1 * sn;
        const uint16_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(y1));
        const uint16_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(y2));
        if (hh < Hq) {
            uint16_t *qo = q_out + ((size_t)r * Hq + hh) * D;
            qo[i] = b1;
            qo[i + half] = b2;
        } else {
            const int kh = hh - Hq;
            uint16_t *dst = nullptr;
            if (k_stage)
                dst = k_stage + ((size_t)r * Hkv + kh) * D;
            else if (phys >= 0)
                dst = k_cache + (((size_t)phys * Hkv + kh) * 16 + slot) * D;
            if (dst) {
                dst[i] = b1;
                dst[i + half] = b2;
            }
        }
    }
    // v: no rotation
    for (int e = threadIdx.x; e < Hkv * D; e += blockDim.x) {
        const int kh = e / D, d = e % D;
        const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(row[(Hq + Hkv) * D + e]));
        if (v_stage)
            v_stage[((size_t)r * Hkv + kh) * D + d] = b;
        else if (phys >= 0)
            v_cache[(((size_t)phys * Hkv + kh) * 16 + slot) * D + d] = b;
    }
}

__device__ __forceinline__ uint16_t swiglu1(float x, float u) { return dev::swiglu_bf16(x, u); }

// grid (ceil(F / 1024), R): each thread one group of four consecutive features
// (16-byte loads when F % 4 == 0 and the buffers are aligned, one element at a time otherwise)
__global__ void swiglu_kernel(const float *__restrict__ gu, int F, uint16_t *__restrict__ out, int vec,
                              uint8_t *__restrict__ xpk) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.y;
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    const float *g = gu + (size_t)r * 2 * F;
    uint16_t *o = out + (size_t)r * F;
    if (i >= F) {
        // nothing of this thread's own
    } else if (vec) {
        const float4 x = *reinterpret_cast<const float4 *>(g + i);
        const float4 u = *reinterpret_cast<const float4 *>(g + F + i);
        const uint2 v = make_uint2((uint32_t)swiglu1(x.x, u.x) | ((uint32_t)swiglu1(x.y, u.y) << 16),
                                   (uint32_t)swiglu1(x.z, u.z) | ((uint32_t)swiglu1(x.w, u.w) << 16));
        *reinterpret_cast<uint2 *>(o + i) = v;
    } else {
        for (int e = i; e < i + 4 && e < F; ++e) o[e] = swiglu1(g[e], g[F + e]);
    }
    if (xpk) {
        // the row is column r of an 80-column K1 pass: pack this CTA's 32-feature blocks too
        __syncthreads();   // the CTA's bf16 values, stored above, are visible to the block
        const int f0 = blockIdx.x * blockDim.x * 4;
        for (int b = threadIdx.x; b < (int)blockDim.x / 8; b += blockDim.x) {
            const int kb = f0 + 32 * b;
            if (kb < F) qmm::pack_wide_block(o + kb, kb, r, xpk);
        }
    }
}

__global__ void cast_bf16_kernel(const float *__restrict__ in, size_t n, uint16_t *__restrict__ out) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(in[i]));
}

// one warp per sequence: most recent earlier occurrence of the last n tokens
__global__ void ngram_draft_kernel(const int32_t *__restrict__ hist, int hist_cap, const int32_t *__restrict__ hist_len,
                                   int S, int W, const int32_t *__restrict__ pad, int32_t *__restrict__ drafts,
                                   int32_t *__restrict__ matched_n, int32_t *__restrict__ block_tokens) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= S) return;
    const int32_t *h = hist + (size_t)s * hist_cap;
    int len = hist_len[s];
    if (len > hist_cap) len = hist_cap;
    if (len < 0) len = 0;
    int found_j = -1, found_n = 0;
    for (int n = 3; n >= 1 && found_j < 0; --n) {
        if (len < n + 1) continue;
        // candidates j = len-n-1 down to 0, 32 at a time; lane 0 takes the largest j
        for (int top = len - n - 1; top >= 0 && found_j < 0; top -= 32) {
            const int j = top - lane;
            bool match = j >= 0;
            for (int t = 0; t < n && match; ++t) match = (h[j + t] == h[len - n + t]);
            const unsigned m = __ballot_sync(0xffffffffu, match);
            if (m) {
                found_j = top - (__ffs(m) - 1);
                found_n = n;
            }
        }
    }
    for (int c = lane; c < W; c += 32) {
        int v = pad[(size_t)s * W + c];
        if (found_j >= 0 && found_j + found_n + c < len) v = h[found_j + found_n + c];
        drafts[(size_t)s * W + c] = v;
        if (block_tokens) block_tokens[(size_t)s * (W + 1) + 1 + c] = v;
    }
    if (lane == 0) {
        if (matched_n) matched_n[s] = found_n;
        if (block_tokens) block_tokens[(size_t)s * (W + 1)] = len > 0 ? h[len - 1] : 0;
    }
}

// append the accepted drafts and the correction token to each history and
// move the sequence length forward: ctx = ctx_new
__global__ void commit_accepted_kernel(int32_t *__restrict__ hist, int hist_cap, int32_t *__restrict__ hist_len,
                                       const int32_t *__restrict__ drafts, int W, const int32_t *__restrict__ accepted,
                                       const int32_t *__restrict__ correction, const int32_t *__restrict__ ctx_new,
                                       int32_t *__restrict__ ctx, int S, int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= S) return;
    const int a = accepted[s];
    int len = hist_len[s];
    if (a < 0 || a > W || len < 0 || len + a + 1 > hist_cap) {
        dev::report(dev_err, SPEC_DEVERR_LENGTH);
        return;
    }
    int32_t *h = hist + (size_t)s * hist_cap;
    for (int i = 0; i < a; ++i) h[len + i] = drafts[(size_t)s * W + i];
    h[len + a] = correction[s];
    hist_len[s] = len + a + 1;
    ctx[s] = ctx_new[s];
}

}  // namespace

extern "C" spec_status spec_embed(const uint16_t *emb, int V, int H, const int32_t *tokens, int R, float *h,
                                  int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(V >= 1 && H >= 1 && R >= 0, "embed: bad sizes");
    SPEC_CHECK_ARG(emb && (tokens || R == 0) && (h || R == 0), "embed: NULL pointer");
    if (R == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(embed_kernel, dim3(R), dim3(256), 0, (cudaStream_t)stream, emb, V, H, tokens, h, dev_err);
    if (le != cudaSuccess) return spec::cuda_status(le, "embed launch");
    return spec::cuda_status(cudaGetLastError(), "embed launch");
}

extern "C" spec_status spec_add_rmsnorm(float *h, const float *delta, const float *w, int R, int H, float eps,
                                        uint16_t *out, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 0 && H >= 4 && H % 4 == 0, "add_rmsnorm: need H %% 4 == 0 (H=%d)", H);
    SPEC_CHECK_ARG((h && w && out) || R == 0, "add_rmsnorm: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(h) && spec::aligned16(delta) && spec::aligned16(w) && spec::aligned16(out),
                   "add_rmsnorm: pointers must be 16-byte aligned");
    if (R == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(add_rmsnorm_kernel, dim3(R), dim3(NT_NORM), 0, (cudaStream_t)stream, h, delta, w, H, eps, out,
                                      (uint8_t *)nullptr);
    if (le != cudaSuccess) return spec::cuda_status(le, "add_rmsnorm launch");
    return spec::cuda_status(cudaGetLastError(), "add_rmsnorm launch");
}

extern "C" spec_status spec_add_rmsnorm_packed(float *h, const float *delta, const float *w, int R, int H, float eps,
                                               uint16_t *out, void *xpk, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 0 && R <= qmm::WIDE_COLS && H >= 256 && H % 256 == 0,
                   "add_rmsnorm_packed: need R <= 80 and H a multiple of 256 (R=%d H=%d)", R, H);
    SPEC_CHECK_ARG((h && w && out && xpk) || R == 0, "add_rmsnorm_packed: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(h) && spec::aligned16(delta) && spec::aligned16(w) && spec::aligned16(out) &&
                       spec::aligned16(xpk),
                   "add_rmsnorm_packed: pointers must be 16-byte aligned");
    if (R == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(add_rmsnorm_kernel, dim3(R), dim3(NT_NORM), 0, (cudaStream_t)stream, h, delta, w, H, eps, out,
                                      reinterpret_cast<uint8_t *>(xpk));
    if (le != cudaSuccess) return spec::cuda_status(le, "add_rmsnorm_packed launch");
    return spec::cuda_status(cudaGetLastError(), "add_rmsnorm_packed launch");
}

extern "C" spec_status spec_rope_table(float *tab, int max_pos, int D, float theta, spec_stream_t stream) {
    SPEC_CHECK_ARG(tab && max_pos >= 1 && D >= 2 && D % 2 == 0 && theta > 0.f, "rope_table: bad arguments");
    const long long n = (long long)max_pos * (D / 2);
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    cudaError_t le = spec::launch_pdl(rope_table_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, tab, max_pos, D, (double)theta);
    if (le != cudaSuccess) return spec::cuda_status(le, "rope_table launch");
    return spec::cuda_status(cudaGetLastError(), "rope_table launch");
}

extern "C" spec_status spec_rope_append(const float *qkv, int R, int Hq, int Hkv, int D, const float *rope_tab,
                                        int max_pos, const int32_t *cu_rows, const int32_t *ctx_start, int S,
                                        uint16_t *q_out, uint16_t *k_cache, uint16_t *v_cache, int num_pages,
                                        const int32_t *block_table, int max_blocks, uint16_t *k_stage,
                                        uint16_t *v_stage, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 0 && S >= 0 && Hq >= 1 && Hkv >= 1 && D >= 2 && D % 2 == 0 && max_pos >= 1,
                   "rope_append: bad sizes");
    SPEC_CHECK_ARG((k_stage == nullptr) == (v_stage == nullptr), "rope_append: k_stage and v_stage both or neither");
    SPEC_CHECK_ARG(R == 0 || (qkv && rope_tab && cu_rows && ctx_start && q_out), "rope_append: NULL pointer");
    SPEC_CHECK_ARG(k_stage || R == 0 || (k_cache && v_cache && block_table && num_pages >= 1 && max_blocks >= 1),
                   "rope_append: cache arguments needed when not staging");
    if (R == 0 || S == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(rope_append_kernel, dim3(R), dim3(256), 0, (cudaStream_t)stream, qkv, Hq, Hkv, D,
                                      rope_tab, max_pos, cu_rows, ctx_start, S, q_out, k_cache, v_cache, num_pages,
                                      block_table, max_blocks, k_stage, v_stage, dev_err);
    if (le != cudaSuccess) return spec::cuda_status(le, "rope_append launch");
    return spec::cuda_status(cudaGetLastError(), "rope_append launch");
}

extern "C" spec_status spec_swiglu(const float *gu, int R, int F, uint16_t *out, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 0 && F >= 1, "swiglu: bad sizes");
    SPEC_CHECK_ARG((gu && out) || R == 0, "swiglu: NULL pointer");
    if (R == 0) return SPEC_OK;
    SPEC_CHECK_ARG(R <= 65535, "swiglu: at most 65535 rows per call");
    const int vec = (F % 4 == 0) && spec::aligned16(gu) && (reinterpret_cast<uintptr_t>(out) % 8 == 0);
    cudaError_t le = spec::launch_pdl(swiglu_kernel, dim3((F + 1023) / 1024, R), dim3(256), 0, (cudaStream_t)stream,
                                      gu, F, out, vec, (uint8_t *)nullptr);
    if (le != cudaSuccess) return spec::cuda_status(le, "swiglu launch");
    return spec::cuda_status(cudaGetLastError(), "swiglu launch");
}

extern "C" spec_status spec_swiglu_packed(const float *gu, int R, int F, uint16_t *out, void *xpk, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 0 && R <= qmm::WIDE_COLS && F >= 256 && F % 256 == 0,
                   "swiglu_packed: need R <= 80 and F a multiple of 256 (R=%d F=%d)", R, F);
    SPEC_CHECK_ARG((gu && out && xpk) || R == 0, "swiglu_packed: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(gu) && spec::aligned16(out) && spec::aligned16(xpk),
                   "swiglu_packed: pointers must be 16-byte aligned");
    if (R == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(swiglu_kernel, dim3((F + 1023) / 1024, R), dim3(256), 0, (cudaStream_t)stream,
                                      gu, F, out, 1, reinterpret_cast<uint8_t *>(xpk));
    if (le != cudaSuccess) return spec::cuda_status(le, "swiglu_packed launch");
    return spec::cuda_status(cudaGetLastError(), "swiglu_packed launch");
}

extern "C" spec_status spec_cast_bf16(const float *in, size_t n, uint16_t *out, spec_stream_t stream) {
    SPEC_CHECK_ARG((in && out) || n == 0, "cast_bf16: NULL pointer");
    if (n == 0) return SPEC_OK;
    size_t blocks = (n + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    cudaError_t le = spec::launch_pdl(cast_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream, in, n, out);
    if (le != cudaSuccess) return spec::cuda_status(le, "cast_bf16 launch");
    return spec::cuda_status(cudaGetLastError(), "cast_bf16 launch");
}

extern "C" spec_status spec_ngram_draft(const int32_t *hist, int hist_cap, const int32_t *hist_len, int S, int W,
                                        const int32_t *pad, int32_t *drafts, int32_t *matched_n,
                                        int32_t *block_tokens, spec_stream_t stream) {
    SPEC_CHECK_ARG(S >= 0 && W >= 0 && hist_cap >= 1, "ngram_draft: bad sizes");
    SPEC_CHECK_ARG(S == 0 || (hist && hist_len && (W == 0 || (pad && drafts))), "ngram_draft: NULL pointer");
    if (S == 0 || (W == 0 && !block_tokens && !matched_n)) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(ngram_draft_kernel, dim3((S + 3) / 4), dim3(128), 0, (cudaStream_t)stream, hist,
                                      hist_cap, hist_len, S, W, pad, drafts, matched_n, block_tokens);
    if (le != cudaSuccess) return spec::cuda_status(le, "ngram_draft launch");
    return spec::cuda_status(cudaGetLastError(), "ngram_draft launch");
}

extern "C" spec_status spec_commit_accepted(int32_t *hist, int hist_cap, int32_t *hist_len, const int32_t *drafts,
                                            int W, const int32_t *accepted, const int32_t *correction,
                                            const int32_t *ctx_new, int32_t *ctx, int S, int32_t *dev_err,
                                            spec_stream_t stream) {
    SPEC_CHECK_ARG(S >= 0 && W >= 0 && hist_cap >= 1, "commit_accepted: bad sizes");
    SPEC_CHECK_ARG(S == 0 || (hist && hist_len && accepted && correction && ctx_new && ctx && (W == 0 || drafts)),
                   "commit_accepted: NULL pointer");
    if (S == 0) return SPEC_OK;
    cudaError_t le = spec::launch_pdl(commit_accepted_kernel, dim3((S + 127) / 128), dim3(128), 0, (cudaStream_t)stream,
                                      hist, hist_cap, hist_len, drafts, W, accepted, correction, ctx_new, ctx, S,
                                      dev_err);
    if (le != cudaSuccess) return spec::cuda_status(le, "commit_accepted launch");
    return spec::cuda_status(cudaGetLastError(), "commit_accepted launch");
}
