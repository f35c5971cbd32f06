// Margin-gated re-check of the LM head (sm_103a).
//
// tokenstrom.com, "'Lossless,' but not quite", sections "Why the math checks
// out and the text still flips" (only steps whose top-2 margin is small can
// flip) and "What the big servers offer and what it costs" (re-check only the
// uncertain steps).  A verify block's logits come from a fast, non-invariant
// evaluation of the LM head; every entry of it lies within err_r of the
// invariant evaluation's (err_r = coef * ||x_r||_1, the summation-order bound
// the caller derives for its matrix).  A row whose top-2 margin exceeds 2 err_r
// has the same argmax in both; every other row is listed for an invariant
// re-evaluation, so the argmax of every row equals the invariant argmax.
//
//  * gate_partial_kernel: (split, row) CTAs scan the fp32 logits with exact
//    comparisons for the top value (lowest index on ties) and the largest
//    value at any other index; split 0 also forms ||x_r||_1.
//  * gate_finalize_kernel: one CTA folds the splits in order, flags rows with
//    margin <= 2 err_r, numbers them in row order (a block-wide scan, so the
//    list is deterministic), gathers their activations into a compact buffer
//    (at most `capacity` rows) and writes the count, plus R in an overflow
//    word when more rows were flagged than the buffer holds (the caller then
//    re-evaluates every row).
//  * gate_scatter_kernel: copies each re-evaluated row into its logits row.
#include "common.cuh"

namespace {

constexpr int GT = 256;          // threads of the scan kernels

struct Top2 {
    float v1;    // the largest value
    int i1;      // its lowest index
    float v2;    // the largest value at any other index
};

__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

__device__ __forceinline__ Top2 merge(const Top2 &a, const Top2 &b) {
    Top2 r;
    if (beats(b.v1, b.i1, a.v1, a.i1)) {
        r.v1 = b.v1, r.i1 = b.i1;
        r.v2 = fmaxf(a.v1, fmaxf(a.v2, b.v2));
    } else {
        r.v1 = a.v1, r.i1 = a.i1;
        r.v2 = fmaxf(b.v1, fmaxf(a.v2, b.v2));
    }
    return r;
}

__device__ __forceinline__ void push(Top2 &t, float x, int idx) {
    if (beats(x, idx, t.v1, t.i1)) {
        t.v2 = fmaxf(t.v2, t.v1);
        t.v1 = x, t.i1 = idx;
    } else {
        t.v2 = fmaxf(t.v2, x);
    }
}

__global__ void __launch_bounds__(GT)
gate_partial_kernel(const float *__restrict__ logits, int V, int split, int R, const uint16_t *__restrict__ x, int H,
                    int ldx, Top2 *__restrict__ part, float *__restrict__ xnorm, int32_t *dev_err) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int r = blockIdx.y, sp = blockIdx.x;
    if (r >= R) return;
    const int nvec = V / 4;
    const int v0 = (int)((long long)nvec * sp / split), v1 = (int)((long long)nvec * (sp + 1) / split);
    const float4 *row = reinterpret_cast<const float4 *>(logits + (size_t)r * V);
    Top2 t{-INFINITY, INT_MAX, -INFINITY};
    bool nan = false;
    for (int v = v0 + threadIdx.x; v < v1; v += GT) {
        const float4 w = __ldcs(row + v);
        const float e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (e[q] != e[q]) {
                nan = true;
                continue;
            }
            push(t, e[q], 4 * v + q);
        }
    }
    if (nan) dev::report(dev_err, SPEC_DEVERR_NAN);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Top2 u{__shfl_xor_sync(0xffffffffu, t.v1, o), __shfl_xor_sync(0xffffffffu, t.i1, o),
               __shfl_xor_sync(0xffffffffu, t.v2, o)};
        t = merge(t, u);
    }
    __shared__ Top2 wt[GT / 32];
    __shared__ float wn[GT / 32];
    float ns = 0.f;
    if (sp == 0) {
        // ||x_r||_1, each thread over its k in order, then a fixed tree
        const uint16_t *xr = x + (size_t)r * ldx;
        for (int k = threadIdx.x; k < H; k += GT) ns += fabsf(__uint_as_float((uint32_t)xr[k] << 16));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ns += __shfl_xor_sync(0xffffffffu, ns, o);
    }
    if ((threadIdx.x & 31) == 0) {
        wt[threadIdx.x >> 5] = t;
        wn[threadIdx.x >> 5] = ns;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Top2 a = wt[0];
        float n = wn[0];
        for (int w = 1; w < GT / 32; ++w) a = merge(a, wt[w]), n += wn[w];
        part[(size_t)r * split + sp] = a;
        // an upper bound on ||x_r||_1 despite the fp32 sum's rounding
        if (sp == 0) xnorm[r] = n * (1.0f + 1e-3f);
    }
}

__global__ void __launch_bounds__(GT)
gate_finalize_kernel(const Top2 *__restrict__ part, int split, int R, const float *__restrict__ xnorm, float coef,
                     const uint16_t *__restrict__ x, int H, int ldx, int32_t *__restrict__ top,
                     int32_t *__restrict__ rows, int32_t *__restrict__ count, int32_t *__restrict__ overflow,
                     int capacity, uint16_t *__restrict__ xg) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    __shared__ int scan[GT];
    __shared__ int base;
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    for (int r0 = 0; r0 < R; r0 += GT) {
        const int r = r0 + threadIdx.x;
        int flag = 0;
        if (r < R) {
            Top2 a = part[(size_t)r * split];
            for (int q = 1; q < split; ++q) a = merge(a, part[(size_t)r * split + q]);
            const float err = coef * xnorm[r];
            // margin = v1 - v2 (v2 = -inf for a one-entry row: never re-checked)
            flag = !(a.v1 - a.v2 > 2.0f * err);
            top[r] = a.i1 == INT_MAX ? 0 : a.i1;
        }
        scan[threadIdx.x] = flag;
        __syncthreads();
        for (int o = 1; o < GT; o <<= 1) {   // inclusive scan in row order
            const int v = threadIdx.x >= o ? scan[threadIdx.x - o] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            __syncthreads();
        }
        const int slot = base + scan[threadIdx.x] - flag;
        if (flag && slot < capacity) rows[slot] = r;
        __syncthreads();
        if (threadIdx.x == GT - 1) base += scan[GT - 1];
        __syncthreads();
    }
    const int n = base;
    if (threadIdx.x == 0) {
        *count = n;
        *overflow = n > capacity ? R : 0;
    }
    // gather the listed rows' activations (16-byte vectors; H % 8 == 0, ldx % 8 == 0)
    const int m = n < capacity ? n : capacity;
    const int hv = H / 8;
    for (int e = threadIdx.x; e < m * hv; e += GT) {
        const int s = e / hv, c = e % hv;
        const int r = rows[s];
        reinterpret_cast<uint4 *>(xg + (size_t)s * H)[c] = reinterpret_cast<const uint4 *>(x + (size_t)r * ldx)[c];
    }
}

__global__ void __launch_bounds__(GT)
gate_scatter_kernel(const float *__restrict__ yg, int V, const int32_t *__restrict__ rows,
                    const int32_t *__restrict__ count, int capacity, float *__restrict__ logits) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    const int s = blockIdx.x;
    const int n = *count;
    if (s >= n || s >= capacity) return;
    const float4 *src = reinterpret_cast<const float4 *>(yg + (size_t)s * V);
    float4 *dst = reinterpret_cast<float4 *>(logits + (size_t)rows[s] * V);
    for (int v = threadIdx.x; v < V / 4; v += GT) dst[v] = src[v];
}

int gate_split(int R, int V) {
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    int sp = (8 * sms + R - 1) / R;
    const int max_sp = V / 2048 > 0 ? V / 2048 : 1;
    if (sp > max_sp) sp = max_sp;
    return sp < 1 ? 1 : sp;
}

}  // namespace

extern "C" size_t spec_margin_gate_workspace(int R, int V) {
    if (R <= 0 || V <= 0) return 0;
    return (size_t)R * gate_split(R, V) * sizeof(Top2) + (size_t)R * sizeof(float);
}

extern "C" spec_status spec_margin_gate(const float *logits, int V, int R, const uint16_t *x, int H, int ldx,
                                        float err_coef, int32_t *top, int32_t *rows, int32_t *count,
                                        int32_t *overflow, int capacity, uint16_t *x_gathered, void *workspace,
                                        size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(R >= 1 && V >= 4 && V % 4 == 0, "margin_gate: need R >= 1 and V a positive multiple of 4 (R=%d V=%d)",
                   R, V);
    SPEC_CHECK_ARG(H >= 8 && H % 8 == 0 && ldx >= H && ldx % 8 == 0,
                   "margin_gate: H and ldx must be multiples of 8 with ldx >= H (H=%d ldx=%d)", H, ldx);
    SPEC_CHECK_ARG(capacity >= 1, "margin_gate: capacity must be >= 1");
    SPEC_CHECK_ARG(err_coef >= 0.f && err_coef == err_coef, "margin_gate: err_coef must be a finite value >= 0");
    SPEC_CHECK_ARG(logits && x && top && rows && count && overflow && x_gathered, "margin_gate: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(logits) && spec::aligned16(x) && spec::aligned16(x_gathered),
                   "margin_gate: logits, x and x_gathered must be 16-byte aligned");
    const int split = gate_split(R, V);
    const size_t need = spec_margin_gate_workspace(R, V);
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "margin_gate: workspace needs %zu bytes (16-byte aligned), got %zu", need,
                          ws_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    Top2 *part = reinterpret_cast<Top2 *>(workspace);
    float *xnorm = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + (size_t)R * split * sizeof(Top2));
    cudaError_t e = spec::launch_pdl(gate_partial_kernel, dim3(split, R), dim3(GT), 0, st, logits, V, split, R, x, H,
                                     ldx, part, xnorm, dev_err);
    if (e != cudaSuccess) return spec::cuda_status(e, "margin_gate scan launch");
    e = spec::launch_pdl(gate_finalize_kernel, dim3(1), dim3(GT), 0, st, (const Top2 *)part, split, R,
                         (const float *)xnorm, err_coef, x, H, ldx, top, rows, count, overflow, capacity, x_gathered);
    return spec::cuda_status(e, "margin_gate finalize launch");
}

extern "C" spec_status spec_gate_scatter(const float *y_gathered, int V, const int32_t *rows, const int32_t *count,
                                         int capacity, float *logits, spec_stream_t stream) {
    SPEC_CHECK_ARG(V >= 4 && V % 4 == 0 && capacity >= 1, "gate_scatter: V must be a multiple of 4, capacity >= 1");
    SPEC_CHECK_ARG(y_gathered && rows && count && logits, "gate_scatter: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(y_gathered) && spec::aligned16(logits), "gate_scatter: buffers must be 16-byte aligned");
    cudaError_t e = spec::launch_pdl(gate_scatter_kernel, dim3(capacity), dim3(GT), 0, (cudaStream_t)stream,
                                     y_gathered, V, rows, count, capacity, logits);
    return spec::cuda_status(e, "gate_scatter launch");
}
