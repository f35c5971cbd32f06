// K1: batch-invariant int4 block-32 dequantising matmul (sm_103a).
//
//   y[j][n] = sum_k x[j][k] * d[n][k/32] * (nib(n, k) - 8)
//
// Why it is width-invariant.  Output element (n, j) is computed as follows and
// nothing in the sequence depends on how many columns the call has or where
// column j sits:
//  * K is cut into `ksplit(K)` segments of whole 256-k stages (a function of
//    K alone).  Segment s is reduced by CTA rank s of a thread-block cluster.
//  * Inside a segment, for every 32-k block b in ascending order, one warp
//    computes the block partial P_b = sum_{k in b} q x with two chained
//    m16n8k16 bf16 MMAs (C starts at +0), then acc = fma(d_b, P_b, acc).
//    The MMA instruction stream is identical for every call; column j's value
//    depends only on A (the weights), on B column j and on C column j.
//    Unused columns are zero, never a different instruction.
//  * The cluster's segment partials are summed in ascending rank order.
// Which CTA, warp or column tile handles column j is a scheduling choice and
// may depend on n_cols; the arithmetic applied to column j never does.
//
// Data movement: TMA (cp.async.bulk.tensor) streams, per 256-k stage, a
// 64-row x 128-byte weight tile (128B swizzle), the 64 x 8 fp16 scales and
// the 4 x 64-k activation tiles of the CTA's column group into a ring of
// shared-memory stages guarded by mbarriers; a producer warp issues the
// copies, four consumer warps (16 rows each) read weights with ldmatrix,
// dequantise nibbles to bf16 in registers and feed mma.sync.
//
// The weight format (int4 block 32, fp16 scale, even k in the low nibble) is
// the stand-in for the block-quantised formats named in ramgpt.org, "When
// Lossless Speculation Stops Being Lossless on Blackwell", section
// "Quantized Matrix Multiplication Shows the Same Class of Failure".
#include "common.cuh"

namespace {

constexpr int BM = 64;                        // weight rows per CTA
constexpr int KST = 256;                      // k per pipeline stage
constexpr int W_BYTES = BM * KST / 2;         // 8192: int4 codes of one stage
constexpr int S_BYTES = BM * (KST / 32) * 2;  // 1024: fp16 scales of one stage
constexpr int NCONS = 4;                      // consumer warps
constexpr int THREADS = (NCONS + 1) * 32;     // + one producer warp
constexpr int SMEM_BUDGET = 100 * 1024;       // two CTAs per SM

template <int NT>
struct Cfg {
    static constexpr int X_BOX = 8 * NT * 128;          // one 64-k activation box
    static constexpr int X_BYTES = 4 * X_BOX;           // 4 boxes per stage
    static constexpr int STAGE = W_BYTES + X_BYTES + S_BYTES;
    static constexpr int NST = (SMEM_BUDGET / STAGE) < 2 ? 2 : (SMEM_BUDGET / STAGE);
    static constexpr int SMEM = 1024 + NST * STAGE + 2 * NST * 8;
    static_assert(W_BYTES % 1024 == 0 && X_BOX % 1024 == 0 && STAGE % 1024 == 0, "1024-byte swizzle alignment");
    static_assert(8 * NT * BM * 4 <= STAGE * NST, "partial tile fits in the stage ring");
};

// K-split as a function of K alone: segments of >= 4 stages, at most 8.
__host__ __device__ inline int ksplit_of(int K) {
    int nst = K / KST;
    int s = nst / 4;
    return s < 1 ? 1 : (s > 8 ? 8 : s);
}

// nibble codes of one 32-bit word (8 codes, k = 8t .. 8t+7 of a block) to
// four bf16x2 registers holding (q_m, q_{m+4}) for m = 0..3
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t MASK = 0x000F000Fu, MAGIC = 0x43004300u;  // bf16 128.0 in each half
    const __nv_bfloat162 OFF = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t v = dev::lop3_and_or(w >> (4 * m), MASK, MAGIC);  // (128 + code) per half, exact
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
        h = __hsub2(h, OFF);                                         // code - 8 = q, exact
        o[m] = *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int NT, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 2)
qmm_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ts,
           const __grid_constant__ CUtensorMap tx, int N, int K, int n_cols, void *__restrict__ y, int ldy,
           int accumulate, int ksplit, int32_t *dev_err) {
    using C = Cfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE);
    uint64_t *empty = full + C::NST;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * BM;
    const int seg = blockIdx.y;
    const int col0 = blockIdx.z * 8 * NT;
    const int nst_total = K / KST;
    const int st_begin = seg * nst_total / ksplit;
    const int nst = (seg + 1) * nst_total / ksplit - st_begin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NST; ++s) {
            dev::mbar_init(&full[s], 1);
            dev::mbar_init(&empty[s], NCONS);
        }
        dev::fence_barrier_init();
    }
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int c = 0; c < NT; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;

    if (warp == NCONS) {
        // ---------------- producer ----------------
        if (lane == 0) {
            dev::prefetch_tmap(&tw);
            dev::prefetch_tmap(&tx);
            dev::prefetch_tmap(&ts);
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % C::NST;
                if (i >= C::NST && !dev::mbar_wait(&empty[s], ((i / C::NST) - 1) & 1)) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    break;
                }
                uint8_t *base = smem + s * C::STAGE;
                const int k0 = (st_begin + i) * KST;
                dev::mbar_arrive_expect_tx(&full[s], C::STAGE);
                dev::tma_load_2d(base, &tw, k0 / 2, row0, &full[s]);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    dev::tma_load_2d(base + W_BYTES + b * C::X_BOX, &tx, k0 + 64 * b, col0, &full[s]);
                dev::tma_load_2d(base + W_BYTES + C::X_BYTES, &ts, k0 / 32, row0, &full[s]);
                issued = i + 1;
            }
            // never leave copies in flight: wait (bounded) for every issued stage
            for (int i = (issued > C::NST ? issued - C::NST : 0); i < issued; ++i)
                if (!dev::mbar_wait(&full[i % C::NST], (i / C::NST) & 1)) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
        }
    } else {
        // ---------------- consumers ----------------
        const int r = lane >> 2, t = lane & 3;
        const int wrow = warp * 16;
        // B-fragment column of this lane: MMA column slot g = lane/4 carries
        // activation column pi(g) = (g & 1) * 4 + g / 2 (bank-conflict-free rows)
        const int g = lane >> 2;
        const int xcol = (g & 1) * 4 + (g >> 1);
        for (int i = 0; i < nst; ++i) {
            const int s = i % C::NST;
            if (!dev::mbar_wait(&full[s], (i / C::NST) & 1)) {
                dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                break;
            }
            uint8_t *base = smem + s * C::STAGE;
            const uint32_t wbase = dev::smem_u32(base);
            const uint32_t xbase = wbase + W_BYTES;
            const uint32_t sbase = xbase + C::X_BYTES;
            uint32_t sr[4], sr8[4];
            dev::lds128(sr[0], sr[1], sr[2], sr[3], sbase + (wrow + r) * 16);
            dev::lds128(sr8[0], sr8[1], sr8[2], sr8[3], sbase + (wrow + r + 8) * 16);
#pragma unroll
            for (int bp = 0; bp < 4; ++bp) {
                uint32_t wv[4];
                {
                    const int m = lane >> 3, rr = lane & 7;
                    const int row = wrow + (m & 1) * 8 + rr;
                    const int blk = 2 * bp + (m >> 1);
                    dev::ldmatrix_x4(wv[0], wv[1], wv[2], wv[3], wbase + row * 128 + ((blk ^ (row & 7)) << 4));
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int blk = 2 * bp + h;
                    uint32_t ar[4], ar8[4];
                    dequant_word(wv[2 * h], ar);       // row r
                    dequant_word(wv[2 * h + 1], ar8);  // row r + 8
                    const uint32_t s2 = sr[blk >> 1], s28 = sr8[blk >> 1];
                    const float d_r = __half2float(__ushort_as_half((unsigned short)((blk & 1) ? (s2 >> 16) : (s2 & 0xFFFF))));
                    const float d_r8 = __half2float(__ushort_as_half((unsigned short)((blk & 1) ? (s28 >> 16) : (s28 & 0xFFFF))));
#pragma unroll
                    for (int ct = 0; ct < NT; ++ct) {
                        const int xrow = ct * 8 + xcol;
                        const int chunk = ((blk & 1) * 4 + t) ^ (xrow & 7);
                        uint32_t e01, e23, e45, e67;
                        dev::lds128(e01, e23, e45, e67, xbase + (blk >> 1) * C::X_BOX + xrow * 128 + (chunk << 4));
                        const uint32_t b00 = dev::prmt(e01, e45, 0x5410), b01 = dev::prmt(e01, e45, 0x7632);
                        const uint32_t b10 = dev::prmt(e23, e67, 0x5410), b11 = dev::prmt(e23, e67, 0x7632);
                        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
                        float p[4];
                        dev::mma_bf16(p, ar[0], ar8[0], ar[1], ar8[1], b00, b01, zero);
                        dev::mma_bf16(p, ar[2], ar8[2], ar[3], ar8[3], b10, b11, p);
                        acc[ct][0] = fmaf(d_r, p[0], acc[ct][0]);
                        acc[ct][1] = fmaf(d_r, p[1], acc[ct][1]);
                        acc[ct][2] = fmaf(d_r8, p[2], acc[ct][2]);
                        acc[ct][3] = fmaf(d_r8, p[3], acc[ct][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&empty[s]);
        }
    }

    // ---------------- segment partial -> shared tile [8NT cols][64 rows] ----------------
    __syncthreads();
    float *part = reinterpret_cast<float *>(smem);
    if (warp < NCONS) {
        const int r = lane >> 2, t = lane & 3;
        const int wrow = warp * 16;
#pragma unroll
        for (int ct = 0; ct < NT; ++ct) {
            // C slot 2t <-> column t, slot 2t+1 <-> column t + 4 (see xcol)
            part[(ct * 8 + t) * BM + wrow + r] = acc[ct][0];
            part[(ct * 8 + t + 4) * BM + wrow + r] = acc[ct][1];
            part[(ct * 8 + t) * BM + wrow + r + 8] = acc[ct][2];
            part[(ct * 8 + t + 4) * BM + wrow + r + 8] = acc[ct][3];
        }
    }
    if (ksplit > 1)
        dev::cluster_sync();
    else
        __syncthreads();

    // ---------------- fixed-order combine of the segments and store ----------------
    const int rank = (ksplit > 1) ? (int)dev::cluster_ctarank() : 0;
    const int elems = 8 * NT * BM;
    for (int e = rank * THREADS + threadIdx.x; e < elems; e += ksplit * THREADS) {
        float v;
        if (ksplit > 1) {
            const uint32_t local = dev::smem_u32(part + e);
            v = dev::ld_shared_cluster_f32(dev::map_shared_rank(local, 0));
            for (int q = 1; q < ksplit; ++q) v += dev::ld_shared_cluster_f32(dev::map_shared_rank(local, q));
        } else {
            v = part[e];
        }
        const int col = col0 + e / BM, row = row0 + e % BM;
        if (col < n_cols && row < N) {
            if (OUT_BF16) {
                reinterpret_cast<__nv_bfloat16 *>(y)[(size_t)col * ldy + row] = __float2bfloat16_rn(v);
            } else {
                float *yp = reinterpret_cast<float *>(y) + (size_t)col * ldy + row;
                *yp = accumulate ? (*yp + v) : v;
            }
        }
    }
    if (ksplit > 1) dev::cluster_sync();  // keep shared memory alive until every rank has read it
}

template <int NT, bool OUT_BF16>
spec_status launch_nt(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int N, int K, int n_cols,
                      int ldx, void *y, int ldy, int accumulate, int ksplit, int32_t *dev_err, cudaStream_t stream) {
    using C = Cfg<NT>;
    CUtensorMap tx;
    {
        uint64_t dims[2] = {(uint64_t)K, (uint64_t)n_cols};
        uint64_t strides[1] = {(uint64_t)ldx * 2};
        uint32_t box[2] = {64, (uint32_t)(8 * NT)};
        if (!spec::encode_tiled(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return SPEC_ERR_CUDA;
    }
    auto kern = qmm_kernel<NT, OUT_BF16>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return spec::cuda_status(e, "cudaFuncSetAttribute(qmm smem)");
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + BM - 1) / BM, ksplit, (n_cols + 8 * NT - 1) / (8 * NT));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ksplit;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, ts, tx, N, K, n_cols, y, ldy, accumulate, ksplit, dev_err);
    return spec::cuda_status(e, "qmm launch");
}

spec_status qmm_run(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x, int n_cols, int ldx,
                    void *y, spec_dtype y_dt, int ldy, int accumulate, int ksplit, int nt_force, int32_t *dev_err,
                    cudaStream_t stream) {
    CUtensorMap tw, ts;
    {
        uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)K / 2};
        uint32_t box[2] = {128, BM};
        if (!spec::encode_tiled(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return SPEC_ERR_CUDA;
    }
    {
        uint64_t dims[2] = {(uint64_t)K / 32, (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)K / 32 * 2};
        uint32_t box[2] = {8, BM};
        if (!spec::encode_tiled(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, ws, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return SPEC_ERR_CUDA;
    }
    int nt = nt_force ? nt_force : (n_cols <= 8 ? 1 : (n_cols <= 16 ? 2 : 4));
    const bool bf = (y_dt == SPEC_BF16);
    switch (nt) {
    case 1: return bf ? launch_nt<1, true>(tw, ts, x, N, K, n_cols, ldx, y, ldy, 0, ksplit, dev_err, stream)
                      : launch_nt<1, false>(tw, ts, x, N, K, n_cols, ldx, y, ldy, accumulate, ksplit, dev_err, stream);
    case 2: return bf ? launch_nt<2, true>(tw, ts, x, N, K, n_cols, ldx, y, ldy, 0, ksplit, dev_err, stream)
                      : launch_nt<2, false>(tw, ts, x, N, K, n_cols, ldx, y, ldy, accumulate, ksplit, dev_err, stream);
    default: return bf ? launch_nt<4, true>(tw, ts, x, N, K, n_cols, ldx, y, ldy, 0, ksplit, dev_err, stream)
                       : launch_nt<4, false>(tw, ts, x, N, K, n_cols, ldx, y, ldy, accumulate, ksplit, dev_err, stream);
    }
}

spec_status check_args(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x, int n_cols, int ldx,
                       const void *y, int ldy) {
    SPEC_CHECK_ARG(N >= 1 && K >= 256 && n_cols >= 0, "qmatmul: need N >= 1, K >= 256, n_cols >= 0 (N=%d K=%d n_cols=%d)",
                   N, K, n_cols);
    SPEC_CHECK_ARG(K % 256 == 0, "qmatmul: K must be a multiple of 256 (K=%d)", K);
    SPEC_CHECK_ARG(ldx >= K && ldx % 8 == 0, "qmatmul: ldx must be >= K and a multiple of 8 (ldx=%d)", ldx);
    SPEC_CHECK_ARG(ldy >= N, "qmatmul: ldy must be >= N (ldy=%d)", ldy);
    SPEC_CHECK_ARG(wq && ws && y && (x || n_cols == 0), "qmatmul: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(wq) && spec::aligned16(ws) && spec::aligned16(x),
                   "qmatmul: wq, ws and x must be 16-byte aligned");
    SPEC_CHECK_ARG((long long)N * (K / 2) < (1ll << 40), "qmatmul: matrix too large");
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_qmatmul(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                    int n_cols, int ldx, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                    int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, ksplit_of(K), 0, dev_err,
                   (cudaStream_t)stream);
}

extern "C" spec_status spec_qmatmul_noninvariant(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                                 const uint16_t *x, int n_cols, int ldx, float *y, int ldy,
                                                 spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    if (n_cols == 0) return SPEC_OK;
    // split of K chosen per call: enough CTAs for two per SM, whatever K is
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    const int nt = n_cols <= 8 ? 1 : (n_cols <= 16 ? 2 : 4);
    const long long tiles = (long long)((N + BM - 1) / BM) * ((n_cols + 8 * nt - 1) / (8 * nt));
    int ks = (int)((2ll * sms + tiles - 1) / tiles);
    const int nst = K / KST;
    if (ks > 8) ks = 8;
    if (ks > nst) ks = nst;
    if (ks < 1) ks = 1;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, ks, nt, nullptr, (cudaStream_t)stream);
}

// Test hook: run the invariant kernel with an explicit column-tile width so the
// tests can show the per-column result does not depend on it.
extern "C" spec_status spec_qmatmul_debug_nt(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                             int n_cols, int ldx, float *y, int ldy, int nt, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(nt == 1 || nt == 2 || nt == 4, "nt must be 1, 2 or 4");
    if (n_cols == 0) return SPEC_OK;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, ksplit_of(K), nt, nullptr,
                   (cudaStream_t)stream);
}
