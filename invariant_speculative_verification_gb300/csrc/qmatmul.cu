// K1: batch-invariant int4 block-32 dequantising matmul on the 5th-generation
// tensor cores (sm_103a: tcgen05.mma, tensor memory, TMA).
//
//   y[j][n] = sum_k x[j][k] * d[n][k/32] * (nib(n, k) - 8)
//
// Per-element arithmetic (identical for every call, whatever n_cols is and
// wherever column j sits):
//  * K is cut into segments of 512 (when K / 256 is odd the last segment is
//    256 long).  The cut depends on K only.
//  * Inside a segment, for every 32-k block b in ascending order, the block
//    partial P_b is one chain of two K=16 tensor-core MMAs (fp32 accumulator,
//    the first starting from zero) of A = q = code - 8 (bf16, exact) and B =
//    column j of x (bf16); then s = fma(d_b, P_b, s) with s starting at +0.
//  * The segment sums are folded in ascending order: y = ((s_0 + s_1) + s_2)...
// Column j's P_b depends only on A and on B column j: the MMA's N (the number
// of columns a pass carries, 16 or 80) does not change it, and unused columns
// are zero.  Which CTA handles a column, and where a CTA's share of the work
// starts and ends, is scheduling that may depend on the call; the arithmetic
// above never does.
//
// Execution: a persistent grid of one CTA per SM over (128-row tile x
// K-segment) units dealt out in equal contiguous ranges (stream-K).  Per CTA:
//  * a TMA warp streams each 256-k stage into a ring of shared-memory slots:
//    the int4 codes (128 rows x 128 bytes, 128-byte swizzle), the fp16 scales
//    and the pass's activation columns (four 64-k x NP-row boxes, 128-byte
//    swizzle: the MMA's B operand as it lands; columns past n_cols arrive as
//    zeros);
//  * eight dequantising warps (two per TMEM lane quarter, alternate blocks)
//    turn each block's codes into bf16 q and store them into one of eight
//    TMEM A buffers (lane = weight row);
//  * one thread issues the two MMAs of each block into one of several TMEM
//    accumulator buffers and commits them to mbarriers;
//  * eight epilogue warps (thread = weight row, half of the columns each) load
//    each block's accumulator from TMEM and apply the scale FMA in registers,
//    keep the tile's segment fold in TMEM and write y.
// A tile covered by one CTA is written directly.  A tile shared by several
// CTAs: the CTAs holding its later segments store their segment sums and count
// themselves in, without waiting; the CTA holding the leading segments folds
// them in segment order once all have arrived (the usual case when it gets
// there), else leaves its prefix for whichever CTA arrives last.  No CTA waits
// for another; the counters end at zero.
//
// The weight format (int4 block 32, fp16 scale, even k in the low nibble) is
// the stand-in for the block-quantised formats named in ramgpt.org, "When
// Lossless Speculation Stops Being Lossless on Blackwell", section
// "Quantized Matrix Multiplication Shows the Same Class of Failure".
#include <mutex>

#include "common.cuh"

namespace {

constexpr int SEG_K = 512;                   // k per K-segment (the invariant reduction unit)
constexpr int KS = 256;                      // k per stage
constexpr int NBLK = KS / 32;                // 32-k blocks per stage
constexpr int BM = 128;                      // weight rows per tile (= TMEM lanes)
constexpr int NEW = 8;                       // epilogue warps 0..7
constexpr int NQW = 8;                       // dequantising warps 8..15
constexpr int W_TMA = NEW + NQW;             // warp 16
constexpr int W_MMA = W_TMA + 1;             // warp 17 (also owns the TMEM allocation)
constexpr int THREADS = (W_MMA + 1) * 32;
constexpr int W_BYTES = BM * 128;            // one stage of codes
constexpr int S_BYTES = BM * NBLK * 2;       // one stage of scales
constexpr int SMEM_BUDGET = 226 * 1024;
constexpr int MAX_NP = 80;                   // columns per pass, at most
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t YCOL = 288;               // TMEM columns of the running segment fold
constexpr uint32_t ACOL = 384;               // TMEM columns of the eight A buffers (16 each)

template <int NP>
struct Cfg {
    static_assert(NP % 16 == 0 && NP >= 16 && NP <= MAX_NP, "columns per pass");
    static constexpr int NH = NP / 2;                          // columns per epilogue thread
    static constexpr int X_BOX = NP * 128;                     // 64 k of the pass's columns
    static constexpr int S_OFF = W_BYTES, X_OFF = W_BYTES + S_BYTES;
    static constexpr int STAGE = X_OFF + 4 * X_BOX;
    static constexpr int NS_FIT = (SMEM_BUDGET - 2048) / STAGE;
    static constexpr int NS = NS_FIT > 8 ? 8 : NS_FIT;         // ring slots
    static constexpr int ND = NP <= 32 ? 8 : 3;                // TMEM accumulator buffers
    static constexpr uint32_t DP = NP <= 32 ? 32 : 96;         // their column pitch
    static constexpr int NBAR = 2 * NS + 2 * NBLK + 2 * ND + 1;
    static constexpr int SMEM = 1024 + NS * STAGE + NBAR * 8 + 64;
    static constexpr uint32_t IDESC = dev::mma_idesc_bf16(BM, NP);
    static_assert(ND * DP <= YCOL && YCOL + NP <= ACOL && ACOL + 16 * NBLK <= TMEM_COLS, "TMEM map");
    static_assert(STAGE % 1024 == 0 && X_OFF % 1024 == 0 && X_BOX % 1024 == 0, "swizzle atoms 1024-aligned");
    static_assert(NS >= 2, "at least two stages");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// the pass width used for the columns col0 .. n_cols - 1 that remain
inline int pass_np(int remaining) { return remaining <= 16 ? 16 : MAX_NP; }

// number of K-segments of length seg_k (the last may be shorter)
inline int n_segments(int K, int seg_k) { return (K + seg_k - 1) / seg_k; }

struct Sched {
    int G;          // CTAs
    long long U;    // units = tiles * ks
    int ks, tiles, seg_st;   // segments, tiles, stages per segment
    __device__ long long begin(int c) const { return (long long)c * U / G; }
    __device__ int cta_of(long long u) const { return (int)(((u + 1) * G - 1) / U); }
};

// The 32 codes of one block of one weight row (16 bytes, byte i = k 2i in the
// low nibble, k 2i+1 in the high one) -> 16 bf16x2 registers of q = code - 8,
// register m = (k 2m, k 2m+1), exact.
__device__ __forceinline__ void codes_to_q(const uint4 &w4, uint32_t (&a)[16]) {
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t u = w[t] >> 4;   // byte i of u holds k 8t+2i+1 in its low nibble
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            // byte 0 <- byte m of w (k 8t+2m), byte 2 <- byte m of u (k 8t+2m+1)
            const uint32_t p = dev::prmt(w[t], u, 0x0400u + 0x0101u * (uint32_t)m);
            const uint32_t b = dev::lop3_and_or(p, 0x000F000Fu, 0x43004300u);   // 128 + code, two bf16
            uint32_t r;
            asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(0x3F803F80u), "r"(0xC308C308u));   // - 136
            a[4 * t + m] = r;
        }
    }
}

// TMEM <-> registers for one epilogue thread's NH columns
template <int NH>
__device__ __forceinline__ void tm_load(uint32_t taddr, float (&v)[NH]) {
    if constexpr (NH == 8) {
        dev::tmem_ld8(taddr, v);
    } else {
        static_assert(NH == 40, "epilogue width");
        dev::tmem_ld32(taddr, v);
        float t[8];
        dev::tmem_ld8(taddr + 32, t);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[32 + j] = t[j];
    }
}

template <int NH>
__device__ __forceinline__ void tm_store(uint32_t taddr, const float (&v)[NH]) {
    if constexpr (NH == 8) {
        dev::tmem_st8(taddr, v);
    } else {
        dev::tmem_st32(taddr, v);
        dev::tmem_st8(taddr + 32, v + 32);
    }
}

__device__ __forceinline__ void named_sync_epilogue() {
    asm volatile("bar.sync 1, %0;" ::"n"(NEW * 32) : "memory");
}

// all lanes agree: every lane's wait succeeded
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, dev::mbar_wait(bar, parity)) != 0;
}

template <int NP, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1)
qmm_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ts,
           const __grid_constant__ CUtensorMap tx, int N, int K, int n_cols, int col0, void *__restrict__ y, int ldy,
           int accumulate, Sched sch, float *__restrict__ wsp_prefix, float *__restrict__ wsp_seg,
           int *__restrict__ counters, int32_t *dev_err) {
    using C = Cfg<NP>;
    constexpr int NH = C::NH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NS * C::STAGE);
    uint64_t *empty = full + C::NS;
    uint64_t *afull = empty + C::NS;
    uint64_t *aempty = afull + NBLK;
    uint64_t *dfull = aempty + NBLK;
    uint64_t *dempty = dfull + C::ND;
    uint64_t *done = dempty + C::ND;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *flag = reinterpret_cast<int *>(tslot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nst_total = K / KS;                     // stages of K
    const int seg_st = sch.seg_st, ks = sch.ks;       // stages per segment, segments
    const long long ua = sch.begin(blockIdx.x), ub = sch.begin(blockIdx.x + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            dev::mbar_init(&full[s], 1);
            dev::mbar_init(&empty[s], NQW + NEW + 1);   // codes, scales and (by commit) activations read
        }
        for (int b = 0; b < NBLK; ++b) {
            dev::mbar_init(&afull[b], 4);               // the four lane quarters of the A buffer
            dev::mbar_init(&aempty[b], 1);
        }
        for (int d = 0; d < C::ND; ++d) {
            dev::mbar_init(&dfull[d], 1);
            dev::mbar_init(&dempty[d], NEW);
        }
        dev::mbar_init(done, 1);
        dev::fence_barrier_init();
    }
    if (warp == W_MMA) dev::tmem_alloc(tslot, TMEM_COLS);
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = *tslot;
    // The weights and scales are constant inputs: the TMA warp starts streaming
    // them at once, overlapping the tail of the preceding kernel on the stream.
    // Activations are read, and anything global is written, only after that
    // kernel has finished (pdl_wait).
    dev::pdl_launch_dependents();

    // stage sequence of this CTA: units ua..ub-1, each 1 or 2 stages (seg_st for the non-invariant variant)
    auto unit_stages = [&](long long u) { return min(seg_st, nst_total - (int)(u % ks) * seg_st); };

    if (warp == W_TMA) {
        // ============================ TMA warp ============================
        if (lane == 0) {
            dev::prefetch_tmap(&tw);
            dev::prefetch_tmap(&ts);
            dev::prefetch_tmap(&tx);
            auto load_x = [&](int slot, int k0) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    dev::tma_load_2d(smem + slot * C::STAGE + C::X_OFF + c * C::X_BOX, &tx, k0 + 64 * c, col0,
                                     &full[slot]);
            };
            long long iu = ua;
            int ist = 0, issued = 0;
            int k0s[C::NS];   // the first NS stages: their activations follow the preceding kernel
            bool x_sent = false;
            for (; iu < ub; ++issued) {
                const int s = issued % C::NS;
                if (issued >= C::NS && !dev::mbar_wait(&empty[s], ((issued / C::NS) - 1) & 1)) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    break;
                }
                const int tile = (int)(iu / ks);
                const int k0 = ((int)(iu % ks) * seg_st + ist) * KS;
                uint8_t *base = smem + s * C::STAGE;
                dev::mbar_arrive_expect_tx(&full[s], W_BYTES + S_BYTES + 4 * C::X_BOX);
                dev::tma_load_2d(base, &tw, k0 / 2, tile * BM, &full[s]);
                dev::tma_load_2d(base + C::S_OFF, &ts, k0 / 32, tile * BM, &full[s]);
                if (x_sent) {
                    load_x(s, k0);
                } else {
                    k0s[issued] = k0;
                    if (issued + 1 == C::NS) {
                        dev::pdl_wait();
                        for (int j = 0; j < C::NS; ++j) load_x(j, k0s[j]);
                        x_sent = true;
                    }
                }
                if (++ist == unit_stages(iu)) {
                    ist = 0;
                    ++iu;
                }
            }
            if (!x_sent) {
                dev::pdl_wait();
                for (int j = 0; j < issued; ++j) load_x(j, k0s[j]);
            }
            // no copy may still be landing in shared memory when the CTA ends
            for (int j = issued > C::NS ? issued - C::NS : 0; j < issued; ++j)
                (void)dev::mbar_wait(&full[j % C::NS], (j / C::NS) & 1);
        }
    } else if (warp == W_MMA) {
        // ============================ MMA issue ============================
        if (lane == 0) {
            long long u = ua;
            int i = 0;
            bool ok = true;
            for (; u < ub && ok; ++u) {
                const int nstg = unit_stages(u);
                for (int st = 0; st < nstg && ok; ++st, ++i) {
                    const int s = i % C::NS;
                    if (!dev::mbar_wait(&full[s], (i / C::NS) & 1)) {
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after();
                    const uint32_t xb = dev::smem_u32(smem + s * C::STAGE + C::X_OFF);
                    for (int b = 0; b < NBLK; ++b) {
                        const int g = i * NBLK + b, db = g % C::ND;
                        if (!dev::mbar_wait(&afull[b], i & 1) ||
                            !dev::mbar_wait(&dempty[db], ((g / C::ND) & 1) ^ 1)) {
                            ok = false;
                            break;
                        }
                        dev::tc_fence_after();
                        const uint32_t d = tmem + db * C::DP, a = tmem + ACOL + 16 * b;
                        const uint32_t bx = xb + (b >> 1) * C::X_BOX + (b & 1) * 64;
                        dev::mma_bf16_tmem_a(d, a, dev::sw128_kmajor_desc(bx), C::IDESC, 0u);
                        dev::mma_bf16_tmem_a(d, a + 8, dev::sw128_kmajor_desc(bx + 32), C::IDESC, 1u);
                        dev::tc_commit(&aempty[b]);
                        dev::tc_commit(&dfull[db]);
                    }
                    if (ok) dev::tc_commit(&empty[s]);
                }
            }
            if (!ok) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
            // every MMA is complete before the TMEM is released
            dev::tc_commit(done);
            (void)dev::mbar_wait(done, 0);
        }
    } else if (warp >= NEW) {
        // ======================== dequantising warps ========================
        const int q = warp & 3, h = (warp - NEW) >> 2;
        const int row = 32 * q + lane;
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + ACOL;
        long long u = ua;
        int i = 0;
        bool ok = true;
        for (; u < ub && ok; ++u) {
            const int nstg = unit_stages(u);
            for (int st = 0; st < nstg; ++st, ++i) {
                const int s = i % C::NS;
                if (!warp_wait(&full[s], (i / C::NS) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t wrow = dev::smem_u32(smem + s * C::STAGE) + row * 128;
                for (int b = h; b < NBLK; b += 2) {
                    if (!warp_wait(&aempty[b], (i & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    uint4 w4;
                    dev::lds128(w4.x, w4.y, w4.z, w4.w, wrow + ((b ^ (row & 7)) << 4));
                    uint32_t a[16];
                    codes_to_q(w4, a);
                    dev::tmem_st16(ta + 16 * b, a);
                    dev::tmem_wait_st();
                    dev::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&afull[b]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&empty[s]);
            }
        }
        if (!ok && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    } else {
        // ============================ epilogue ============================
        const int q = warp & 3, e = warp >> 2;
        const int row = 32 * q + lane;
        const int cbeg = e * NH;                                   // this thread's first column of the pass
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        float *seg_base = wsp_seg + (size_t)row * NP + cbeg;        // + (tile * ks + seg) * BM * NP
        dev::pdl_wait();   // y (accumulate), the workspace and y writes follow the preceding kernel
        float acc[NH];
        float yr[NH];
        int i = 0;
        bool ok = true;
        long long u = ua;
        int nh_tile = -1, nh_prev = 0, nh_touch = 0;   // thread 0: this CTA's later-segment part, if any

        auto store_tile = [&](int tile) {
            const int n = tile * BM + row;
            if (n >= N) return;
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                const int col = col0 + cbeg + j;
                if (col < n_cols) {
                    if (OUT_BF16) {
                        reinterpret_cast<__nv_bfloat16 *>(y)[(size_t)col * ldy + n] = __float2bfloat16_rn(yr[j]);
                    } else {
                        float *yp = reinterpret_cast<float *>(y) + (size_t)col * ldy + n;
                        *yp = accumulate ? (*yp + yr[j]) : yr[j];
                    }
                }
            }
        };
        // yr holds the fold of segments 0 .. seg_from-1 of `tile`: add the stored
        // sums of segments seg_from .. ks-1 in ascending order, write y and reset
        // the tile's counter.  Each stored sum is zeroed once read, so the whole
        // workspace is left zero-filled: a later call whose counters lie where
        // this call kept sums finds them at zero.
        auto fold_tile = [&](int tile, int seg_from) {
            for (int sg = seg_from; sg < ks; ++sg) {
                float4 *p = reinterpret_cast<float4 *>(seg_base + ((size_t)tile * ks + sg) * BM * NP);
                float4 l[NH / 4];
#pragma unroll
                for (int j = 0; j < NH / 4; ++j) l[j] = __ldcg(p + j);
#pragma unroll
                for (int j = 0; j < NH / 4; ++j) __stcg(p + j, make_float4(0.f, 0.f, 0.f, 0.f));
#pragma unroll
                for (int j = 0; j < NH / 4; ++j) {
                    yr[4 * j] += l[j].x;
                    yr[4 * j + 1] += l[j].y;
                    yr[4 * j + 2] += l[j].z;
                    yr[4 * j + 3] += l[j].w;
                }
            }
            store_tile(tile);
            if (threadIdx.x == 0) counters[tile] = 0;
        };
        auto load_y_fold = [&]() {
            if (ok) {
                tm_load<NH>(tq + YCOL + cbeg, yr);
                dev::tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < NH; ++j) yr[j] = 0.f;
            }
        };

        while (u < ub) {
            const int tile = (int)(u / ks);
            const long long tile_u0 = (long long)tile * ks;
            const long long u_end = min(ub, tile_u0 + ks);     // this CTA's units of this tile
            const bool head = (u == tile_u0);
            const bool whole = head && (u_end == tile_u0 + ks);
            for (; u < u_end; ++u) {
                const int seg = (int)(u - tile_u0);
                const int nstg = unit_stages(u);
#pragma unroll
                for (int j = 0; j < NH; ++j) acc[j] = 0.f;
                for (int st = 0; st < nstg; ++st, ++i) {
                    const int s = i % C::NS;
                    if (ok && !warp_wait(&full[s], (i / C::NS) & 1)) ok = false;
                    uint4 sc = make_uint4(0, 0, 0, 0);
                    if (ok)
                        dev::lds128(sc.x, sc.y, sc.z, sc.w,
                                    dev::smem_u32(smem + s * C::STAGE + C::S_OFF) + row * (2 * NBLK));
                    const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll 1
                    for (int b = 0; b < NBLK; ++b) {
                        const int g = i * NBLK + b, db = g % C::ND;
                        if (ok && !warp_wait(&dfull[db], (g / C::ND) & 1)) ok = false;
                        if (ok) {
                            dev::tc_fence_after();
                            float v[NH];
                            tm_load<NH>(tq + db * C::DP + cbeg, v);
                            dev::tmem_wait_ld();
                            dev::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) dev::mbar_arrive(&dempty[db]);
                            const float d =
                                __half2float(__ushort_as_half((unsigned short)(scw[b >> 1] >> (16 * (b & 1)))));
#pragma unroll
                            for (int j = 0; j < NH; ++j) acc[j] = fmaf(d, v[j], acc[j]);
                        }
                    }
                    __syncwarp();
                    if (ok && lane == 0) dev::mbar_arrive(&empty[s]);
                }
                if (head) {
                    // this CTA holds the tile's leading segments: fold them in order (in TMEM)
                    if (seg == 0) {
#pragma unroll
                        for (int j = 0; j < NH; ++j) yr[j] = acc[j];
                    } else {
                        load_y_fold();
#pragma unroll
                        for (int j = 0; j < NH; ++j) yr[j] = yr[j] + acc[j];
                    }
                    if (ok) {
                        tm_store<NH>(tq + YCOL + cbeg, yr);
                        dev::tmem_wait_st();
                    }
                } else {
                    // a later CTA's segment: store its sum for the final fold
                    float4 *ps = reinterpret_cast<float4 *>(wsp_seg + ((size_t)tile * ks + seg) * BM * NP +
                                                            (size_t)row * NP + cbeg);
#pragma unroll
                    for (int j = 0; j < NH / 4; ++j)
                        __stcg(ps + j, make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
                }
            }
            // ---------------- finish this CTA's part of the tile ----------------
            if (whole) {
                load_y_fold();
                store_tile(tile);
                continue;
            }
            const int touch = sch.cta_of(tile_u0 + ks - 1) - sch.cta_of(tile_u0) + 1;   // CTAs sharing the tile
            if (!head) {
                // Later segments of a shared tile: publish their sums and move on.  Whether
                // this CTA was the last to arrive is looked at only after all its units.
                named_sync_epilogue();             // all partial stores of this CTA are issued
                if (threadIdx.x == 0) {
                    __threadfence();               // ... and visible device-wide before the counter moves
                    nh_prev = atomicAdd(&counters[tile], 1);
                    nh_tile = tile;
                    nh_touch = touch;
                }
                continue;
            }
            // Leading segments of a shared tile (the end of this CTA's range).  Usually
            // every other CTA has arrived long ago: then fold at once.
            load_y_fold();
            if (threadIdx.x == 0) {
                int seen;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(counters + tile) : "memory");
                flag[0] = (seen == touch - 1) ? 1 : 0;
            }
            named_sync_epilogue();
            int fold_now = flag[0];
            if (!fold_now) {
                // not yet: leave the prefix for whichever CTA arrives last
                float4 *pp = reinterpret_cast<float4 *>(wsp_prefix + ((size_t)tile * BM + row) * NP + cbeg);
#pragma unroll
                for (int j = 0; j < NH / 4; ++j)
                    __stcg(pp + j, make_float4(yr[4 * j], yr[4 * j + 1], yr[4 * j + 2], yr[4 * j + 3]));
                named_sync_epilogue();             // prefix stores issued; flag[0] read by all
                if (threadIdx.x == 0) {
                    __threadfence();
                    const int prev = atomicAdd(&counters[tile], 1);
                    if (prev == touch - 1) __threadfence();
                    flag[0] = (prev == touch - 1) ? 1 : 0;
                }
                named_sync_epilogue();
                fold_now = flag[0];
                if (fold_now) {
                    // this part arrived last after all: its prefix is not needed, clear it
#pragma unroll
                    for (int j = 0; j < NH / 4; ++j) __stcg(pp + j, make_float4(0.f, 0.f, 0.f, 0.f));
                }
            }
            if (fold_now) {
                const long long head_end = min(sch.begin(blockIdx.x + 1), tile_u0 + ks);
                fold_tile(tile, (int)(head_end - tile_u0));
            }
            named_sync_epilogue();   // flag[0] is read by everyone before it is reused
        }

        // A later-segment part that turned out to arrive last folds its tile now,
        // the prefix and every segment sum coming from the workspace.
        if (threadIdx.x == 0) {
            flag[0] = (nh_tile >= 0 && nh_prev == nh_touch - 1) ? 1 : 0;
            flag[1] = nh_tile;
            if (flag[0]) __threadfence();
        }
        named_sync_epilogue();
        if (flag[0]) {
            const int tile = flag[1];
            const long long tile_u0 = (long long)tile * ks;
            const int head_cta = sch.cta_of(tile_u0);
            const long long head_end = min(sch.begin(head_cta + 1), tile_u0 + ks);
            float4 *pp = reinterpret_cast<float4 *>(wsp_prefix + ((size_t)tile * BM + row) * NP + cbeg);
#pragma unroll
            for (int j = 0; j < NH / 4; ++j) {
                const float4 v = __ldcg(pp + j);
                yr[4 * j] = v.x, yr[4 * j + 1] = v.y, yr[4 * j + 2] = v.z, yr[4 * j + 3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < NH / 4; ++j) __stcg(pp + j, make_float4(0.f, 0.f, 0.f, 0.f));
            fold_tile(tile, (int)(head_end - tile_u0));
        }
        if (!ok && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    }

    // ============================ teardown ============================
    dev::tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        __syncwarp();
        dev::tc_fence_after();
        dev::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// seg512: segment length in units of 512 k (1 for the invariant entry points)
template <int NP, bool OUT_BF16>
spec_status launch_np(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int ldx, int N, int K,
                      int n_cols, int col0, void *y, int ldy, int accumulate, int seg512, void *workspace,
                      int32_t *dev_err, cudaStream_t stream) {
    using C = Cfg<NP>;
    auto kern = qmm_kernel<NP, OUT_BF16>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return spec::cuda_status(e, "cudaFuncSetAttribute(qmm smem)");
        configured = true;
    }
    CUtensorMap tx;
    {
        // the activations: rows = columns j of the product, K contiguous bf16 each
        uint64_t dims[2] = {(uint64_t)K, (uint64_t)n_cols};
        uint64_t strides[1] = {(uint64_t)ldx * 2};
        uint32_t box[2] = {64, (uint32_t)NP};
        if (!spec::encode_tiled(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, x, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return SPEC_ERR_CUDA;
    }
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    Sched sch;
    sch.seg_st = seg512 * (SEG_K / KS);
    sch.ks = n_segments(K, seg512 * SEG_K);
    sch.tiles = (N + BM - 1) / BM;
    sch.U = (long long)sch.tiles * sch.ks;
    sch.G = (int)(sch.U < sms ? sch.U : sms);
    const size_t tiles = (size_t)sch.tiles;
    const size_t cnt_bytes = ((tiles * sizeof(int)) + 255) & ~size_t(255);
    int *counters = reinterpret_cast<int *>(workspace);
    float *prefix = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + cnt_bytes);
    float *segs = prefix + tiles * BM * NP;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sch.G);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, ts, tx, N, K, n_cols, col0, y, ldy, accumulate, sch, prefix,
                                       segs, counters, dev_err);
    return spec::cuda_status(e, "qmm launch");
}

size_t ws_bytes_for(int N, int K, int np, int seg512) {
    const size_t tiles = (size_t)(N + BM - 1) / BM;
    const size_t cnt = ((tiles * sizeof(int)) + 255) & ~size_t(255);
    return cnt + tiles * (1 + (size_t)n_segments(K, seg512 * SEG_K)) * BM * np * sizeof(float);
}

// np_force: 0 = pick each pass's width from the columns left, else that width for every pass
spec_status qmm_run(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x, int n_cols, int ldx,
                    void *y, spec_dtype y_dt, int ldy, int accumulate, int seg512, int np_force, void *workspace,
                    int32_t *dev_err, cudaStream_t stream) {
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
        uint32_t box[2] = {(uint32_t)NBLK, BM};
        if (!spec::encode_tiled(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, ws, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return SPEC_ERR_CUDA;
    }
    const bool bf = (y_dt == SPEC_BF16);
    // passes run back to back on the stream
    for (int col0 = 0; col0 < n_cols;) {
        const int np = np_force ? np_force : pass_np(n_cols - col0);
        spec_status st;
#define SPEC_QMM_CASE(NPV)                                                                                         \
    st = bf ? launch_np<NPV, true>(tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, 0, seg512, workspace, dev_err, stream) \
            : launch_np<NPV, false>(tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, accumulate, seg512, workspace, dev_err, \
                                    stream)
        if (np == 16) {
            SPEC_QMM_CASE(16);
        } else {
            SPEC_QMM_CASE(MAX_NP);
        }
#undef SPEC_QMM_CASE
        if (st != SPEC_OK) return st;
        col0 += np;
    }
    return SPEC_OK;
}

// workspace bytes for any pass of a call with n_cols columns (the widest pass it may run)
size_t ws_bytes_call(int N, int K, int n_cols, int seg512) {
    return ws_bytes_for(N, K, pass_np(n_cols), seg512);
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

spec_status check_ws(const void *workspace, size_t ws_bytes, size_t need) {
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "qmatmul: workspace needs %zu bytes (16-byte aligned, zero-filled "
                                              "before its first use), got %zu", need, ws_bytes);
    return SPEC_OK;
}

}  // namespace

extern "C" size_t spec_qmatmul_workspace(int N, int K, int n_cols) {
    if (N <= 0 || K < 256 || n_cols <= 0) return 0;
    // the largest layout either entry point may use for this shape (one-stage segments)
    return ws_bytes_call(N, K, n_cols, 1);
}

extern "C" spec_status spec_qmatmul(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                    int n_cols, int ldx, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                    void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    st = check_ws(workspace, ws_bytes, ws_bytes_call(N, K, n_cols, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, 0, workspace, dev_err,
                   (cudaStream_t)stream);
}

extern "C" spec_status spec_qmatmul_noninvariant(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                                 const uint16_t *x, int n_cols, int ldx, float *y, int ldy,
                                                 int seg_stages, void *workspace, size_t ws_bytes,
                                                 spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    if (n_cols == 0) return SPEC_OK;
    const int nst = n_segments(K, SEG_K);   // 512-k units
    int seg = seg_stages;
    if (seg <= 0) {
        // per-call choice: the longest segment that still deals every SM about eight units
        const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
        const long long tiles = (N + BM - 1) / BM;
        seg = nst;
        while (seg > 1 && tiles * n_segments(K, seg * SEG_K) < 8ll * sms) seg = (seg + 1) / 2;
    }
    SPEC_CHECK_ARG(seg >= 1, "qmatmul_noninvariant: seg_stages must be >= 0");
    if (seg > nst) seg = nst;
    st = check_ws(workspace, ws_bytes, ws_bytes_call(N, K, n_cols, seg));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, seg, 0, workspace, nullptr,
                   (cudaStream_t)stream);
}

// Test hook: run the invariant kernel with an explicit pass width so the tests
// can show the per-column result does not depend on it.
extern "C" spec_status spec_qmatmul_debug_nt(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                             int n_cols, int ldx, float *y, int ldy, int nt, void *workspace,
                                             size_t ws_bytes, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(nt == 2 || nt == MAX_NP / 8, "nt must be 2 (16 columns per pass) or 10 (80)");
    if (n_cols == 0) return SPEC_OK;
    st = check_ws(workspace, ws_bytes, ws_bytes_for(N, K, 8 * nt, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, 1, 8 * nt, workspace, nullptr,
                   (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// spec_qmatmul_static_scratch: the invariant product with its scratch in a
// fixed, statically sized device array instead of a caller-supplied buffer.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

// One scratch area per device (module-scope __device__ storage is per device).
// Its front holds the per-tile arrival counters, which must be zero when a
// launch starts; the rest holds partial sums that each call writes before it
// reads them.
static __device__ __align__(256) unsigned char g_qmm_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch; looked up on the first call made
// with that device current.
spec_status static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return spec::cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return spec::fail(SPEC_ERR_INVALID_ARG, "qmatmul_static_scratch: device %d", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_qmm_static_scratch);
        if (e != cudaSuccess) return spec::cuda_status(e, "cudaGetSymbolAddress(qmatmul scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_qmatmul_static_scratch(const uint8_t *wq, const uint16_t *ws, int N, int K,
                                                   const uint16_t *x, int n_cols, int ldx, void *y, spec_dtype y_dt,
                                                   int ldy, int accumulate, int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    const size_t need = ws_bytes_call(N, K, n_cols, 1);
    if (need > kStaticScratchBytes)
        return spec::fail(SPEC_ERR_WORKSPACE,
                          "qmatmul_static_scratch: N=%d K=%d n_cols=%d needs %zu bytes of scratch, more than the "
                          "fixed %zu; use spec_qmatmul with a workspace",
                          N, K, n_cols, need, kStaticScratchBytes);
    void *scratch = nullptr;
    st = static_scratch(&scratch);
    if (st != SPEC_OK) return st;
    // the arrival counters must start at zero: clear them on the stream first
    const size_t tiles = (size_t)(N + BM - 1) / BM;
    cudaError_t e = cudaMemsetAsync(scratch, 0, tiles * sizeof(int), (cudaStream_t)stream);
    if (e != cudaSuccess) return spec::cuda_status(e, "cudaMemsetAsync(qmatmul scratch counters)");
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, 0, scratch, dev_err,
                   (cudaStream_t)stream);
}
