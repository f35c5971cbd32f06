// K1's 80-column pass on the 5th-generation tensor cores (sm_103a):
// tcgen05.mma with the dequantised weights in tensor memory (TMEM), the
// activation columns in shared memory, fp32 accumulators in TMEM.
//
// Arithmetic: exactly that of the mma.sync passes in qmatmul.cu, bit for bit.
// For every 32-k block b of a K-segment, in ascending order, the block product
// T_b of column j is one chain of two K = 16 tensor-core products from a zero
// accumulator, with A = 128 + code (bf16, exact) and B = column j's bf16
// activations, each k of the block in the same MMA slot as in the mma.sync
// fragments (slot 2t, 2t+1, 2t+8, 2t+9 of the first product hold k = 8t, 8t+4,
// 8t+1, 8t+5; of the second 8t+2, 8t+6, 8t+3, 8t+7); then
// s = fma(d_b, T_b + c_b, s) from s = +0 with c_b = -136 x the column's block
// sum, and the segment sums are folded in segment order.  The tensor core
// evaluates a K = 16 chain identically through tcgen05.mma and
// mma.sync.m16n8k16 (measured on this GPU: all 2^14 elements of a 128 x 16 x 32
// product equal bit for bit, from zero and from a given C; the tests compare
// every column position across pass widths), so a column's result does not
// depend on the pass that computed it.
//
// Execution: a persistent grid of one CTA per SM over (128-row tile x
// K-segment) units dealt out in equal contiguous ranges (the schedule of
// qmatmul.cu).  Per CTA, 14 warps:
//  * warp 0 (one lane): TMA -- per 256-k stage the codes (128 rows x 128 bytes,
//    128-byte swizzle), the fp16 scales and, by one bulk copy, the pass's
//    packed activations (the MMA's B operand in the 128-byte-swizzle K-major
//    layout, then the -136 x block sums) into a 3-slot mbarrier ring;
//  * warp 1: owns the TMEM allocation; one lane issues the two MMAs of each
//    block into one of four accumulators (N = 80, the first from zero) and
//    commits them;
//  * warps 2-5 (one per TMEM lane quarter): turn each block's codes into
//    128 + code bf16 pairs (4 LOP3 + 3 shifts per 8 weights) and store them
//    into TMEM A buffers (lane = weight row), handing them to the MMA four
//    blocks (half a stage) at a time, three such groups in flight;
//  * warps 6-13 (two per lane quarter, 40 columns each): per block, load the
//    accumulator from TMEM and release it to the MMA at once, then apply
//    s = fma(d_b, T_b + c_b, s) in registers; fold segments (in shared
//    memory), write y, or publish split-tile sums as qmatmul.cu's consumers
//    do (no CTA ever waits for another).
// Measured on this GPU (80 columns, graph of calls): 60.6 us at 32000 x 2048
// and 37.4 us at 11264 x 2048, against 59.2 and 34.5 us for the mma.sync
// kernel; the two MMAs of a block take ~80 cycles of tensor-core time, but
// each 80-column accumulator goes MMA -> epilogue -> MMA once per block and,
// with four of them in tensor memory, that round trip (~3600 cycles in place)
// sets the rate.  Reworked hand-overs (shared counters instead of mbarriers,
// a warp that alone waits on the MMA completions, sixteen epilogue warps of
// 20 columns) were each slower.  The kernel is therefore not chosen by
// default; spec_qmatmul_debug_nt(nt = 11) runs it, and the tests hold it to
// the mma.sync kernel's bits.
// Every wait is bounded; on expiry the kernel sets SPEC_DEVERR_TIMEOUT, lets
// its own copies and MMAs finish (bounded), frees TMEM and returns.
//
// Source of the operation: ramgpt.org, "When Lossless Speculation Stops Being
// Lossless on Blackwell", section "Quantized Matrix Multiplication Shows the
// Same Class of Failure" (the batched product must equal per-column products).
#include "qmm_shared.cuh"

namespace {
using namespace qmm;

constexpr int NBLK = 8;                          // 32-k blocks per 256-k stage
constexpr int NP = WIDE_COLS;                    // columns per pass (MMA N)
constexpr int W_BYTES = BM * 128;                // one stage of codes
constexpr int S_BYTES = BM * NBLK * 2;           // one stage of fp16 scales
constexpr int X_BOX = NP * 128;                  // 64 k of the pass's columns (B operand)
constexpr int S_OFF = W_BYTES;
constexpr int X_OFF = W_BYTES + S_BYTES;         // 1024-aligned (swizzle atoms)
constexpr int CI_OFF = X_OFF + 4 * X_BOX;        // [8 blocks][80] fp32: -136 x block sums
constexpr int STAGE = (X_OFF + WIDE_XC_BYTES + 1023) / 1024 * 1024;
constexpr int NS = 3;                            // ring slots
constexpr int HB = 4;                            // blocks per half-stage (the A hand-over unit)
constexpr int NA = 3;                            // TMEM A groups (HB buffers of 16 columns each)
constexpr int ND = 4;                            // TMEM accumulators
constexpr uint32_t DP = 80;                      // accumulator column pitch
constexpr uint32_t ACOL = ND * DP;               // first A column
constexpr uint32_t TMEM_COLS = 512;
constexpr int W_TMA = 0, W_MMA = 1, W_EP = 6;   // warps 2..5 dequantise
constexpr int NDQ = 4, NEP = 8, EPC = NP / 2;    // dequant warps, epilogue warps, columns per epilogue thread
constexpr int THREADS = (W_EP + NEP) * 32;
constexpr int NBAR = 2 * NS + 2 * NA + 2 * ND + 1;
constexpr int YS_BYTES = BM * NP * 4;            // the tile's running segment fold, [column][row] fp32
constexpr int SMEM = 1024 + NS * STAGE + YS_BYTES + NBAR * 8 + 64;
constexpr uint32_t IDESC = dev::mma_idesc_bf16(BM, NP);
constexpr int TILE_ELEMS = BM * NP;
static_assert(X_OFF % 1024 == 0 && X_BOX % 1024 == 0 && STAGE % 1024 == 0, "swizzle atoms 1024-byte aligned");
static_assert(ACOL + 16 * HB * NA <= TMEM_COLS && NBLK % HB == 0, "TMEM map");
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(EPC == 40, "epilogue loads: 32 + 8 columns");

// 8 codes (k = 8t .. 8t+7 of a block) -> (128 + c_8t, 128 + c_8t+4), (.. 8t+1, 8t+5),
// (.. 8t+2, 8t+6), (.. 8t+3, 8t+7), bf16 pairs, exact
__device__ __forceinline__ void codes8(uint32_t w, uint32_t &o0, uint32_t &o1, uint32_t &o2, uint32_t &o3) {
    o0 = dev::lop3_and_or(w, 0x000F000Fu, 0x43004300u);
    o1 = dev::lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u);
    o2 = dev::lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u);
    o3 = dev::lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u);
}

__device__ __forceinline__ void named_sync_epilogue() { asm volatile("bar.sync 1, %0;" ::"n"(NEP * 32) : "memory"); }

// every lane of the warp waits (bounded); true when every lane's wait succeeded
// (one lane polling and broadcasting measured slower: its try_wait wakes later)
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, dev::mbar_wait(bar, parity)) != 0;
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1)
qmm_tc_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ts, int N, int K,
              int n_cols, int col0, void *__restrict__ y, int ldy, int accumulate, Sched sch,
              float *__restrict__ wsp_prefix, float *__restrict__ wsp_seg, int *__restrict__ counters,
              const uint8_t *__restrict__ xpk, int32_t *dev_err, const int32_t *dev_cols, int min_cols) {
    if (dev_cols) {
        // the column count is the preceding kernel's output: no early streaming
        dev::pdl_wait();
        n_cols = gated_cols(n_cols, dev_cols, min_cols);
    }
    if (col0 >= n_cols) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *ysm = reinterpret_cast<float *>(smem + NS * STAGE);   // per tile: fold of its leading segments
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * STAGE + YS_BYTES);
    uint64_t *empty = full + NS;
    uint64_t *afull = empty + NS;
    uint64_t *aempty = afull + NA;
    uint64_t *dfull = aempty + NA;
    uint64_t *dempty = dfull + ND;
    uint64_t *done = dempty + ND;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *flag = reinterpret_cast<int *>(tslot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nst_total = K / WIDE_KS;
    const int seg_st = sch.seg_st, ks = sch.ks;
    const long long ua = sch.begin(blockIdx.x), ub = sch.begin(blockIdx.x + 1);
    auto unit_stages = [&](long long u) { return min(seg_st, nst_total - (int)(u % ks) * seg_st); };
    // stages of this CTA
    int my_stages = 0;
    for (long long u = ua; u < ub; ++u) my_stages += unit_stages(u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            dev::mbar_init(&full[s], 1);
            dev::mbar_init(&empty[s], NDQ + NEP + 1);
        }
        for (int a = 0; a < NA; ++a) {
            dev::mbar_init(&afull[a], NDQ);
            dev::mbar_init(&aempty[a], 1);
        }
        for (int d = 0; d < ND; ++d) {
            dev::mbar_init(&dfull[d], 1);
            dev::mbar_init(&dempty[d], NEP);
        }
        dev::mbar_init(done, 1);
        dev::fence_barrier_init();
    }
    if (warp == W_MMA) dev::tmem_alloc(tslot, TMEM_COLS);
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tmem = *tslot;
    // weights and scales are constant inputs: stream them at once; the packed
    // activations, y and the workspace follow the preceding kernels (pdl_wait)
    dev::pdl_launch_dependents();

    if (warp == W_TMA) {
        // ============================ TMA ============================
        if (lane == 0) {
            dev::prefetch_tmap(&tw);
            dev::prefetch_tmap(&ts);
            long long iu = ua;
            int ist = 0, issued = 0;
            int k0s[NS];
            bool x_sent = false, ok = true;
            for (; iu < ub; ++issued) {
                const int s = issued % NS;
                if (issued == NS) {
                    // the first NS stages' weights are on their way; their activations
                    // are written by the preceding kernel
                    x_sent = true;
                    dev::pdl_wait();
                    for (int j = 0; j < NS; ++j)
                        dev::bulk_load(smem + j * STAGE + X_OFF, xpk + (size_t)(k0s[j] / WIDE_KS) * WIDE_XC_BYTES,
                                       WIDE_XC_BYTES, &full[j]);
                }
                if (issued >= NS && !dev::mbar_wait(&empty[s], ((issued / NS) - 1) & 1)) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    ok = false;
                    break;
                }
                const int tile = (int)(iu / ks);
                const int k0 = ((int)(iu % ks) * seg_st + ist) * WIDE_KS;
                uint8_t *base = smem + s * STAGE;
                dev::mbar_arrive_expect_tx(&full[s], W_BYTES + S_BYTES + WIDE_XC_BYTES);
                dev::tma_load_2d(base, &tw, k0 / 2, tile * BM, &full[s]);
                dev::tma_load_2d(base + S_OFF, &ts, k0 / 32, tile * BM, &full[s]);
                if (issued < NS)
                    k0s[issued] = k0;
                else
                    dev::bulk_load(base + X_OFF, xpk + (size_t)(k0 / WIDE_KS) * WIDE_XC_BYTES, WIDE_XC_BYTES,
                                   &full[s]);
                if (++ist == unit_stages(iu)) {
                    ist = 0;
                    ++iu;
                }
            }
            if (!x_sent) {
                dev::pdl_wait();
                for (int j = 0; j < issued && j < NS; ++j)
                    dev::bulk_load(smem + j * STAGE + X_OFF, xpk + (size_t)(k0s[j] / WIDE_KS) * WIDE_XC_BYTES,
                                   WIDE_XC_BYTES, &full[j]);
            }
            // copies still in flight land before the CTA may exit: wait for the last
            // NS stages' arrivals (they have normally long completed)
            for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
                if (!dev::mbar_wait(&full[j % NS], (j / NS) & 1) && ok) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    ok = false;
                }
        }
    } else if (warp == W_MMA) {
        // ============================ MMA ============================
        // The whole warp runs the loop; one elected lane issues each MMA and
        // commit.  Every operand is kept warp-uniform and as much as possible
        // fixed at compile time (a stage's eight blocks are unrolled; a stage
        // starts at a block count that is a multiple of eight): the issue
        // rate of tcgen05.mma depends on it.
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint64_t desc0 = dev::sw128_kmajor_desc(dev::smem_u32(smem + X_OFF));
        bool ok = true;
        for (int st = 0; st < my_stages && ok; ++st) {
            const int s = st % NS;
            ok = warp_wait(&full[s], (st / NS) & 1);
            if (!ok) break;
            dev::tc_fence_after();
            // the start-address field (address / 16, 14 bits) advances without a carry
            const uint64_t sdesc = desc0 + (uint64_t)((s * STAGE) >> 4);
#pragma unroll
            for (int h = 0; h < NBLK / HB; ++h) {
                const int hs = 2 * st + h, g = hs % NA;   // the half-stage and its A group
                ok = ok && warp_wait(&afull[g], (hs / NA) & 1);
                const uint32_t ag = tm + ACOL + g * HB * 16;
#pragma unroll
                for (int b = 0; b < HB; ++b) {
                    const int jb = h * HB + b, d = jb % ND;   // block jb of the stage; i % ND == jb % ND
                    const int i = NBLK * st + jb;
                    ok = ok && (i < ND || warp_wait(&dempty[d], ((i / ND) - 1) & 1));
                    if (!ok) break;
                    dev::tc_fence_after();
                    const uint64_t bd = sdesc + (uint64_t)(((jb >> 1) * X_BOX + (jb & 1) * 64) >> 4);
                    dev::mma_bf16_tmem_a(tm + d * DP, ag + b * 16, bd, IDESC, 0);
                    dev::mma_bf16_tmem_a(tm + d * DP, ag + b * 16 + 8, bd + 2, IDESC, 1);
                    dev::tc_commit(&dfull[d]);
                }
                if (ok) dev::tc_commit(&aempty[g]);   // the group's A buffers are read
            }
            if (ok) dev::tc_commit(&empty[s]);
        }
        if (!ok && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
        // every MMA issued has completed before TMEM is released
        dev::tc_commit(done);
        if (!warp_wait(done, 0) && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    } else if (warp < W_EP) {
        // ========================= dequantisers =========================
        const int q = warp & 3;                  // TMEM lane quarter
        const int row = 32 * q + lane;           // weight row of the tile
        const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + ACOL;
        bool ok = true;
        int i = 0;
        for (int st = 0; st < my_stages && ok; ++st) {
            const int s = st % NS;
            ok = warp_wait(&full[s], (st / NS) & 1);
            const uint32_t cb = dev::smem_u32(smem + s * STAGE) + row * 128;
            for (int jb = 0; jb < NBLK && ok; ++jb, ++i) {
                const int hs = i / HB, g = hs % NA;
                if (jb % HB == 0) {
                    if (hs >= NA && !warp_wait(&aempty[g], ((hs / NA) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after();
                }
                uint32_t w0, w1, w2, w3;
                dev::lds128(w0, w1, w2, w3, cb + ((jb ^ (row & 7)) << 4));
                uint32_t r[16];
                codes8(w0, r[0], r[4], r[8], r[12]);
                codes8(w1, r[1], r[5], r[9], r[13]);
                codes8(w2, r[2], r[6], r[10], r[14]);
                codes8(w3, r[3], r[7], r[11], r[15]);
                dev::tmem_st16(tbase + (g * HB + jb % HB) * 16, r);
                if (jb % HB == HB - 1) {
                    // the group's four blocks are in tensor memory: hand them to the MMA
                    dev::tmem_wait_st();
                    dev::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&afull[g]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) dev::mbar_arrive(&empty[s]);
        }
        if (!ok && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    } else {
        // =========================== epilogue ===========================
        dev::pdl_wait();   // y (accumulate) and the workspace follow the preceding kernel
        const int q = warp & 3, h = (warp - W_EP) >> 2;
        const int row = 32 * q + lane;
        const int c0 = h * EPC;                  // this thread's first column of the pass
        const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16) + c0;
        const int frag = c0 * BM + row;          // + c * BM: [column][row] layout of the tile's sums
        const int ep_tid = threadIdx.x - W_EP * 32;
        bool ok = true;
        float s_acc[EPC];
#pragma unroll
        for (int c = 0; c < EPC; ++c) s_acc[c] = 0.f;
        float *yrun = ysm + frag;                // this thread's fold entries: yrun[c * BM]

        auto store_y = [&](int tile) {
            const int n = tile * BM + row;
            if (n >= N) return;
            float yv[EPC];
#pragma unroll
            for (int c = 0; c < EPC; ++c) yv[c] = yrun[c * BM];
#pragma unroll
            for (int c = 0; c < EPC; ++c) {
                const int col = col0 + c0 + c;
                if (col < n_cols) {
                    const float v = yv[c];
                    if (OUT_BF16) {
                        reinterpret_cast<__nv_bfloat16 *>(y)[(size_t)col * ldy + n] = __float2bfloat16_rn(v);
                    } else {
                        float *yp = reinterpret_cast<float *>(y) + (size_t)col * ldy + n;
                        *yp = accumulate ? (*yp + v) : v;
                    }
                }
            }
        };
        auto clear_low = [&](float *p) {
            if ((size_t)(reinterpret_cast<const uint8_t *>(p) - reinterpret_cast<const uint8_t *>(counters)) <
                CNT_LIMIT)
                __stcg(p, 0.f);
        };
        const bool col_live[1] = {col0 + c0 < n_cols};   // any of this thread's columns in range
        // yrun holds the fold of segments 0 .. seg_from-1: add the stored sums of
        // segments seg_from .. ks-1 in order, write y, reset the counter, clear what
        // a later call could take for counters
        auto fold_tile = [&](int tile, int seg_from) {
            const float *p0 = wsp_seg + (size_t)tile * ks * TILE_ELEMS + frag;
            if (col_live[0]) {
                // the fold in registers, each segment's loads all in flight before they are added
                // (through shared memory the adds would wait for every load in turn)
                float f[EPC];
#pragma unroll
                for (int c = 0; c < EPC; ++c) f[c] = yrun[c * BM];
                for (int sg = seg_from; sg < ks; ++sg) {
                    float l[EPC];
#pragma unroll
                    for (int c = 0; c < EPC; ++c) l[c] = __ldcg(p0 + (size_t)sg * TILE_ELEMS + c * BM);
#pragma unroll
                    for (int c = 0; c < EPC; ++c) f[c] += l[c];
                }
#pragma unroll
                for (int c = 0; c < EPC; ++c) yrun[c * BM] = f[c];
            }
            store_y(tile);
            if (ep_tid == 0) counters[tile] = 0;
            if (col_live[0])
                for (int sg = seg_from; sg < ks; ++sg)
#pragma unroll
                    for (int c = 0; c < EPC; ++c) clear_low(const_cast<float *>(p0) + (size_t)sg * TILE_ELEMS + c * BM);
        };

        int i = 0, st_i = 0;
        int nh_tile = -1, nh_prev = 0, nh_touch = 0;   // ep_tid 0: this CTA's later-segment part, if any
        long long u = ua;
        while (u < ub) {
            const int tile = (int)(u / ks);
            const long long tile_u0 = (long long)tile * ks;
            const long long u_end = min(ub, tile_u0 + ks);
            const bool head = (u == tile_u0);
            const bool whole = head && (u_end == tile_u0 + ks);
            for (; u < u_end; ++u) {
                const int seg = (int)(u - tile_u0);
                const int nstg = unit_stages(u);
                for (int st = 0; st < nstg; ++st, ++st_i) {
                    const int s = st_i % NS;
                    if (ok) ok = warp_wait(&full[s], (st_i / NS) & 1);
                    // this row's eight fp16 block scales of the stage
                    const uint4 sc = *reinterpret_cast<const uint4 *>(smem + s * STAGE + S_OFF + row * 16);
                    const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
                    for (int jb = 0; jb < NBLK; ++jb, ++i) {
                        const int d = i % ND;
                        if (ok) ok = warp_wait(&dfull[d], (i / ND) & 1);
                        dev::tc_fence_after();
                        uint32_t v[EPC];
                        dev::tmem_ld32(tlane + d * DP, v);
                        dev::tmem_ld8(tlane + d * DP + 32, v + 32);
                        dev::tmem_wait_ld();
                        // the accumulator is read: the MMA may reuse it
                        dev::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) dev::mbar_arrive(&dempty[d]);
                        const float dsc = __half2float(__ushort_as_half((unsigned short)(sw[jb >> 1] >> (16 * (jb & 1)))));
                        const float *ci = reinterpret_cast<const float *>(smem + s * STAGE + CI_OFF) + jb * NP + c0;
#pragma unroll
                        for (int g = 0; g < EPC / 4; ++g) {
                            const float4 cv = *reinterpret_cast<const float4 *>(ci + 4 * g);
                            dev::fma_add_f32x2(s_acc[4 * g], s_acc[4 * g + 1], dsc, __uint_as_float(v[4 * g]),
                                               __uint_as_float(v[4 * g + 1]), cv.x, cv.y);
                            dev::fma_add_f32x2(s_acc[4 * g + 2], s_acc[4 * g + 3], dsc, __uint_as_float(v[4 * g + 2]),
                                               __uint_as_float(v[4 * g + 3]), cv.z, cv.w);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&empty[s]);
                }
                if (head) {
#pragma unroll
                    for (int c = 0; c < EPC; ++c) yrun[c * BM] = (seg == 0) ? s_acc[c] : yrun[c * BM] + s_acc[c];
                } else if (col_live[0]) {
                    float *ps = wsp_seg + ((size_t)tile * ks + seg) * TILE_ELEMS + frag;
#pragma unroll
                    for (int c = 0; c < EPC; ++c) __stcg(ps + c * BM, s_acc[c]);
                }
#pragma unroll
                for (int c = 0; c < EPC; ++c) s_acc[c] = 0.f;
            }
            // ---------------- finish this CTA's part of the tile ----------------
            if (whole) {
                store_y(tile);
                continue;
            }
            const int touch = sch.cta_of(tile_u0 + ks - 1) - sch.cta_of(tile_u0) + 1;
            if (!head) {
                named_sync_epilogue();
                if (ep_tid == 0) {
                    __threadfence();
                    nh_prev = atomicAdd(&counters[tile], 1);
                    nh_tile = tile;
                    nh_touch = touch;
                }
                continue;
            }
            if (ep_tid == 0) {
                int seen;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(counters + tile) : "memory");
                flag[0] = (seen == touch - 1) ? 1 : 0;
            }
            named_sync_epilogue();
            int fold_now = flag[0];
            if (!fold_now) {
                float *pp = wsp_prefix + (size_t)tile * TILE_ELEMS + frag;
                if (col_live[0]) {
#pragma unroll 8
                    for (int c = 0; c < EPC; ++c) __stcg(pp + c * BM, yrun[c * BM]);
                }
                named_sync_epilogue();
                if (ep_tid == 0) {
                    __threadfence();
                    const int prev = atomicAdd(&counters[tile], 1);
                    if (prev == touch - 1) __threadfence();
                    flag[0] = (prev == touch - 1) ? 1 : 0;
                }
                named_sync_epilogue();
                fold_now = flag[0];
                if (fold_now) {
                    const long long head_end = min(sch.begin(blockIdx.x + 1), tile_u0 + ks);
                    fold_tile(tile, (int)(head_end - tile_u0));
                    if (col_live[0]) {
#pragma unroll
                        for (int c = 0; c < EPC; ++c) clear_low(pp + c * BM);
                    }
                    fold_now = 0;
                }
            }
            if (fold_now) {
                const long long head_end = min(sch.begin(blockIdx.x + 1), tile_u0 + ks);
                fold_tile(tile, (int)(head_end - tile_u0));
            }
            named_sync_epilogue();
        }
        // a later-segment part that arrived last folds its tile now
        if (ep_tid == 0) {
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
            float *pp = wsp_prefix + (size_t)tile * TILE_ELEMS + frag;
            if (col_live[0]) {
                float l[EPC];
#pragma unroll
                for (int c = 0; c < EPC; ++c) l[c] = __ldcg(pp + c * BM);
#pragma unroll
                for (int c = 0; c < EPC; ++c) yrun[c * BM] = l[c];
            }
            fold_tile(tile, (int)(head_end - tile_u0));
            if (col_live[0]) {
#pragma unroll
                for (int c = 0; c < EPC; ++c) clear_low(pp + c * BM);
            }
        }
        if (!ok && lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    }

    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    if (warp == W_MMA) dev::tmem_dealloc(tmem, TMEM_COLS);
}

// Packs the activations of one 80-column pass for every 256-k stage of K: per
// (stage, block, column) the block's 32 bf16 values in MMA slot order (first
// product: k = 0, 4, 8, .. 28, then 1, 5, .. 29; second: 2, 6, .. 30, then 3,
// 7, .. 31) at the column's 128-byte row of the stage's 64-k group, 16-byte
// chunks swizzled by the row (the 128-byte-swizzle K-major layout the MMA
// reads), and -136 x the block sum (four 8-k chunk sums, each in k order,
// added in chunk order; the same expression as qmatmul.cu's activation warps).
__global__ void __launch_bounds__(256) xpack_tc_kernel(const uint16_t *__restrict__ x, int ldx, int K, int n_cols,
                                                       int col0, uint8_t *__restrict__ out, const int32_t *dev_cols,
                                                       int min_cols) {
    dev::pdl_wait();   // x is the preceding kernel's output; out may still be read by it
    dev::pdl_launch_dependents();
    if (dev_cols) n_cols = gated_cols(n_cols, dev_cols, min_cols);
    if (col0 >= n_cols) return;
    constexpr int PAIRS = NBLK * NP;   // per stage
    const long long p = blockIdx.x * 256ll + threadIdx.x;
    const int st = (int)(p / PAIRS), pr = (int)(p % PAIRS);
    if (st * WIDE_KS >= K) return;
    const int blk = pr / NP, c = pr % NP;
    const int col = col0 + c, kb = st * WIDE_KS + 32 * blk;
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = make_uint4(0, 0, 0, 0);
        if (col < n_cols) v[q] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)col * ldx + kb + 8 * q));
    }
    float sum = 0.f;
    uint32_t o[4][4];   // [q][pair]: (k 8q+e, 8q+e+4) for e = 0..3
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
        float cs = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            cs += __uint_as_float(w4[e] << 16);
            cs += __uint_as_float(w4[e] & 0xFFFF0000u);
        }
        sum = (q == 0) ? cs : sum + cs;
        o[q][0] = dev::prmt(w4[0], w4[2], 0x5410);   // (x 8q,   x 8q+4)
        o[q][1] = dev::prmt(w4[0], w4[2], 0x7632);   // (x 8q+1, x 8q+5)
        o[q][2] = dev::prmt(w4[1], w4[3], 0x5410);   // (x 8q+2, x 8q+6)
        o[q][3] = dev::prmt(w4[1], w4[3], 0x7632);   // (x 8q+3, x 8q+7)
    }
    uint8_t *base = out + (size_t)st * WIDE_XC_BYTES;
    uint8_t *rowp = base + (blk >> 1) * X_BOX + (c >> 3) * 1024 + (c & 7) * 128;
    // logical 16-byte chunk 4 (blk & 1) + e holds pair e of chunks q = 0..3
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int chunk = ((blk & 1) * 4 + e) ^ (c & 7);
        *reinterpret_cast<uint4 *>(rowp + (chunk << 4)) = make_uint4(o[0][e], o[1][e], o[2][e], o[3][e]);
    }
    reinterpret_cast<float *>(base + 4 * X_BOX)[blk * NP + c] = -136.0f * sum;
}

}  // namespace

namespace qmm {

spec_status tc_wide_pass(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int ldx, int N, int K,
                         int n_cols, int col0, void *y, bool out_bf16, int ldy, int accumulate, int seg512,
                         void *workspace, int32_t *dev_err, const int32_t *dev_cols, int min_cols,
                         cudaStream_t stream) {
    static spec::SmemOptIn opt_f32, opt_bf16;
    spec_status so = out_bf16 ? spec::smem_opt_in(qmm_tc_kernel<true>, SMEM, opt_bf16, "cudaFuncSetAttribute(qmm tc)")
                              : spec::smem_opt_in(qmm_tc_kernel<false>, SMEM, opt_f32, "cudaFuncSetAttribute(qmm tc)");
    if (so != SPEC_OK) return so;
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    const Sched sch = make_sched(N, K, seg512, WIDE_KS, sms);
    const WsLayout w = ws_layout(workspace, sch.tiles, sch.ks, TILE_ELEMS);
    const long long pairs = (long long)(K / WIDE_KS) * NBLK * NP;
    cudaError_t e = spec::launch_pdl(xpack_tc_kernel, dim3((unsigned)((pairs + 255) / 256)), dim3(256), 0, stream, x,
                                     ldx, K, n_cols, col0, w.xpk, dev_cols, min_cols);
    if (e != cudaSuccess) return spec::cuda_status(e, "qmm tc activation pack launch");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sch.G);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (out_bf16)
        e = cudaLaunchKernelEx(&cfg, qmm_tc_kernel<true>, tw, ts, N, K, n_cols, col0, y, ldy, 0, sch, w.prefix, w.segs,
                               w.counters, (const uint8_t *)w.xpk, dev_err, dev_cols, min_cols);
    else
        e = cudaLaunchKernelEx(&cfg, qmm_tc_kernel<false>, tw, ts, N, K, n_cols, col0, y, ldy, accumulate, sch,
                               w.prefix, w.segs, w.counters, (const uint8_t *)w.xpk, dev_err, dev_cols, min_cols);
    return spec::cuda_status(e, "qmm tc launch");
}

}  // namespace qmm
