// K1: batch-invariant int4 block-32 dequantising matmul (sm_103a).
//
//   y[j][n] = sum_k x[j][k] * d[n][k/32] * (nib(n, k) - 8)
//
// Per-element arithmetic (identical for every call, whatever n_cols is and
// wherever column j sits):
//  * K is cut into segments of 512 (when K / 256 is odd the last segment is
//    256 long).  The cut depends on K only.
//  * Inside a segment, for every 32-k block b in ascending order, the block
//    product T_b is one chain of two m16n8k16 bf16 MMAs from a zero
//    accumulator whose A operand is the code c = q + 8 plus 128 (exactly
//    representable); the block partial is P_b = T_b + (-136 * sum_{k in b}
//    x[j][k]) in fp32 (column j's block sum in fp32, its four 8-k chunks
//    summed in k order and then in chunk order), so P_b = sum q x up to
//    rounding; then s = fma(d_b, P_b, s) with s starting at +0.
//  * The segment sums are folded in ascending order: y = ((s_0 + s_1) + s_2)...
// The MMA instruction stream is the same for every column tile and column j's
// result depends only on A, on B column j and on C column j; unused columns
// are zero, never a different instruction.  Which CTA, warp or column tile
// handles a column, and where a CTA's share of the work starts and ends, is
// scheduling that may depend on the call; the arithmetic above never does.
//
// Execution: a persistent grid of one CTA per SM, each with eight consumer
// warps (128 rows per tile: 16 rows x all columns each in passes of up to 16
// columns, 32 rows x 40 columns each in the 80-column pass).  The (128-row tile
// x K-segment) units are dealt out in equal contiguous ranges (stream-K), so
// every SM streams the same number of bytes; a matrix with nearly one tile per
// SM gives each CTA one whole tile instead.  One lane issues cp.async.bulk.tensor
// copies of each stage -- the int4 codes (128-row x 128-byte boxes, 128B
// swizzle) and the scales (fp16 per block, or the super-block records of
// spec_qmatmul_sb) -- into a ring of mbarrier-guarded stages: lane 0 of a TMA
// warp in the narrow passes, lane 0 of consumer warp 0 in the 80-column pass
// (eight warps let a thread hold 255 registers, nine only 168; that pass's
// consumers issue each warp's ten MMA chains together and need them).  Passes of up to 16 columns use 512-k stages and
// two activation warps, which read the stage's activation columns from L2,
// write them in MMA B-fragment order together with the block sums and hand the
// stage on.  The 80-column pass uses 256-k stages (a segment is two stages;
// only the delivery changes, not the arithmetic); its activations are packed
// into that same layout once per call by xpack_kernel (or beforehand by the
// kernel that produced them: spec_qmatmul_packed) and copied in with the
// stage by one cp.async.bulk.  Consumers issue only ldmatrix, 4 LOP3 + 3
// shifts per 8 weights, lds, mma.sync and the FADD/FFMA of each block partial.
// A tile covered by one CTA is folded in registers and written directly.  A
// tile shared by several CTAs: the CTAs holding its later segments store their segment sums and count themselves
// in, without waiting; the CTA holding the leading segments folds them in
// segment order once all have arrived (the usual case when it gets there),
// else leaves its prefix for whichever CTA arrives last.  No CTA waits for
// another; the counters end at zero, and consumed sums lying where a later
// call keeps its counters (the workspace's first 64 KB) are cleared.
//
// The weight format (int4 block 32, fp16 scale, even k in the low nibble) is
// the stand-in for the block-quantised formats named in ramgpt.org, "When
// Lossless Speculation Stops Being Lossless on Blackwell", section
// "Quantized Matrix Multiplication Shows the Same Class of Failure".
#include <mutex>

#include "qmm_shared.cuh"

namespace {
using namespace qmm;

constexpr int NCW = 8;                       // consumer warps (16 rows each)
// what a pass writes: fp32 (optionally added into y), bf16, or for a gate/up
// matrix whose rows come in groups of 8 gate rows and their 8 up rows, the
// bf16 SwiGLU of each feature (spec_qmatmul_swiglu)
constexpr int OUT_F32 = 0, OUT_BF16 = 1, OUT_SWIGLU = 2;
constexpr int W_BOX = BM * 128;              // one 128-row x 128-byte code box (256 k)
constexpr int MAX_NT = 10;                   // column tiles per pass (80 columns)

// Narrow passes (<= 16 columns) stream 512-k stages and prepare each stage's
// activations in the CTA (two activation warps).  The 80-column pass uses
// 256-k stages (its activations are 5x larger); its activations are prepared
// once per call by a small kernel (xpack_kernel) into the workspace, in the
// very byte layout of a stage, and each stage's part is copied in by TMA.
// The stage size only changes how a segment is delivered, never its arithmetic.

template <int NT, int FMT = SC_BLOCK>
struct Cfg {
    static constexpr int KS = NT >= 10 ? 256 : 512;         // k per stage
    static constexpr int NBLK = KS / 32;                    // 32-k blocks per stage
    static constexpr int NWBOX = KS / 256;                  // code boxes per stage
    static constexpr bool XPACK = NT >= 10;                 // activations pre-packed per call
    static constexpr int NXW = XPACK ? 0 : 2;               // activation warps
    // a TMA warp, except in the 80-column pass, where consumer warp 0 issues the
    // copies: with eight warps a thread may hold 255 registers, with nine 168
    static constexpr int NTMA = XPACK ? 0 : 1;
    static constexpr int THREADS = (NCW + NTMA + NXW) * 32;
    static constexpr int W_BYTES = NWBOX * W_BOX;
    // scales of a stage: fp16 per block, or the row's 16-byte record pair holding the stage
    static constexpr int S_BYTES = FMT == SC_BLOCK ? BM * NBLK * 2 : BM * 16;
    static constexpr int X_BOX = 8 * NT * 128;              // 64 k of the pass's activation columns
    static constexpr int X_BYTES = (NBLK / 2) * X_BOX;
    static constexpr int CI_BYTES = NBLK * 8 * NT * 4;      // [blocks][8 NT slots] fp32
    // stage layout: codes | scales | activations (B-fragment order) | -136 x block sums
    static constexpr int S_OFF = W_BYTES, X_OFF = W_BYTES + S_BYTES, CI_OFF = X_OFF + X_BYTES;
    static constexpr int XC_BYTES = X_BYTES + CI_BYTES;     // one stage of packed activations
    static constexpr int RAW = W_BYTES + X_BYTES + S_BYTES + CI_BYTES;
    static constexpr int STAGE = (RAW + 1023) / 1024 * 1024;
    static constexpr int NS = (SMEM_BUDGET / STAGE) > 6 ? 6 : (SMEM_BUDGET / STAGE);
    static constexpr int SMEM = 1024 + NS * STAGE + 3 * NS * 8 + 64;
    static_assert(NS >= 2, "at least two stages");
    static_assert(X_OFF % 128 == 0 && XC_BYTES % 16 == 0, "activation area alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
};

static_assert(Cfg<MAX_NT>::X_BYTES == SYNC_WIDE_X_BYTES && Cfg<MAX_NT>::XC_BYTES == WIDE_XC_BYTES &&
                  Cfg<MAX_NT>::KS == WIDE_KS && MAX_NT == SYNC_WIDE_NT,
              "the packed layout producers write (qmm_shared.cuh) is the 80-column pass's stage layout");

// 32-k blocks per stage of a pass with nt column tiles (the scale box width)
inline int stage_blocks(int nt) { return nt >= MAX_NT ? Cfg<MAX_NT>::NBLK : nt == 2 ? Cfg<2>::NBLK : Cfg<1>::NBLK; }


// nibble codes (k = 8t .. 8t+7 of a block) -> (128 + code_m, 128 + code_{m+4}), exact
__device__ __forceinline__ void codes_to_bf16(uint32_t w, uint32_t (&o)[4]) {
    o[0] = dev::lop3_and_or(w, 0x000F000Fu, 0x43004300u);
    o[1] = dev::lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u);
    o[2] = dev::lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u);
    o[3] = dev::lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u);
}

// Block j's scale from a super-block record (little-endian: s_j = bits 6j..6j+5,
// fp16 D = bits 48..63): D * s_j, exact in fp32 (11 + 6 significant bits).
__device__ __forceinline__ float super_scale(const uint2 &rec, int j) {
    const uint64_t w = ((uint64_t)rec.y << 32) | rec.x;
    const float D = __half2float(__ushort_as_half((unsigned short)(rec.y >> 16)));
    return D * (float)(uint32_t)((w >> (6 * j)) & 63u);
}

// The activations of one (32-k block, column) pair of a stage: four 16-byte
// chunks of k = kb .. kb + 31 of column col (zero past K or n_cols).
__device__ __forceinline__ void load_pair(uint4 (&v)[4], const uint16_t *__restrict__ x, int ldx, int K, int n_cols,
                                          int col, int kb) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = make_uint4(0, 0, 0, 0);
        if (col < n_cols && kb + 8 * q < K) v[q] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)col * ldx + kb + 8 * q));
    }
}

// Packs the activations of one pass (columns col0 .. col0 + 8 NT - 1) for every
// stage of K into out: stage st occupies out[st * XC_BYTES ...] in the byte
// layout of a stage's activation and block-sum areas.
template <int NT>
__global__ void __launch_bounds__(256) xpack_kernel(const uint16_t *__restrict__ x, int ldx, int K, int n_cols, int col0,
                                                    uint8_t *__restrict__ out, const int32_t *dev_cols, int min_cols) {
    using C = Cfg<NT>;
    dev::pdl_wait();   // x is the preceding kernel's output; out may still be read by it
    dev::pdl_launch_dependents();
    if (dev_cols) n_cols = gated_cols(n_cols, dev_cols, min_cols);
    if (col0 >= n_cols) return;
    constexpr int PAIRS = C::NBLK * 8 * NT;   // per stage
    const long long p = blockIdx.x * 256ll + threadIdx.x;
    const int st = (int)(p / PAIRS), pr = (int)(p % PAIRS);
    if (st * C::KS >= K) return;
    const int blk = pr / (8 * NT), c = pr % (8 * NT);
    uint4 v[4];
    load_pair(v, x, ldx, K, n_cols, col0 + c, st * C::KS + 32 * blk);
    uint8_t *base = out + (size_t)st * C::XC_BYTES;
    pack_pair<NT>(v, blk, c, base, reinterpret_cast<float *>(base + C::X_BYTES));
}

__device__ __forceinline__ void named_sync_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

template <int NT, int OUTM, int FMT>
__global__ void __launch_bounds__(Cfg<NT, FMT>::THREADS, 1)
qmm_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ts,
           const uint16_t *__restrict__ x, int ldx, int N, int K, int n_cols, int col0, void *__restrict__ y, int ldy,
           int accumulate, Sched sch, float *__restrict__ wsp_prefix, float *__restrict__ wsp_seg,
           int *__restrict__ counters, const uint8_t *__restrict__ xpk, int32_t *dev_err, const int32_t *dev_cols,
           int min_cols) {
    using C = Cfg<NT, FMT>;
    if (dev_cols) {
        // the column count is the preceding kernel's output: no early streaming
        dev::pdl_wait();
        n_cols = gated_cols(n_cols, dev_cols, min_cols);
    }
    if (col0 >= n_cols) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NS * C::STAGE);
    uint64_t *ready = full + C::NS;
    uint64_t *empty = ready + C::NS;
    int *flag = reinterpret_cast<int *>(empty + C::NS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nst_total = (K + C::KS - 1) / C::KS;   // stages of this pass's size
    const int seg_st = sch.seg_st, ks = sch.ks;       // stages per segment, segments
    const long long ua = sch.begin(blockIdx.x), ub = sch.begin(blockIdx.x + 1);
    constexpr int TILE_ELEMS = BM * 8 * NT;     // one tile's values for this pass
    // Partial sums in the workspace keep the accumulator fragments as the
    // consumer threads hold them: [fragment][warp][lane][4] floats, so every
    // store and load is a coalesced 16-byte access by the thread that owns it.
    const int frag = ((warp * 32 + (threadIdx.x & 31)) * 4);   // + f * NCW * 128

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            dev::mbar_init(&full[s], 1);
            dev::mbar_init(&ready[s], 1);
            dev::mbar_init(&empty[s], NCW);
        }
        dev::fence_barrier_init();
    }
    __syncthreads();
    // The weights and scales are constant inputs: the TMA warp starts streaming
    // them at once, overlapping the tail of the preceding kernel on the stream.
    // Activations are read, and anything global is written, only after that
    // kernel has finished (pdl_wait).
    dev::pdl_launch_dependents();

    // stage sequence of this CTA: units ua..ub-1, each 1 or 2 stages
    auto unit_stages = [&](long long u) { return min(seg_st, nst_total - (int)(u % ks) * seg_st); };

    if (!C::XPACK && warp == NCW) {
        // ============================ TMA warp ============================
        // lane 0 streams the codes (two 128-row x 128-byte boxes per 512-k stage)
        // and the scales of every stage of this CTA, NS stages ahead of the
        // consumers, reusing a slot once its consumers have released it.
        if (lane == 0) {
            dev::prefetch_tmap(&tw);
            dev::prefetch_tmap(&ts);
            long long iu = ua;
            int ist = 0;
            for (int issued = 0; iu < ub; ++issued) {
                const int s = issued % C::NS;
                if (issued >= C::NS && !dev::mbar_wait(&empty[s], ((issued / C::NS) - 1) & 1)) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    break;
                }
                const int tile = (int)(iu / ks) / sch.ncg;   // 128-row tile
                const int k0 = ((int)(iu % ks) * seg_st + ist) * C::KS;
                uint8_t *base = smem + s * C::STAGE;
                dev::mbar_arrive_expect_tx(&full[s], C::W_BYTES + C::S_BYTES);
#pragma unroll
                for (int b = 0; b < C::NWBOX; ++b)
                    dev::tma_load_2d(base + b * W_BOX, &tw, k0 / 2 + 128 * b, tile * BM, &full[s]);
                if constexpr (FMT == SC_BLOCK)
                    dev::tma_load_2d(base + C::S_OFF, &ts, k0 / 32, tile * BM, &full[s]);
                else   // the 16-byte record pair holding this stage's super-block(s)
                    dev::tma_load_2d(base + C::S_OFF, &ts, (k0 / 512) * 16, tile * BM, &full[s]);
                if (++ist == unit_stages(iu)) {
                    ist = 0;
                    ++iu;
                }
            }
        }
        return;
    }
    if constexpr (!C::XPACK) {
    if (warp > NCW) {
        // ======================== activation warps ========================
        // warp NCW + 1 + h prepares stages i with i % C::NXW == h: it reads the
        // stage's activation columns from L2 (all loads of a group in flight),
        // writes them in B-fragment order with their block sums, waits for the
        // stage's TMA bytes, then hands the stage to the consumers.
        const int h = warp - NCW - 1;
        dev::pdl_wait();   // x may be the preceding kernel's output
        bool ok = true;
        long long pu = ua;
        int pst = 0;
        for (int i = 0; pu < ub; ++i) {
            const int k0 = ((int)(pu % ks) * seg_st + pst) * C::KS;
            const int cb = col0 + (int)((pu / ks) % sch.ncg) * 8 * NT;   // the unit's column group
            if (++pst == unit_stages(pu)) {
                pst = 0;
                ++pu;
            }
            if (i % C::NXW != h) continue;
            const int s = i % C::NS;
            bool slot_free = (i < C::NS);   // the slot's previous stage must be released before writing
            uint8_t *xs = smem + s * C::STAGE + C::X_OFF;
            float *ci = reinterpret_cast<float *>(smem + s * C::STAGE + C::CI_OFF);
            // (block, column) pairs p = lane + 32 j
            constexpr int PAIRS = C::NBLK * 8 * NT / 32;   // per lane
            constexpr int GROUP = 4;                  // pairs whose loads are in flight together
#pragma unroll 1
            for (int j0 = 0; j0 < PAIRS; j0 += GROUP) {
                uint4 v[GROUP][4];
#pragma unroll
                for (int jj = 0; jj < GROUP; ++jj) {
                    const int p = lane + 32 * (j0 + jj);
                    const int blk = p / (8 * NT), c = p % (8 * NT);
                    load_pair(v[jj], x, ldx, K, n_cols, cb + c, k0 + 32 * blk);
                }
                if (!slot_free) {   // loads are in flight; now wait for the consumers' release
                    int got = 1;
                    if (lane == 0 && ok) got = dev::mbar_wait(&empty[s], ((i / C::NS) - 1) & 1) ? 1 : 0;
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got && ok) {
                        if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                        ok = false;
                    }
                    slot_free = true;
                }
#pragma unroll
                for (int jj = 0; jj < GROUP; ++jj) {
                    const int p = lane + 32 * (j0 + jj);
                    pack_pair<NT>(v[jj], p / (8 * NT), p % (8 * NT), xs, ci);
                }
            }
            int got = 1;
            if (lane == 0 && ok) got = dev::mbar_wait(&full[s], (i / C::NS) & 1) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got && ok) {
                if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                ok = false;
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&ready[s]);
        }
        return;
    }
    }

    // ============================ consumers ============================
    // The 80-column pass: lane 0 of warp 0 issues the copies.  It sends the
    // first NS stages' codes and scales at once (constant inputs), their packed
    // activations once the preceding kernel has finished, and, at the start of
    // each later stage i, stage i - 1 + NS into the slot that stage i - 1 has
    // released.  The cursor is kept by every lane of warp 0, so that its
    // decisions are warp-uniform.
    int my_stages = 0, issued = 0;
    long long p_iu = ua;
    int p_ist = 0;
    int k0s[C::NS];   // the first stages, whose activations are copied after pdl_wait
    auto issue_stage = [&](bool with_x) {
        const int s = issued % C::NS;
        const int k0 = ((int)(p_iu % ks) * seg_st + p_ist) * C::KS;
        if (lane == 0) {
            const int tile = (int)(p_iu / ks) / sch.ncg;
            uint8_t *base = smem + s * C::STAGE;
            dev::mbar_arrive_expect_tx(&full[s], C::W_BYTES + C::S_BYTES + C::XC_BYTES);
#pragma unroll
            for (int b = 0; b < C::NWBOX; ++b)
                dev::tma_load_2d(base + b * W_BOX, &tw, k0 / 2 + 128 * b, tile * BM, &full[s]);
            if constexpr (FMT == SC_BLOCK)
                dev::tma_load_2d(base + C::S_OFF, &ts, k0 / 32, tile * BM, &full[s]);
            else
                dev::tma_load_2d(base + C::S_OFF, &ts, (k0 / 512) * 16, tile * BM, &full[s]);
            if (with_x)
                dev::bulk_load(base + C::X_OFF, xpk + (size_t)(k0 / C::KS) * C::XC_BYTES, C::XC_BYTES, &full[s]);
        }
        if (!with_x) k0s[issued] = k0;
        if (++p_ist == unit_stages(p_iu)) {
            p_ist = 0;
            ++p_iu;
        }
        ++issued;
    };
    if constexpr (C::XPACK) {
        for (long long uu = ua; uu < ub; ++uu) my_stages += unit_stages(uu);
        if (warp == 0) {
            if (lane == 0) {
                dev::prefetch_tmap(&tw);
                dev::prefetch_tmap(&ts);
            }
            while (issued < my_stages && issued < C::NS) issue_stage(false);
        }
    }
    dev::pdl_wait();   // y (accumulate), the workspace, y writes and the packed activations follow the preceding kernel
    if constexpr (C::XPACK) {
        if (warp == 0 && lane == 0)
            for (int j = 0; j < issued; ++j)
                dev::bulk_load(smem + j * C::STAGE + C::X_OFF, xpk + (size_t)(k0s[j] / C::KS) * C::XC_BYTES,
                               C::XC_BYTES, &full[j]);
    }
    const int r = lane >> 2, t = lane & 3;
    // A consumer warp owns RG 16-row groups x CT 8-column tiles (RG x CT = NT
    // fragments f = rg * CT + ctl).  Narrow passes: one row group, all columns.
    // The 80-column pass: 32 rows x 40 columns per warp, so that each activation
    // fragment read from shared memory feeds two row groups' MMAs (with 16 rows
    // x 80 columns the eight warps read 40 KB of activations per 32-k block).
    // Which warp computes a fragment is scheduling: its operations are the same.
    constexpr int RG = NT >= 10 ? 2 : 1;
    constexpr int CT = NT / RG;
    constexpr int RSLOTS = NCW / (NT >= 10 ? 2 : 1);   // warps along the rows
    static_assert(RG * CT == NT && RSLOTS * 16 * RG == BM, "consumer mapping");
    const int wrow0 = (warp % RSLOTS) * 16 * RG;         // row group rg starts at wrow0 + 16 rg
    const int ctb = (warp / RSLOTS) * CT;                 // first column tile of this warp
    int colb = col0;   // first column of the current tile's column group
    auto fcol = [&](int f) { return colb + (ctb + f % CT) * 8; };   // first column of fragment f
    const int g = lane >> 2;
    const int xcol = (g & 1) * 4 + (g >> 1);   // activation column of this lane's B fragment
    float yrun[NT][4];
    int i = 0;
    bool ok = true;
    long long u = ua;
    int nh_tile = -1, nh_prev = 0, nh_touch = 0;   // thread 0: this CTA's later-segment part, if any

    // y for this thread's fragments of `tile` from yrun
    auto store_tile = [&](int tile) {
        if constexpr (OUTM == OUT_SWIGLU) {
            // a fragment's rows r and r + 8 of its 16-row group are a feature's gate
            // and up rows: write that feature's SwiGLU for the fragment's two columns
#pragma unroll
            for (int f = 0; f < NT; ++f) {
                const int c8 = (ctb + f % CT) * 8, wr = wrow0 + 16 * (f / CT);
                const int n = (tile / sch.ncg) * BM + wr + r;   // the gate row
                if (n < N) {
                    const int feat = (n >> 4) * 8 + (n & 7);
                    const int c0 = colb + c8 + t, c1 = c0 + 4;
                    uint16_t *act = reinterpret_cast<uint16_t *>(y);
                    if (c0 < n_cols) act[(size_t)c0 * ldy + feat] = dev::swiglu_bf16(yrun[f][0], yrun[f][2]);
                    if (c1 < n_cols) act[(size_t)c1 * ldy + feat] = dev::swiglu_bf16(yrun[f][1], yrun[f][3]);
                }
            }
            return;
        }
        auto store_y = [&](int c, int row, float v) {
            const int col = colb + c, n = (tile / sch.ncg) * BM + row;
            if (col < n_cols && n < N) {
                if (OUTM == OUT_BF16) {
                    reinterpret_cast<__nv_bfloat16 *>(y)[(size_t)col * ldy + n] = __float2bfloat16_rn(v);
                } else {
                    float *yp = reinterpret_cast<float *>(y) + (size_t)col * ldy + n;
                    *yp = accumulate ? (*yp + v) : v;
                }
            }
        };
#pragma unroll
        for (int f = 0; f < NT; ++f) {
            const int c8 = (ctb + f % CT) * 8, wr = wrow0 + 16 * (f / CT);
            store_y(c8 + t, wr + r, yrun[f][0]);
            store_y(c8 + t + 4, wr + r, yrun[f][1]);
            store_y(c8 + t, wr + r + 8, yrun[f][2]);
            store_y(c8 + t + 4, wr + r + 8, yrun[f][3]);
        }
    };
    // yrun holds the fold of segments 0 .. seg_from-1 of `tile`: add the stored
    // sums of segments seg_from .. ks-1 in ascending order, write y and reset the
    // tile's counter.  Each stored sum is zeroed once read, so the partial-sum
    // area is left zero-filled: a later call whose counters lie where this call
    // kept sums (it has more tiles) finds them at zero.
    // zero a stored float4 of the workspace if it lies where a call's counters may be
    auto clear_low = [&](float *p, bool used) {
        if (used && (size_t)(reinterpret_cast<const uint8_t *>(p) - reinterpret_cast<const uint8_t *>(counters)) <
                        CNT_LIMIT)
            __stcg(reinterpret_cast<float4 *>(p), make_float4(0.f, 0.f, 0.f, 0.f));
    };
    auto fold_tile = [&](int tile, int seg_from) {
        float *p0 = wsp_seg + (size_t)tile * ks * TILE_ELEMS + frag;
        // segments whose loads are in flight together (a short last group is
        // predicated: no load and no add past the last segment)
        constexpr int SG = NT >= 8 ? 3 : (NT >= 2 ? 8 : 16);
        for (int sg = seg_from; sg < ks; sg += SG) {
            float4 l[SG][NT];
#pragma unroll
            for (int q = 0; q < SG; ++q)
#pragma unroll
                for (int ct = 0; ct < NT; ++ct)
                    l[q][ct] = (sg + q < ks && fcol(ct) < n_cols)
                                   ? __ldcg(reinterpret_cast<const float4 *>(p0 + (size_t)(sg + q) * TILE_ELEMS +
                                                                             ct * NCW * 128))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < SG; ++q)
                if (sg + q < ks) {
#pragma unroll
                    for (int ct = 0; ct < NT; ++ct) {
                        yrun[ct][0] += l[q][ct].x;
                        yrun[ct][1] += l[q][ct].y;
                        yrun[ct][2] += l[q][ct].z;
                        yrun[ct][3] += l[q][ct].w;
                    }
                }
        }
        store_tile(tile);
        if (threadIdx.x == 0) counters[tile] = 0;
        // every sum is read: clear those a later call could take for counters
        // (after all loads, so none waits behind these stores)
        for (int sg = seg_from; sg < ks; ++sg)
#pragma unroll
            for (int ct = 0; ct < NT; ++ct)
                clear_low(p0 + (size_t)sg * TILE_ELEMS + ct * NCW * 128, fcol(ct) < n_cols);
    };

    while (u < ub) {
        const int tile = (int)(u / ks);
        colb = col0 + (tile % sch.ncg) * 8 * NT;
        const long long tile_u0 = (long long)tile * ks;
        const long long u_end = min(ub, tile_u0 + ks);     // this CTA's units of this tile
        const bool head = (u == tile_u0);
        const bool whole = head && (u_end == tile_u0 + ks);
#pragma unroll
        for (int ct = 0; ct < NT; ++ct) yrun[ct][0] = yrun[ct][1] = yrun[ct][2] = yrun[ct][3] = 0.f;
        for (; u < u_end; ++u) {
            const int seg = (int)(u - tile_u0);
            const int nstg = unit_stages(u);
            float acc[NT][4];
#pragma unroll
            for (int ct = 0; ct < NT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
            for (int st = 0; st < nstg; ++st, ++i) {
                const int s = i % C::NS;
                if constexpr (C::XPACK) {
                    // stage i - 1 + NS into the slot of stage i - 1, once every consumer warp released it
                    if (warp == 0 && i >= 1 && issued < my_stages && ok) {
                        int got = 1;
                        if (lane == 0) got = dev::mbar_wait(&empty[issued % C::NS], ((issued / C::NS) - 1) & 1) ? 1 : 0;
                        got = __shfl_sync(0xffffffffu, got, 0);
                        if (got) {
                            issue_stage(true);
                        } else {
                            if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                            ok = false;
                        }
                    }
                }
                if (ok && !dev::mbar_wait(C::XPACK ? &full[s] : &ready[s], (i / C::NS) & 1)) {
                    dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    ok = false;
                }
                const uint32_t wbase = dev::smem_u32(smem + s * C::STAGE);
                const uint32_t xbase = wbase + C::X_OFF;
                const uint32_t sbase = wbase + C::S_OFF;
                const uint32_t cbase = wbase + C::CI_OFF;
                // super-block scales: rows r and r+8's record pair of this stage, per row group
                // (a 512-k stage uses both records, a 256-k stage the one its k offset selects)
                uint2 rec_r[RG][2] = {}, rec_r8[RG][2] = {};
                int rsel = 0;
                if constexpr (FMT == SC_SUPER) {
#pragma unroll
                    for (int rg = 0; rg < RG; ++rg) {
                        const uint2 *pr = reinterpret_cast<const uint2 *>(smem + s * C::STAGE + C::S_OFF +
                                                                          (wrow0 + 16 * rg + r) * 16);
                        const uint2 *pr8 = pr + 16;   // 8 rows further on
                        rec_r[rg][0] = pr[0], rec_r[rg][1] = pr[1], rec_r8[rg][0] = pr8[0], rec_r8[rg][1] = pr8[1];
                    }
                    rsel = ((((int)(u % ks) * seg_st + st) * C::KS) >> 8) & 1;
                }
                constexpr int BP_UNROLL = NT > 4 ? 1 : C::NBLK / 2;
#pragma unroll BP_UNROLL
                for (int bp = 0; bp < C::NBLK / 2; ++bp) {
                    uint32_t wv[RG][4];
                    uint32_t s2[RG] = {}, s28[RG] = {};   // fp16 scales of blocks 2bp, 2bp+1 for rows r and r+8
#pragma unroll
                    for (int rg = 0; rg < RG; ++rg) {
                        const int wr = wrow0 + 16 * rg;
                        {
                            // blocks 2bp, 2bp+1: box bp/4 (256 k each), 16-byte chunk (2bp + m/2) % 8
                            const int m = lane >> 3, rr = lane & 7;
                            const int row = wr + (m & 1) * 8 + rr;
                            const int blk = 2 * bp + (m >> 1);
                            dev::ldmatrix_x4(wv[rg][0], wv[rg][1], wv[rg][2], wv[rg][3],
                                             wbase + (blk >> 3) * W_BOX + row * 128 + (((blk & 7) ^ (row & 7)) << 4));
                        }
                        if constexpr (FMT == SC_BLOCK) {
                            asm volatile("ld.shared.u32 %0, [%1];"
                                         : "=r"(s2[rg])
                                         : "r"(sbase + (wr + r) * (2 * C::NBLK) + bp * 4));
                            asm volatile("ld.shared.u32 %0, [%1];"
                                         : "=r"(s28[rg])
                                         : "r"(sbase + (wr + r + 8) * (2 * C::NBLK) + bp * 4));
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int blk = 2 * bp + h;
                        uint32_t ar[RG][4], ar8[RG][4];
                        float d_r[RG], d_r8[RG];
#pragma unroll
                        for (int rg = 0; rg < RG; ++rg) {
                            codes_to_bf16(wv[rg][2 * h], ar[rg]);
                            codes_to_bf16(wv[rg][2 * h + 1], ar8[rg]);
                            if constexpr (FMT == SC_BLOCK) {
                                d_r[rg] = __half2float(__ushort_as_half((unsigned short)(s2[rg] >> (16 * h))));
                                d_r8[rg] = __half2float(__ushort_as_half((unsigned short)(s28[rg] >> (16 * h))));
                            } else {
                                const int pi = C::KS == 512 ? (bp >> 2) : rsel;
                                d_r[rg] = super_scale(pi ? rec_r[rg][1] : rec_r[rg][0], blk & 7);
                                d_r8[rg] = super_scale(pi ? rec_r8[rg][1] : rec_r8[rg][0], blk & 7);
                            }
                        }
                        if constexpr (NT >= MAX_NT) {
                            // The 80-column pass: the ten chains of this warp (RG row groups x
                            // CT column tiles) are issued together -- all first products, then
                            // all second products, then the fmas -- so that no MMA waits on
                            // the one just issued.  Every chain and every accumulator's
                            // sequence of operations is the same as one chain at a time.
                            uint32_t bq[CT][4];
                            float cq[CT][2];
#pragma unroll
                            for (int ctl = 0; ctl < CT; ++ctl) {
                                const int ct = ctb + ctl;
                                const int xrow = ct * 8 + xcol;
                                const int chunk = ((blk & 1) * 4 + t) ^ (xrow & 7);
                                dev::lds128(bq[ctl][0], bq[ctl][1], bq[ctl][2], bq[ctl][3],
                                            xbase + (blk >> 1) * C::X_BOX + xrow * 128 + (chunk << 4));
                                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                                             : "=f"(cq[ctl][0]), "=f"(cq[ctl][1])
                                             : "r"(cbase + (blk * 8 * NT + ct * 8 + 2 * t) * 4));
                            }
                            const float zero[4] = {0.f, 0.f, 0.f, 0.f};
                            float pp[CT][RG][4];
#pragma unroll
                            for (int ctl = 0; ctl < CT; ++ctl)
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg)
                                    dev::mma_bf16(pp[ctl][rg], ar[rg][0], ar8[rg][0], ar[rg][1], ar8[rg][1], bq[ctl][0],
                                                  bq[ctl][1], zero);
#pragma unroll
                            for (int ctl = 0; ctl < CT; ++ctl)
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg)
                                    dev::mma_bf16(pp[ctl][rg], ar[rg][2], ar8[rg][2], ar[rg][3], ar8[rg][3], bq[ctl][2],
                                                  bq[ctl][3], pp[ctl][rg]);
#pragma unroll
                            for (int ctl = 0; ctl < CT; ++ctl)
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg) {
                                    float(&a4)[4] = acc[rg * CT + ctl];
                                    dev::fma_add_f32x2(a4[0], a4[1], d_r[rg], pp[ctl][rg][0], pp[ctl][rg][1],
                                                       cq[ctl][0], cq[ctl][1]);
                                    dev::fma_add_f32x2(a4[2], a4[3], d_r8[rg], pp[ctl][rg][2], pp[ctl][rg][3],
                                                       cq[ctl][0], cq[ctl][1]);
                                }
                        } else {
#pragma unroll
                        for (int ctl = 0; ctl < CT; ++ctl) {
                            const int ct = ctb + ctl;   // column tile of the pass
                            const int xrow = ct * 8 + xcol;
                            const int chunk = ((blk & 1) * 4 + t) ^ (xrow & 7);
                            uint32_t b00, b01, b10, b11;
                            dev::lds128(b00, b01, b10, b11, xbase + (blk >> 1) * C::X_BOX + xrow * 128 + (chunk << 4));
                            float c0, c1;
                            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                                         : "=f"(c0), "=f"(c1)
                                         : "r"(cbase + (blk * 8 * NT + ct * 8 + 2 * t) * 4));
                            const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int rg = 0; rg < RG; ++rg) {
                                float p[4];
                                dev::mma_bf16(p, ar[rg][0], ar8[rg][0], ar[rg][1], ar8[rg][1], b00, b01, zero);
                                dev::mma_bf16(p, ar[rg][2], ar8[rg][2], ar[rg][3], ar8[rg][3], b10, b11, p);
                                float(&a4)[4] = acc[rg * CT + ctl];
                                dev::fma_add_f32x2(a4[0], a4[1], d_r[rg], p[0], p[1], c0, c1);
                                dev::fma_add_f32x2(a4[2], a4[3], d_r8[rg], p[2], p[3], c0, c1);
                            }
                        }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&empty[s]);
            }
            if (head) {
                // this CTA holds the tile's leading segments: fold them in order
#pragma unroll
                for (int ct = 0; ct < NT; ++ct)
#pragma unroll
                    for (int e = 0; e < 4; ++e) yrun[ct][e] = (seg == 0) ? acc[ct][e] : yrun[ct][e] + acc[ct][e];
            } else {
                // a later CTA's segment: store its sum for the final fold
                float *ps = wsp_seg + ((size_t)tile * ks + seg) * TILE_ELEMS + frag;
#pragma unroll
                for (int ct = 0; ct < NT; ++ct)
                    if (fcol(ct) < n_cols)
                        __stcg(reinterpret_cast<float4 *>(ps + ct * NCW * 128),
                               make_float4(acc[ct][0], acc[ct][1], acc[ct][2], acc[ct][3]));
            }
        }
        // ---------------- finish this CTA's part of the tile ----------------
        if (whole) {
            store_tile(tile);
            continue;
        }
        const int touch = sch.cta_of(tile_u0 + ks - 1) - sch.cta_of(tile_u0) + 1;   // CTAs sharing the tile
        if (!head) {
            // Later segments of a shared tile: publish their sums and move on.  Whether
            // this CTA was the last to arrive is looked at only after all its units.
            named_sync_consumers();             // all partial stores of this CTA are issued
            if (threadIdx.x == 0) {
                __threadfence();                // ... and visible device-wide before the counter moves
                nh_prev = atomicAdd(&counters[tile], 1);
                nh_tile = tile;
                nh_touch = touch;
            }
            continue;
        }
        // Leading segments of a shared tile (the end of this CTA's range).  Usually
        // every other CTA has arrived long ago: then fold at once from registers.
        if (threadIdx.x == 0) {
            int seen;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(counters + tile) : "memory");
            flag[0] = (seen == touch - 1) ? 1 : 0;
        }
        named_sync_consumers();
        int fold_now = flag[0];
        if (!fold_now) {
            // not yet: leave the prefix for whichever CTA arrives last
            float *pp = wsp_prefix + (size_t)tile * TILE_ELEMS + frag;
#pragma unroll
            for (int ct = 0; ct < NT; ++ct)
                if (fcol(ct) < n_cols)
                    __stcg(reinterpret_cast<float4 *>(pp + ct * NCW * 128),
                           make_float4(yrun[ct][0], yrun[ct][1], yrun[ct][2], yrun[ct][3]));
            named_sync_consumers();             // prefix stores issued; flag[0] read by all
            if (threadIdx.x == 0) {
                __threadfence();
                const int prev = atomicAdd(&counters[tile], 1);
                if (prev == touch - 1) __threadfence();
                flag[0] = (prev == touch - 1) ? 1 : 0;
            }
            named_sync_consumers();
            fold_now = flag[0];
            if (fold_now) {
                // this part arrived last after all: fold, then clear the prefix it left
                const long long head_end = min(sch.begin(blockIdx.x + 1), tile_u0 + ks);
                fold_tile(tile, (int)(head_end - tile_u0));
#pragma unroll
                for (int ct = 0; ct < NT; ++ct) clear_low(pp + ct * NCW * 128, fcol(ct) < n_cols);
                fold_now = 0;
            }
        }
        if (fold_now) {
            const long long head_end = min(sch.begin(blockIdx.x + 1), tile_u0 + ks);
            fold_tile(tile, (int)(head_end - tile_u0));
        }
        named_sync_consumers();   // flag[0] is read by everyone before it is reused
    }

    // A later-segment part that turned out to arrive last folds its tile now,
    // the prefix and every segment sum coming from the workspace.
    if (threadIdx.x == 0) {
        flag[0] = (nh_tile >= 0 && nh_prev == nh_touch - 1) ? 1 : 0;
        flag[1] = nh_tile;
        if (flag[0]) __threadfence();
    }
    named_sync_consumers();
    if (flag[0]) {
        const int tile = flag[1];
        colb = col0 + (tile % sch.ncg) * 8 * NT;
        const long long tile_u0 = (long long)tile * ks;
        const int head_cta = sch.cta_of(tile_u0);
        const long long head_end = min(sch.begin(head_cta + 1), tile_u0 + ks);
        float *pp = wsp_prefix + (size_t)tile * TILE_ELEMS + frag;
#pragma unroll
        for (int ct = 0; ct < NT; ++ct) {
            if (fcol(ct) < n_cols) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(pp + ct * NCW * 128));
                yrun[ct][0] = v.x, yrun[ct][1] = v.y, yrun[ct][2] = v.z, yrun[ct][3] = v.w;
            }
        }
        fold_tile(tile, (int)(head_end - tile_u0));
#pragma unroll
        for (int ct = 0; ct < NT; ++ct) clear_low(pp + ct * NCW * 128, fcol(ct) < n_cols);
    }
    if constexpr (C::XPACK) {
        // after a timeout some issued stages may not have been waited for: their
        // copies land before the CTA exits (bounded; at once otherwise)
        if (warp == 0 && lane == 0)
            for (int j = (issued > C::NS ? issued - C::NS : 0); j < issued; ++j)
                if (!dev::mbar_wait(&full[j % C::NS], (j / C::NS) & 1)) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
    }
}

// seg512: segment length in units of 512 k (1 for the invariant entry points)
template <int NT, int OUTM, int FMT>
spec_status launch_nt(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int ldx, int N, int K,
                      int n_cols, int col0, void *y, int ldy, int accumulate, int seg512, void *workspace,
                      int32_t *dev_err, const int32_t *dev_cols, int min_cols, cudaStream_t stream,
                      const uint8_t *xpk_in = nullptr, int ncg = 1) {
    using C = Cfg<NT, FMT>;
    auto kern = qmm_kernel<NT, OUTM, FMT>;
    static spec::SmemOptIn opt_in;
    spec_status so = spec::smem_opt_in(kern, C::SMEM, opt_in, "cudaFuncSetAttribute(qmm smem)");
    if (so != SPEC_OK) return so;
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    const Sched sch = make_sched(N, K, seg512, C::KS, sms, C::XPACK ? 1 : ncg);
    const WsLayout wl = ws_layout(workspace, sch.tiles, sch.ks, BM * 8 * NT);
    int *counters = wl.counters;
    float *prefix = wl.prefix, *segs = wl.segs;
    const uint8_t *xpk = xpk_in ? xpk_in : wl.xpk;
    if (C::XPACK && !xpk_in) {
        // this pass's activations, packed once for every CTA (into the workspace after the partial sums)
        const long long pairs = (long long)(K / C::KS) * C::NBLK * 8 * NT;
        cudaError_t e = spec::launch_pdl(xpack_kernel<NT>, dim3((unsigned)((pairs + 255) / 256)), dim3(256), 0, stream,
                                         x, ldx, K, n_cols, col0, const_cast<uint8_t *>(xpk), dev_cols, min_cols);
        if (e != cudaSuccess) return spec::cuda_status(e, "qmm activation pack launch");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sch.G);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, accumulate, sch, prefix,
                                       segs, counters, xpk, dev_err, dev_cols, min_cols);
    return spec::cuda_status(e, "qmm launch");
}

// Which kernel runs the 80-column pass (both give the same bits).
constexpr int WIDE_AUTO = 0, WIDE_TC = 1, WIDE_MMA_SYNC = 2;

int pass_nt(int n_cols) { return n_cols <= 8 ? 1 : (n_cols <= 16 ? 2 : MAX_NT); }

// workspace of one launch of nt column tiles per column group, ncg column groups
size_t ws_bytes_launch(int N, int K, int nt, int ncg, int seg512) {
    const size_t tiles = (size_t)(N + BM - 1) / BM * ncg;
    const size_t cnt = ((tiles * sizeof(int)) + 255) & ~size_t(255);
    // the 80-column pass also keeps its packed activations: K / 256 stages of XC_BYTES
    const size_t packed = nt >= MAX_NT ? (size_t)(K / Cfg<MAX_NT>::KS) * Cfg<MAX_NT>::XC_BYTES : 0;
    return cnt + tiles * (1 + (size_t)n_segments(K, seg512 * SEG_K)) * BM * 8 * nt * sizeof(float) + packed;
}

// Column groups of one 16-column-pass launch that covers up to 80 columns.
constexpr int MAX_NCG = MAX_NT / 2;

size_t ws_bytes_for(int N, int K, int nt, int seg512) { return ws_bytes_launch(N, K, nt, 1, seg512); }

// The passes of a call: nt column tiles per pass, ncg column groups per launch.
// Every plan gives the same bits -- a column's arithmetic does not depend on the
// pass that computes it -- so the plan decides only the time.
struct Plan {
    int nt, ncg;
};

// Estimated time (us) of a call planned as `p`: per launch a fixed cost plus,
// for the CTA with the most units, its units x the time of one unit (512 k x
// 128 rows of one column group).  Least-squares fit on GB300 over ten shapes
// from 1024 x 4096 to 32000 x 2048 at 32 to 80 columns; the 80-column pass
// also packs its activations in a launch of its own unless the caller's
// producer did.
double plan_cost(int N, int K, int n_cols, Plan p, bool packed_input) {
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    const int per_launch = 8 * p.nt * (p.nt < MAX_NT ? p.ncg : 1);
    const int launches = (n_cols + per_launch - 1) / per_launch;
    const Sched sch = make_sched(N, K, 1, p.nt >= MAX_NT ? Cfg<MAX_NT>::KS : Cfg<1>::KS, sms, p.ncg);
    const long long busiest = (sch.U + sch.G - 1) / sch.G;
    double fixed, unit;
    if (p.nt >= MAX_NT)
        fixed = 6.9 + (packed_input ? 0.0 : 6.0), unit = 6.11;
    else if (p.nt == 2)
        fixed = 6.3, unit = 2.07;
    else
        fixed = 5.4, unit = 1.36;
    return launches * (fixed + busiest * unit);
}

// Up to 8 columns: one 8-column pass; up to 16: one 16-column pass.  Up to
// 80: the cheapest of the 80-column pass and one launch of 16- or 8-column
// groups.  More: 80-column passes.
Plan choose_plan(int N, int K, int n_cols, bool packed_input) {
    if (n_cols <= 8) return {1, 1};
    if (n_cols <= 16) return {2, 1};
    if (n_cols > WIDE_COLS) return {MAX_NT, 1};
    const size_t tiles = (size_t)(N + BM - 1) / BM;
    Plan best = {2, 1};
    double best_t = 1e30;
    const Plan cands[3] = {{MAX_NT, 1}, {2, (n_cols + 15) / 16}, {1, (n_cols + 7) / 8}};
    for (const Plan &p : cands) {
        if (tiles * p.ncg * sizeof(int) > CNT_LIMIT) continue;
        const double t = plan_cost(N, K, n_cols, p, packed_input);
        if (t < best_t) best = p, best_t = t;
    }
    return best;
}

// Workspace for every plan a call of n_cols columns may take.
size_t ws_bytes_cols(int N, int K, int n_cols) {
    size_t need = ws_bytes_for(N, K, pass_nt(n_cols), 1);
    if (n_cols > 16 && n_cols <= WIDE_COLS) {
        const size_t g16 = ws_bytes_launch(N, K, 2, (n_cols + 15) / 16, 1);
        const size_t g8 = ws_bytes_launch(N, K, 1, (n_cols + 7) / 8, 1);
        need = need > g16 ? need : g16;
        need = need > g8 ? need : g8;
    }
    return need;
}

// bytes of super-block scale records per weight row
inline int super_pitch(int K) { return (K + 511) / 512 * 16; }

// One launch of a pass with output mode outm (SwiGLU with block scales only).
template <int NT, int FMT>
spec_status launch_mode(int outm, const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int ldx, int N,
                        int K, int n_cols, int col0, void *y, int ldy, int accumulate, int seg512, void *workspace,
                        int32_t *dev_err, const int32_t *dev_cols, int min_cols, cudaStream_t stream,
                        const uint8_t *xpk_in, int ncg) {
    if (outm == OUT_SWIGLU) {
        if constexpr (FMT == SC_BLOCK)
            return launch_nt<NT, OUT_SWIGLU, FMT>(tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, 0, seg512, workspace,
                                                  dev_err, dev_cols, min_cols, stream, xpk_in, ncg);
        return spec::fail(SPEC_ERR_UNSUPPORTED, "qmatmul: the SwiGLU output needs block scales");
    }
    if (outm == OUT_BF16)
        return launch_nt<NT, OUT_BF16, FMT>(tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, 0, seg512, workspace, dev_err,
                                            dev_cols, min_cols, stream, xpk_in, ncg);
    return launch_nt<NT, OUT_F32, FMT>(tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, accumulate, seg512, workspace,
                                       dev_err, dev_cols, min_cols, stream, xpk_in, ncg);
}

// swiglu: y is the bf16 SwiGLU of a gate/up matrix of N = 2F interleaved rows
// (8 gate rows, then their 8 up rows), [n_cols][ldy] with ldy >= F.
spec_status qmm_run(const uint8_t *wq, const void *ws, int N, int K, const uint16_t *x, int n_cols, int ldx,
                    void *y, spec_dtype y_dt, int ldy, int accumulate, int seg512, int nt, void *workspace,
                    int32_t *dev_err, cudaStream_t stream, int fmt = SC_BLOCK, const int32_t *dev_cols = nullptr,
                    int min_cols = 0, int wide = WIDE_AUTO, const uint8_t *xpk_in = nullptr, int ncg = 1,
                    bool swiglu = false) {
    CUtensorMap tw, ts;
    {
        uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)K / 2};
        uint32_t box[2] = {128, BM};
        if (!spec::encode_tiled(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, wq, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return SPEC_ERR_CUDA;
    }
    if (fmt == SC_BLOCK) {
        uint64_t dims[2] = {(uint64_t)K / 32, (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)K / 32 * 2};
        uint32_t box[2] = {(uint32_t)stage_blocks(nt), BM};
        if (!spec::encode_tiled(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, ws, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return SPEC_ERR_CUDA;
    } else {
        // one 16-byte record pair per row and stage
        uint64_t dims[2] = {(uint64_t)super_pitch(K), (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)super_pitch(K)};
        uint32_t box[2] = {16, BM};
        if (!spec::encode_tiled(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ws, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return SPEC_ERR_CUDA;
    }
    const bool bf = (y_dt == SPEC_BF16);
    const int outm = swiglu ? OUT_SWIGLU : (bf ? OUT_BF16 : OUT_F32);
    // column groups only while their arrival counters fit where counters may lie
    if ((size_t)((N + BM - 1) / BM) * ncg * sizeof(int) > CNT_LIMIT) ncg = 1;
    // One pass per group of 8 nt columns; passes run back to back on the stream.
    // With ncg > 1 (narrow passes only), one launch covers ncg such groups.
    const int step = 8 * nt * (nt < MAX_NT ? ncg : 1);
    for (int col0 = 0; col0 < n_cols; col0 += step) {
        spec_status st;
        const int g = nt < MAX_NT ? min(ncg, (n_cols - col0 + 8 * nt - 1) / (8 * nt)) : 1;
#define SPEC_QMM_FMT(NTV, FMTV)                                                                                    \
    st = launch_mode<NTV, FMTV>(outm, tw, ts, x, ldx, N, K, n_cols, col0, y, ldy, accumulate, seg512, workspace,     \
                                dev_err, dev_cols, min_cols, stream, xpk_in, g)
#define SPEC_QMM_CASE(NTV)                                                                                         \
    if (fmt == SC_BLOCK) {                                                                                         \
        SPEC_QMM_FMT(NTV, SC_BLOCK);                                                                              \
    } else {                                                                                                       \
        SPEC_QMM_FMT(NTV, SC_SUPER);                                                                              \
    }
        switch (nt) {
        case 1: SPEC_QMM_CASE(1); break;
        case 2: SPEC_QMM_CASE(2); break;
        default:
            // the 80-column pass: the mma.sync kernel unless the tcgen05 kernel is asked for.
            // Both give the same bits; the tcgen05 kernel measured slower on every matrix of
            // the decoder (its per-block accumulator round trip through tensor memory, with
            // four accumulators in flight, sets its block rate), so it is not chosen by default.
            if (fmt == SC_BLOCK && wide == WIDE_TC && !swiglu)
                st = tc_wide_pass(tw, ts, x, ldx, N, K, n_cols, col0, y, bf, ldy, accumulate, seg512, workspace,
                                  dev_err, dev_cols, min_cols, stream);
            else
                SPEC_QMM_CASE(MAX_NT);
        }
#undef SPEC_QMM_CASE
#undef SPEC_QMM_FMT
        if (st != SPEC_OK) return st;
    }
    return SPEC_OK;
}

spec_status check_args(const uint8_t *wq, const void *ws, int N, int K, const uint16_t *x, int n_cols, int ldx,
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
    SPEC_CHECK_ARG((size_t)(N + BM - 1) / BM * sizeof(int) <= CNT_LIMIT, "qmatmul: N must be <= %d (N=%d)",
                   (int)(CNT_LIMIT / sizeof(int)) * BM, N);
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
    // the largest layout any plan of either entry point may use for this shape
    return ws_bytes_cols(N, K, n_cols);
}

extern "C" spec_status spec_qmatmul(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                    int n_cols, int ldx, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                    void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    const Plan p = choose_plan(N, K, n_cols, false);
    st = check_ws(workspace, ws_bytes, ws_bytes_launch(N, K, p.nt, p.ncg, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, p.nt, workspace, dev_err,
                   (cudaStream_t)stream, SC_BLOCK, nullptr, 0, WIDE_AUTO, nullptr, p.ncg);
}

extern "C" int spec_qmatmul_plan(int N, int K, int n_cols, int packed_input) {
    if (N <= 0 || K < 256 || n_cols <= 0) return 0;
    const Plan p = choose_plan(N, K, n_cols, packed_input != 0);
    return 8 * p.nt;
}

extern "C" spec_status spec_qmatmul_swiglu(const uint8_t *wq, const uint16_t *ws, int F, int K, const uint16_t *x,
                                           const void *xpk, int n_cols, int ldx, uint16_t *act, int ld_act,
                                           void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(F >= 8 && F % 8 == 0, "qmatmul_swiglu: F must be a positive multiple of 8 (F=%d)", F);
    SPEC_CHECK_ARG(ld_act >= F, "qmatmul_swiglu: ld_act must be >= F (ld_act=%d F=%d)", ld_act, F);
    SPEC_CHECK_ARG(!xpk || spec::aligned16(xpk), "qmatmul_swiglu: xpk must be 16-byte aligned");
    spec_status st = check_args(wq, ws, 2 * F, K, x, n_cols, ldx, act, 2 * F);
    if (st != SPEC_OK) return st;
    if (n_cols == 0) return SPEC_OK;
    // with packed activations the 80-column pass needs no packing launch
    const bool packed = xpk && n_cols > 16 && n_cols <= WIDE_COLS;
    const Plan p = choose_plan(2 * F, K, n_cols, packed);
    st = check_ws(workspace, ws_bytes, ws_bytes_launch(2 * F, K, p.nt, p.ncg, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, 2 * F, K, x, n_cols, ldx, act, SPEC_BF16, ld_act, 0, 1, p.nt, workspace, dev_err,
                   (cudaStream_t)stream, SC_BLOCK, nullptr, 0, WIDE_AUTO,
                   packed && p.nt >= MAX_NT ? reinterpret_cast<const uint8_t *>(xpk) : nullptr, p.ncg, true);
}

extern "C" size_t spec_packed_activation_bytes(int K) {
    if (K < 256 || K % 256 != 0) return 0;
    return (size_t)(K / WIDE_KS) * WIDE_XC_BYTES;
}

extern "C" spec_status spec_qmatmul_packed(const uint8_t *wq, const uint16_t *ws, int N, int K, const void *xpk,
                                           int n_cols, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                           void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    SPEC_CHECK_ARG(N >= 1 && K >= 256 && K % 256 == 0, "qmatmul_packed: need N >= 1 and K a multiple of 256 (N=%d K=%d)",
                   N, K);
    SPEC_CHECK_ARG(n_cols > 16 && n_cols <= WIDE_COLS, "qmatmul_packed: n_cols must be in 17..80 (n_cols=%d)", n_cols);
    SPEC_CHECK_ARG(ldy >= N, "qmatmul_packed: ldy must be >= N (ldy=%d)", ldy);
    SPEC_CHECK_ARG(wq && ws && xpk && y, "qmatmul_packed: NULL pointer");
    SPEC_CHECK_ARG(spec::aligned16(wq) && spec::aligned16(ws) && spec::aligned16(xpk),
                   "qmatmul_packed: wq, ws and xpk must be 16-byte aligned");
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul_packed: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul_packed: accumulate needs SPEC_F32 output");
    spec_status st = check_ws(workspace, ws_bytes, ws_bytes_for(N, K, MAX_NT, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, nullptr, n_cols, K, y, y_dt, ldy, accumulate, 1, MAX_NT, workspace, dev_err,
                   (cudaStream_t)stream, SC_BLOCK, nullptr, 0, WIDE_MMA_SYNC, reinterpret_cast<const uint8_t *>(xpk));
}

extern "C" spec_status spec_qmatmul_devcols(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                            int n_cols, int ldx, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                            const int32_t *dev_cols, int min_cols, void *workspace, size_t ws_bytes,
                                            int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(dev_cols, "qmatmul_devcols: dev_cols is NULL");
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul_devcols: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul_devcols: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    const int nt = pass_nt(n_cols);
    st = check_ws(workspace, ws_bytes, ws_bytes_for(N, K, nt, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, nt, workspace, dev_err,
                   (cudaStream_t)stream, SC_BLOCK, dev_cols, min_cols);
}

extern "C" spec_status spec_qmatmul_sb(const uint8_t *wq, const uint8_t *sbr, int N, int K, const uint16_t *x,
                                       int n_cols, int ldx, void *y, spec_dtype y_dt, int ldy, int accumulate,
                                       void *workspace, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream) {
    spec_status st = check_args(wq, sbr, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(y_dt == SPEC_F32 || y_dt == SPEC_BF16, "qmatmul_sb: y_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(!(accumulate && y_dt != SPEC_F32), "qmatmul_sb: accumulate needs SPEC_F32 output");
    if (n_cols == 0) return SPEC_OK;
    const int nt = pass_nt(n_cols);
    st = check_ws(workspace, ws_bytes, ws_bytes_for(N, K, nt, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, sbr, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, nt, workspace, dev_err,
                   (cudaStream_t)stream, SC_SUPER);
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
    const int nt = pass_nt(n_cols);
    st = check_ws(workspace, ws_bytes, ws_bytes_for(N, K, nt, seg));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, seg, nt, workspace, nullptr,
                   (cudaStream_t)stream);
}

// Test hook: run the invariant kernel with an explicit column-tile width so the
// tests can show the per-column result does not depend on it.
extern "C" spec_status spec_qmatmul_debug_nt(const uint8_t *wq, const uint16_t *ws, int N, int K, const uint16_t *x,
                                             int n_cols, int ldx, float *y, int ldy, int nt, void *workspace,
                                             size_t ws_bytes, spec_stream_t stream) {
    spec_status st = check_args(wq, ws, N, K, x, n_cols, ldx, y, ldy);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(nt == 1 || nt == 2 || (nt >= MAX_NT && nt <= MAX_NT + 3), "nt must be 1, 2, 10, 11, 12 or 13");
    if (n_cols == 0) return SPEC_OK;
    // 10: the 80-column pass on the mma.sync kernel, 11: on the tcgen05 kernel;
    // 12: 16-column passes, up to five column groups per launch; 13: 8-column
    // passes, up to ten column groups per launch
    const int wide = nt == MAX_NT + 1 ? WIDE_TC : WIDE_MMA_SYNC;
    int ncg = 1;
    if (nt == MAX_NT + 2) nt = 2, ncg = MAX_NCG;
    else if (nt == MAX_NT + 3) nt = 1, ncg = 2 * MAX_NCG;
    else nt = nt > MAX_NT ? MAX_NT : nt;
    st = check_ws(workspace, ws_bytes, ws_bytes_launch(N, K, nt, ncg, 1));
    if (st != SPEC_OK) return st;
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, SPEC_F32, ldy, 0, 1, nt, workspace, nullptr,
                   (cudaStream_t)stream, SC_BLOCK, nullptr, 0, wide, nullptr, ncg);
}

// ---------------------------------------------------------------------------
// spec_qmatmul_static_scratch: the invariant product with its scratch in a
// fixed, statically sized device array instead of a caller-supplied buffer.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
// One scratch area per device (module-scope __device__ storage is per device).
// Its front holds the per-tile arrival counters, which must be zero when a
// launch starts; the rest holds partial sums that each call writes before it
// reads them.
static __device__ __align__(256) unsigned char g_qmm_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[spec::kMaxDevices] = {};

// Device address of this device's scratch; looked up on the first call made
// with that device current.
spec_status static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return spec::cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= spec::kMaxDevices) return spec::fail(SPEC_ERR_INVALID_ARG, "qmatmul_static_scratch: device %d", dev);
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
    const int nt = pass_nt(n_cols);
    const size_t need = ws_bytes_for(N, K, nt, 1);
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
    return qmm_run(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, 1, nt, scratch, dev_err,
                   (cudaStream_t)stream);
}
