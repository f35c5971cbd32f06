// Definitions shared by the two K1 kernels: the mma.sync kernel of qmatmul.cu
// (passes of up to 16 columns) and the tcgen05 kernel of qmatmul_tc.cu (the
// 80-column pass).  Both compute the same arithmetic; see qmatmul.cu's header.
#pragma once

#include "common.cuh"

namespace qmm {

constexpr int SEG_K = 512;                   // k per K-segment (the invariant reduction unit)
constexpr int BM = 128;                      // weight rows per tile
constexpr int SMEM_BUDGET = 226 * 1024;
// Arrival counters of a call lie in the workspace's first 4 x tiles bytes; no
// call has more than CNT_LIMIT / 4 tiles.  A call's stored sums and prefixes
// that lie below CNT_LIMIT are cleared once read, so every call finds its
// counters at zero whatever calls of other shapes used the workspace before.
constexpr size_t CNT_LIMIT = 64 * 1024;
// Scale formats: SC_BLOCK = one fp16 scale per 32-k block ([N][K/32]);
// SC_SUPER = per 256-k super-block an 8-byte record of eight 6-bit block scales
// and an fp16 super-scale, records in 16-byte pairs per row ([N][ceil(K/512) 16]
// bytes); block b's scale is D * s_(b mod 8), formed exactly in fp32.
constexpr int SC_BLOCK = 0, SC_SUPER = 1;
// The 80-column pass: its packed activations per 256-k stage (four 64-k groups
// of 80 columns x 128 bytes, then -136 x the block sums, [8 blocks][80] fp32).
constexpr int WIDE_COLS = 80;
constexpr int WIDE_KS = 256;
constexpr int WIDE_XC_BYTES = 4 * WIDE_COLS * 128 + 8 * WIDE_COLS * 4;

// The mma.sync 80-column pass's packed activations (one 256-k stage: four
// 64-k groups of 80 columns x 128 bytes in B-fragment order, then -136 x the
// block sums, [8 blocks][80] fp32).  Producers of an 80-row K1 input may write
// them directly (spec_add_rmsnorm_packed, spec_swiglu_packed) instead of
// leaving it to the matmul's packing kernel; both go through pack_pair.
constexpr int SYNC_WIDE_NT = 10;
constexpr int SYNC_WIDE_X_BYTES = 4 * 8 * SYNC_WIDE_NT * 128;

// Writes pair (blk, c) of a stage of a pass with NT column tiles: the bf16
// values of column c at k = 32 blk .. 32 blk + 31 of the stage (v: 4 x 8 in k
// order) in MMA B-fragment order into the stage's activation area xs, and
// -136 x the block sum into ci (the block sum is the four 8-k chunk sums, each
// summed in k order, added in chunk order).
template <int NT>
__device__ __forceinline__ void pack_pair(const uint4 (&v)[4], int blk, int c, uint8_t *xs, float *ci) {
    constexpr int X_BOX = 8 * NT * 128;   // 64 k of the pass's columns
    uint8_t *row = xs + (blk >> 1) * X_BOX + c * 128;
    float sum = 0.f;
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
        uint4 o;
        o.x = dev::prmt(w4[0], w4[2], 0x5410);   // (x0, x4)
        o.y = dev::prmt(w4[0], w4[2], 0x7632);   // (x1, x5)
        o.z = dev::prmt(w4[1], w4[3], 0x5410);   // (x2, x6)
        o.w = dev::prmt(w4[1], w4[3], 0x7632);   // (x3, x7)
        const int chunk = (((blk & 1) * 4 + q) ^ (c & 7)) << 4;
        *reinterpret_cast<uint4 *>(row + chunk) = o;
    }
    // MMA column slot g carries activation column pi(g) = (g & 1) * 4 + g / 2
    const int cc = c & 7, slot = (cc & 3) * 2 + (cc >> 2);
    ci[blk * 8 * NT + (c & ~7) + slot] = -136.0f * sum;
}

// Column c's 32 bf16 values at k = kb .. kb + 31 (kb a multiple of 32) into
// the mma.sync 80-column pass's packed activations of all stages, xpk.
__device__ __forceinline__ void pack_wide_block(const uint16_t *src, int kb, int c, uint8_t *xpk) {
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = *reinterpret_cast<const uint4 *>(src + 8 * q);
    uint8_t *xs = xpk + (size_t)(kb / WIDE_KS) * WIDE_XC_BYTES;
    pack_pair<SYNC_WIDE_NT>(v, (kb % WIDE_KS) / 32, c, xs, reinterpret_cast<float *>(xs + SYNC_WIDE_X_BYTES));
}

// Columns a call gated by a device-side count computes: none when the count is
// below min_cols, else the first min(n_cols, count).
__device__ __forceinline__ int gated_cols(int n_cols, const int32_t *dev_cols, int min_cols) {
    const int c = *dev_cols;
    return c < min_cols ? 0 : (c < n_cols ? c : n_cols);
}

// number of K-segments of length seg_k (the last may be shorter)
inline int n_segments(int K, int seg_k) { return (K + seg_k - 1) / seg_k; }

// Stream-K schedule: U = tiles x ks (128-row tile, K-segment) units dealt to G
// CTAs in equal contiguous ranges; seg_st = stages per segment.
struct Sched {
    int G;          // CTAs
    long long U;    // units = tiles * ks
    int ks, tiles, seg_st;   // segments, tiles, stages per segment
    // column groups of one launch: tile t is 128-row tile t / ncg of the
    // matrix for column group t % ncg (the groups of a row tile are adjacent,
    // so that its weights are read from DRAM once and then from L2)
    int ncg;
    __device__ long long begin(int c) const { return (long long)c * U / G; }
    __device__ int cta_of(long long u) const { return (int)(((u + 1) * G - 1) / U); }
};

// The schedule of a call with 128-row tiles, segments of seg512 x 512 k and
// stages of stage_k k on `sms` SMs, for ncg column groups.
inline Sched make_sched(int N, int K, int seg512, int stage_k, int sms, int ncg = 1) {
    Sched sch;
    sch.seg_st = seg512 * (SEG_K / stage_k);
    sch.ks = n_segments(K, seg512 * SEG_K);
    sch.ncg = ncg;
    sch.tiles = (N + BM - 1) / BM * ncg;
    sch.U = (long long)sch.tiles * sch.ks;
    sch.G = (int)(sch.U < sms ? sch.U : sms);
    // Nearly one tile per SM: one whole tile per CTA costs at most 15 % more work
    // per CTA than an even split and removes every split tile's publish and fold.
    if (sch.ks > 1 && sch.tiles <= sms && (long long)sch.tiles * 100 >= 85ll * sms) sch.G = sch.tiles;
    return sch;
}

// Workspace of a call: [counters (tiles ints, 256-byte rounded)][prefix: tiles x
// tile_elems floats][segment sums: tiles x ks x tile_elems floats][packed activations].
struct WsLayout {
    int *counters;
    float *prefix, *segs;
    uint8_t *xpk;
};

inline WsLayout ws_layout(void *workspace, int tiles, int ks, int tile_elems) {
    WsLayout w;
    const size_t cnt_bytes = (((size_t)tiles * sizeof(int)) + 255) & ~size_t(255);
    w.counters = reinterpret_cast<int *>(workspace);
    w.prefix = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + cnt_bytes);
    w.segs = w.prefix + (size_t)tiles * tile_elems;
    w.xpk = reinterpret_cast<uint8_t *>(w.segs + (size_t)tiles * ks * tile_elems);
    return w;
}

// The 80-column pass of spec_qmatmul on the 5th-generation tensor cores
// (qmatmul_tc.cu): columns col0 .. col0 + 79 of y, block-fp16 scales.
spec_status tc_wide_pass(const CUtensorMap &tw, const CUtensorMap &ts, const uint16_t *x, int ldx, int N, int K,
                         int n_cols, int col0, void *y, bool out_bf16, int ldy, int accumulate, int seg512,
                         void *workspace, int32_t *dev_err, const int32_t *dev_cols, int min_cols,
                         cudaStream_t stream);

}  // namespace qmm
