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
    __device__ long long begin(int c) const { return (long long)c * U / G; }
    __device__ int cta_of(long long u) const { return (int)(((u + 1) * G - 1) / U); }
};

// The schedule of a call with 128-row tiles, segments of seg512 x 512 k and
// stages of stage_k k on `sms` SMs.
inline Sched make_sched(int N, int K, int seg512, int stage_k, int sms) {
    Sched sch;
    sch.seg_st = seg512 * (SEG_K / stage_k);
    sch.ks = n_segments(K, seg512 * SEG_K);
    sch.tiles = (N + BM - 1) / BM;
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
