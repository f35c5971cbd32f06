// K2 + K3: batch-invariant split-KV causal attention over a paged KV cache.
//
// ramgpt.org, "When Lossless Speculation Stops Being Lossless on Blackwell",
// section "Flash Attention Changes Geometry With Batch Width": choosing tile
// geometry by query width changed the KV traversal and the combine order.
// Here every row's reduction structure is fixed by its own position p:
//  * keys are cut into chunks of CHUNK = 256 (a constant), chunk c covers keys
//    [256c, 256c + 255]; row p has partials for chunks 0 .. p / 256;
//  * a chunk is cut into sub-tiles of 64 keys; for each sub-tile w whose first
//    key is <= p the row gets (m_w, l_w, o_w): the max of its visible scores,
//    the sum of 2^(s - m_w) and the 2^(s - m_w)-weighted values;
//  * the chunk partial merges those sub-tiles in ascending w:
//    m = max_w m_w, l = sum_w l_w 2^(m_w - m), o = sum_w o_w 2^(m_w - m);
//  * K3 combines a row's chunk partials in ascending chunk order.
// The other rows of the call only decide which warp, round or CTA handles a
// row; sub-tiles past p are left out of the row's merge altogether.
//
// K2 (attn_partial_kernel): a resident grid (at most one CTA per SM) walks
// the (chunk, kv head, sequence) items, CTA b taking items b, b + grid, ...,
// the chunk index varying slowest so that each warp's walk ends at the chunks
// the sequences reach, whatever bound max_kv_len puts on them.  When
// sequences average more than one M-tile, a second instance makes each chunk
// two neighbouring items, the lower and the upper half of its M-tiles: for
// sequences of at most SPLIT_CHUNKS chunks, and for all of them when the call
// has items for three or more rounds of the grid.  Each item's K and V are
// staged through a ring of three (D = 128; four at D = 64) half-item buffers
// in the order K0 V0 K1 V1 ..., so that up to 1.5 items' copies run ahead of
// the math.  A producer warp copies an item's K pages and its V pages (one TMA
// box per 16-key page: the cache viewed as 5-D with the head dimension split
// into 64-wide halves, so that each 128-byte row takes the 128B swizzle) into
// a buffer's four 64-key sub-tile slots; consumer warp w owns sub-tile w
// and, for each 16-row M-tile of (query row, grouped head) pairs, runs
// S = Q K^T and O = P V on mma.sync m16n8k16 with fp32 accumulation (P enters
// the PV product as a hi + lo pair of 16-bit values, rounding error ~2^-17),
// leaving its (m_w, l_w, o_w) in shared memory; the four warps then merge
// them and write the chunk partials.  K and V are released separately (K
// after the item's last S, V after its last P V).
// Which CTA computes an item, and when, is scheduling: an item's operations
// are those of a CTA of its own.
// K3 (attn_combine_kernel): one warp per (row, head, 32-value block of the
// head dimension), one value per lane; when every row is within 32 chunks, an
// instance that finishes a one-chunk row from an early request of chunk 0 and
// loads up to 32 chunks' partials in one round (the same operations).
#include <algorithm>
#include <climits>

#include "qmm_shared.cuh"

namespace {

constexpr int CHUNK = 256;
constexpr int SUB = 64;
constexpr int PAGE = 16;
constexpr int NCONS = CHUNK / SUB;   // one consumer warp per sub-tile
constexpr int SPLIT_CHUNKS = 8;      // sequences of at most this many chunks have their M-tiles halved
constexpr int THREADS = (NCONS + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;

// Shared memory: a ring of NBUF buffers, each holding one half-item -- an
// item's K or its V for all four sub-tiles -- in the order K0 V0 K1 V1 ...;
// then the sub-tile partials of MR M-tiles for the merge.
template <int D>
struct ACfg {
    static constexpr int HALVES = D / 64;                 // 64-wide d boxes per key row
    static constexpr int KV_BYTES = HALVES * SUB * 128;   // one of K or V for a sub-tile
    static constexpr int BUF = NCONS * KV_BYTES;          // one half-item
    static constexpr int MR = D == 128 ? 1 : 4;           // M-tiles per round
    static constexpr int OSTR = D + 4;                    // padded row stride of a sub-tile's o (floats)
    static constexpr int PART = 16 * OSTR * 4 + 16 * 8;   // o and (m, l) of one (M-tile, sub-tile)
    static constexpr int PARTS = MR * NCONS * PART;
    static constexpr int NBUF = (232448 - 1024 - PARTS - 256) / BUF > 4 ? 4 : (232448 - 1024 - PARTS - 256) / BUF;
    static constexpr int PART_OFF = NBUF * BUF;
    static constexpr int BAR_OFF = PART_OFF + PARTS;
    static constexpr int NBAR = NBUF * NCONS + NBUF;        // full per (buffer, sub-tile); free per buffer
    static constexpr int SMEM = 1024 + BAR_OFF + NBAR * 8;
    static_assert(NBUF >= 3, "at least three half-items in the ring");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// Byte offset of (key, 64-wide half hh of the head dimension) in a sub-tile's
// K or V slot: one 4 KB box per 16-key page, [page][half][key][128 B] (128-byte
// swizzle within each 1024-byte atom, by key & 7).
__device__ __forceinline__ uint32_t kv_off(int key, int hh, int halves) {
    return (uint32_t)((key >> 4) * (halves * 2048) + hh * 2048 + (key & 15) * 128);
}

template <bool BF16>
__device__ __forceinline__ void mma16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1, const float (&c)[4]) {
    if (BF16)
        dev::mma_bf16(d, a0, a1, a2, a3, b0, b1, c);
    else
        dev::mma_f16(d, a0, a1, a2, a3, b0, b1, c);
}

// pack two fp32 into the 16-bit pair (lo half = a) with round to nearest even,
// and return the residuals a - hi, b - hi (exact in fp32)
template <bool BF16>
__device__ __forceinline__ uint32_t pack_hi(float a, float b, float &ra, float &rb) {
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        float2 f = __bfloat1622float2(h);
        ra = a - f.x;
        rb = b - f.y;
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        float2 f = __half22float2(h);
        ra = a - f.x;
        rb = b - f.y;
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int D, bool BF16, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1)
attn_partial_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const uint16_t *__restrict__ q, int Hq, int Hkv, float scale_log2, int num_pages,
                    const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_start,
                    const int32_t *__restrict__ cu_rows, int S, int R, int max_kv_len, int nc_max,
                    float2 *__restrict__ part_ml, float *__restrict__ part_o, int32_t *dev_err, int split_long) {
    constexpr int parts = SPLIT ? 2 : 1;   // items per chunk: halves of its M-tiles when SPLIT
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    using C = ACfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);   // [buffer][sub-tile]
    uint64_t *freeb = full + C::NBUF * NCONS;   // [buffer]: every consumer warp is done with it

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = Hq / Hkv;

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::NBUF * NCONS; ++b) dev::mbar_init(&full[b], 1);
        for (int b = 0; b < C::NBUF; ++b) dev::mbar_init(&freeb[b], NCONS);
        dev::fence_barrier_init();
    }
    __syncthreads();

    // The chunk index varies slowest over the items, so every item of a chunk
    // no sequence reaches is empty: a warp's walk ends at the chunks the
    // sequences reach (at most nc_max) instead of skipping the rest one by one.
    // Every warp finds the same bound from the same inputs.
    const long long per_chunk = (long long)Hkv * S * parts;
    const long long nitems_all = (long long)nc_max * per_chunk;
    auto chunks_reached = [&]() -> int {
        int nc = 0;
        for (int s = lane; s < S; s += 32) {
            const int rows = cu_rows[s + 1] - cu_rows[s], ctx = ctx_start[s];
            if (rows > 0 && ctx >= 0)
                nc = max(nc, (int)min((long long)nc_max, ((long long)ctx + rows + CHUNK - 1) / CHUNK));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) nc = max(nc, __shfl_xor_sync(0xffffffffu, nc, o));
        return nc;
    };
    // With SPLIT, an even grid and a sequence longer than SPLIT_CHUNKS chunks
    // (whose second parts are empty), odd rounds take each item's partner
    // (it ^ 1): a round covers whole chunk pairs (the grid and the bound are
    // even), so every item is still taken once, the two halves of a chunk stay
    // on CTAs 2j and 2j + 1 of the same round, and a CTA alternates first and
    // second parts instead of half of the CTAs drawing only the empty ones.
    // (With only short sequences the fixed parts measured faster.)
    auto flip_of = [&](int nc) { return SPLIT && (gridDim.x % 2 == 0) && nc > SPLIT_CHUNKS; };
    auto item_of = [&](long long it, long long round, bool flip) -> long long {
        return (flip && (round & 1)) ? (it ^ 1) : it;
    };

    // Item `it` of the call: chunk c of kv head kvh of sequence s, with SPLIT
    // the lower or upper half of the chunk's M-tiles (the two halves are
    // neighbouring items, so they run at the same time on a CTA pair and the
    // second copy of the chunk comes from L2).  Every warp derives the same
    // geometry from the same inputs, so producer and consumers skip the same
    // items.
    struct Item {
        int c, kvh, s, r0, rows, ctx, len, kbeg, kend, nsub, mt_lo, mt_hi;
    };
    auto item = [&](long long it, Item &m) -> bool {
        const int part = SPLIT ? (int)(it & 1) : 0;   // the parts of a chunk are neighbouring items
        if (SPLIT) it >>= 1;
        // the chunk index varies slowest: whatever bound max_kv_len puts on the
        // chunk count, the chunks that exist come first and spread evenly over the CTAs
        m.kvh = (int)(it % Hkv);
        m.s = (int)((it / Hkv) % S);
        m.c = (int)(it / ((long long)Hkv * S));
        m.r0 = cu_rows[m.s];
        m.rows = cu_rows[m.s + 1] - m.r0;
        m.ctx = ctx_start[m.s];
        m.len = m.ctx + m.rows;
        if (m.rows <= 0 || m.ctx < 0) return false;
        if (m.r0 < 0 || m.r0 + m.rows > R) {  // rows outside the workspace the host sized
            if (threadIdx.x == 0 && m.c == 0 && m.kvh == 0) dev::report(dev_err, SPEC_DEVERR_LAYOUT);
            return false;
        }
        if (m.len > max_kv_len || m.len > max_blocks * PAGE) {
            if (threadIdx.x == 0 && m.c == 0 && m.kvh == 0) dev::report(dev_err, SPEC_DEVERR_LENGTH);
            return false;
        }
        m.kbeg = m.c * CHUNK;
        if (m.kbeg >= m.len) return false;
        m.kend = min(m.kbeg + CHUNK, m.len);
        m.nsub = (m.kend - m.kbeg + SUB - 1) / SUB;
        if constexpr (SPLIT) {
            // this part's M-tiles of the chunk: the lower or the upper half when
            // the sequence spans at most SPLIT_CHUNKS chunks or the call has
            // items for several rounds of the grid (split_long, from the host);
            // otherwise a longer sequence keeps its chunks whole in the first
            // part (its second parts are empty)
            const int mtiles = ((m.rows - max(0, m.kbeg - m.ctx)) * G + 15) / 16;
            const int half =
                ((m.len + CHUNK - 1) / CHUNK <= SPLIT_CHUNKS || split_long) ? mtiles / 2 : mtiles;
            m.mt_lo = part ? half : 0;
            m.mt_hi = part ? mtiles : half;
            return m.mt_lo < m.mt_hi;
        }
        return true;
    };

    if (warp == NCONS) {
        // ---------------- producer: each item's K, then its V, into the ring ----------------
        // An item's (at most 16) block-table entries are read by 16 lanes at once,
        // and each of those lanes copies its page once the buffer's previous
        // half-item is released.  Every sub-tile barrier of the buffer completes a
        // phase per half-item (without bytes where the chunk has no such sub-tile),
        // so a buffer's phase parity is the same for every consumer warp.
        if (lane == 0) {
            dev::prefetch_tmap(&tk);
            dev::prefetch_tmap(&tv);
        }
        bool ok = true;
        int jv = 0;   // valid items so far
        // the first item's copies go out before the bound is known (an item past
        // it is empty, so nothing is issued for it either way)
        long long nitems = nitems_all;
        bool flip = false;
        for (long long it = blockIdx.x, rd = 0; it < nitems && ok; it += gridDim.x, ++rd) {
            if (rd == 1) {
                const int nc = chunks_reached();
                nitems = min(nitems, (long long)nc * per_chunk);
                flip = flip_of(nc);
                if (it >= nitems) break;
            }
            const long long jt = item_of(it, rd, flip);
            // the chunk's (at most 16) block-table entries, loaded together with the
            // item's own geometry; an entry past the sequence's pages is not used
            int bt_entry = -1;
            {
                const long long q = SPLIT ? (jt >> 1) : jt;
                const int s = (int)((q / Hkv) % S), c = (int)(q / ((long long)Hkv * S));
                const int e = c * (CHUNK / PAGE) + lane;
                if (lane < CHUNK / PAGE && e < max_blocks) bt_entry = block_table[(size_t)s * max_blocks + e];
            }
            Item m;
            if (!item(jt, m)) continue;
            const int pg_first = m.kbeg / PAGE, pg_end = (m.kend + PAGE - 1) / PAGE;
            int my_phys = 0;
            if (lane < pg_end - pg_first) {
                my_phys = bt_entry;
                if (my_phys < 0 || my_phys >= num_pages) {
                    dev::report(dev_err, SPEC_DEVERR_BLOCK_TABLE);
                    my_phys = 0;
                }
            }
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const int j = 2 * jv + kv, b = j % C::NBUF;   // half-item j of this CTA, its buffer
                uint64_t *fl = full + b * NCONS;
                const CUtensorMap *map = kv ? &tv : &tk;
                int got = 1;
                if (lane == 0 && j >= C::NBUF) got = dev::mbar_wait(&freeb[b], ((j / C::NBUF) - 1) & 1) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (lane == 0)
                    for (int w = m.nsub; w < NCONS; ++w) dev::mbar_arrive(&fl[w]);
                // lane w posts sub-tile w's bytes; then lane l copies the item's page l
                // (sub-tile l / 4; both halves of D in one box), all in one instruction
                if (lane < m.nsub) {
                    const int pg0 = pg_first + lane * (SUB / PAGE), pg1 = min(pg0 + SUB / PAGE, pg_end);
                    dev::mbar_arrive_expect_tx(&fl[lane], (uint32_t)((pg1 - pg0) * C::HALVES * 2048));
                }
                __syncwarp();
                if (lane < pg_end - pg_first)
                    dev::tma_load_5d(smem + b * C::BUF + (lane / (SUB / PAGE)) * C::KV_BYTES +
                                         (lane % (SUB / PAGE)) * C::HALVES * 2048,
                                     map, 0, 0, 0, m.kvh, my_phys, &fl[lane / (SUB / PAGE)]);
            }
            ++jv;
        }
        // every copy issued is waited for by its consumer warp before the CTA can exit
        return;
    }

    // ---------------- consumers: warp w owns sub-tile w of every item ----------------
    const int w = warp;
    const int g = lane >> 2, t = lane & 3;
    bool ok = true;
    int vi = 0;   // valid items so far: item vi's K is half-item 2 vi, its V 2 vi + 1
    const int nc_reached = chunks_reached();
    const long long nitems = min(nitems_all, (long long)nc_reached * per_chunk);
    const bool flip = flip_of(nc_reached);
    for (long long it = blockIdx.x, rd = 0; it < nitems; it += gridDim.x, ++rd) {
        Item itm;
        if (!item(item_of(it, rd, flip), itm)) continue;
        const int c = itm.c, kvh = itm.kvh, r0 = itm.r0, rows = itm.rows, ctx = itm.ctx, len = itm.len;
        const int kbeg = itm.kbeg, nsub = itm.nsub;
        const int i0 = max(0, kbeg - ctx);  // first row whose position reaches this chunk
        const int mrows = (rows - i0) * G;
        // this item's M-tiles: mt_first .. mtiles - 1
        const int mtiles = SPLIT ? itm.mt_hi : (mrows + 15) / 16;
        const int mt_first = SPLIT ? itm.mt_lo : 0;
        const int key0 = kbeg + w * SUB;
        const bool has_sub = w < nsub;
        const int bk = (2 * vi) % C::NBUF, bv = (2 * vi + 1) % C::NBUF;
        const uint32_t pk = (uint32_t)(((2 * vi) / C::NBUF) & 1), pv = (uint32_t)(((2 * vi + 1) / C::NBUF) & 1);
        ++vi;
        uint8_t *kslot = smem + bk * C::BUF + w * C::KV_BYTES;
        uint8_t *vslot = smem + bv * C::BUF + w * C::KV_BYTES;
        const uint32_t kb = dev::smem_u32(kslot), vb = dev::smem_u32(vslot);
        bool kwaited = false, vwaited = false;
        bool karrived = false, varrived = false;   // this warp's release of the item's K / V slots

        for (int mt0 = mt_first; mt0 < mtiles; mt0 += C::MR) {
            // ---- each warp: (m_w, l_w, o_w) of its sub-tile for up to MR M-tiles ----
            const bool last_round = mt0 + C::MR >= mtiles;
            for (int j = 0; j < C::MR && mt0 + j < mtiles && has_sub && ok; ++j) {
                const int mt = mt0 + j;
                const bool last_tile = last_round && (j == C::MR - 1 || mt0 + j + 1 == mtiles);
                int pos[2];
                bool valid[2];
                size_t qoff[2];
    #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = mt * 16 + g + 8 * h;
                    valid[h] = m < mrows;
                    const int i = i0 + (valid[h] ? m / G : 0);
                    const int gg = valid[h] ? m % G : 0;
                    pos[h] = ctx + i;
                    qoff[h] = ((size_t)(r0 + i) * Hq + kvh * G + gg) * D;
                }
                // Q fragments for all k-steps (A operand): row m0 / m1, d = 16 kk + 2t (+8), all loads in flight together
                uint32_t qa[D / 16][4];
    #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int d0 = 16 * kk + 2 * t;
                    qa[kk][0] = valid[0] ? __ldg(reinterpret_cast<const unsigned int *>(q + qoff[0] + d0)) : 0u;
                    qa[kk][1] = valid[1] ? __ldg(reinterpret_cast<const unsigned int *>(q + qoff[1] + d0)) : 0u;
                    qa[kk][2] = valid[0] ? __ldg(reinterpret_cast<const unsigned int *>(q + qoff[0] + d0 + 8)) : 0u;
                    qa[kk][3] = valid[1] ? __ldg(reinterpret_cast<const unsigned int *>(q + qoff[1] + d0 + 8)) : 0u;
                }
                if (!kwaited) {
                    kwaited = true;
                    if (!dev::mbar_wait(&full[bk * NCONS + w], pk)) {
                        if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
                // ---- S = Q K^T (16 rows x 64 keys) ----
                float sc[8][4];
    #pragma unroll
                for (int jj = 0; jj < 8; ++jj) sc[jj][0] = sc[jj][1] = sc[jj][2] = sc[jj][3] = 0.f;
    #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qa0 = qa[kk][0], qa1 = qa[kk][1], qa2 = qa[kk][2], qa3 = qa[kk][3];
                    const int hh = (16 * kk) / 64;
                    const int cbase = ((16 * kk) % 64) / 8;
    #pragma unroll
                    for (int jp = 0; jp < 4; ++jp) {
                        const int mi = lane >> 3;
                        const int key = 8 * (2 * jp + (mi >> 1)) + (lane & 7);
                        const int ch = cbase + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        dev::ldmatrix_x4(b0, b1, b2, b3, kb + kv_off(key, hh, C::HALVES) + ((ch ^ (key & 7)) << 4));
                        mma16<BF16>(sc[2 * jp], qa0, qa1, qa2, qa3, b0, b1, sc[2 * jp]);
                        mma16<BF16>(sc[2 * jp + 1], qa0, qa1, qa2, qa3, b2, b3, sc[2 * jp + 1]);
                    }
                }
                if (last_tile) {
                    // the item's last S of this warp: its K slot may take the next item's keys
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&freeb[bk]);
                    karrived = true;
                }
                // ---- mask, scale to log2 units, softmax within the sub-tile ----
                float mx[2] = {-INFINITY, -INFINITY};
    #pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const int key = key0 + 8 * jj + 2 * t + (e & 1);
                        const bool vis = valid[h] && key <= pos[h];
                        const float v = vis ? sc[jj][e] * scale_log2 : -INFINITY;
                        sc[jj][e] = v;
                        mx[h] = fmaxf(mx[h], v);
                    }
                }
    #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                }
                float rs[2] = {0.f, 0.f};
    #pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const float p = (mx[h] == -INFINITY) ? 0.f : exp2f(sc[jj][e] - mx[h]);
                        sc[jj][e] = p;
                        rs[h] += p;
                    }
                }
    #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
                    rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
                }
                if (!vwaited) {
                    vwaited = true;
                    if (!dev::mbar_wait(&full[bv * NCONS + w], pv)) {
                        if (lane == 0) dev::report(dev_err, SPEC_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int nvalid = len - key0;  // keys of this slot inside the sequence
                    if (nvalid < SUB) {
                        // V rows past the sequence end hold stale or unloaded data: zero them so
                        // that 0-probability keys contribute exactly 0 to P V
                        for (int idx = lane; idx < C::HALVES * (SUB - nvalid) * 8; idx += 32) {
                            const int hh = idx / ((SUB - nvalid) * 8);
                            const int rem = idx % ((SUB - nvalid) * 8);
                            const int key = nvalid + rem / 8, ch = rem % 8;
                            *reinterpret_cast<uint4 *>(vslot + kv_off(key, hh, C::HALVES) + ch * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                    __syncwarp();
                }
                // ---- O = P V with P = hi + lo ----
                float o[D / 8][4];
    #pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    #pragma unroll
                for (int kk = 0; kk < SUB / 16; ++kk) {
                    uint32_t ph[4], pl[4];
                    float r00, r01, r10, r11, r20, r21, r30, r31;
                    ph[0] = pack_hi<BF16>(sc[2 * kk][0], sc[2 * kk][1], r00, r01);
                    ph[1] = pack_hi<BF16>(sc[2 * kk][2], sc[2 * kk][3], r10, r11);
                    ph[2] = pack_hi<BF16>(sc[2 * kk + 1][0], sc[2 * kk + 1][1], r20, r21);
                    ph[3] = pack_hi<BF16>(sc[2 * kk + 1][2], sc[2 * kk + 1][3], r30, r31);
                    pl[0] = pack2<BF16>(r00, r01);
                    pl[1] = pack2<BF16>(r10, r11);
                    pl[2] = pack2<BF16>(r20, r21);
                    pl[3] = pack2<BF16>(r30, r31);
    #pragma unroll
                    for (int ndp = 0; ndp < D / 16; ++ndp) {
                        const int mi = lane >> 3;
                        const int key = 16 * kk + 8 * (mi & 1) + (lane & 7);
                        const int dch = 2 * ndp + (mi >> 1);     // 8-wide d chunk
                        const int hh = dch / 8, ch = dch % 8;
                        uint32_t b0, b1, b2, b3;
                        dev::ldmatrix_x4_trans(b0, b1, b2, b3,
                                               vb + kv_off(key, hh, C::HALVES) + ((ch ^ (key & 7)) << 4));
                        mma16<BF16>(o[2 * ndp], ph[0], ph[1], ph[2], ph[3], b0, b1, o[2 * ndp]);
                        mma16<BF16>(o[2 * ndp], pl[0], pl[1], pl[2], pl[3], b0, b1, o[2 * ndp]);
                        mma16<BF16>(o[2 * ndp + 1], ph[0], ph[1], ph[2], ph[3], b2, b3, o[2 * ndp + 1]);
                        mma16<BF16>(o[2 * ndp + 1], pl[0], pl[1], pl[2], pl[3], b2, b3, o[2 * ndp + 1]);
                    }
                }
                if (last_tile) {
                    // the item's last P V of this warp: its V slot may take the next item's values
                    // (the zeroing above wrote it through the generic proxy: order that first)
                    dev::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(&freeb[bv]);
                    varrived = true;
                }
                // ---- leave (m_w, l_w, o_w) of rows g, g + 8 in shared memory ----
                uint8_t *pb = smem + C::PART_OFF + (j * NCONS + w) * C::PART;
                float *po_s = reinterpret_cast<float *>(pb);
                float2 *pml = reinterpret_cast<float2 *>(pb + 16 * C::OSTR * 4);
    #pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    *reinterpret_cast<float2 *>(po_s + g * C::OSTR + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
                    *reinterpret_cast<float2 *>(po_s + (g + 8) * C::OSTR + 8 * nd + 2 * t) = make_float2(o[nd][2], o[nd][3]);
                }
                if (t == 0) {
                    pml[g] = make_float2(mx[0], rs[0]);
                    pml[g + 8] = make_float2(mx[1], rs[1]);
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(NCONS * 32) : "memory");
            // ---- merge the sub-tiles of each row in ascending order, write the chunk partial ----
            if (ok) {
                constexpr int D4 = D / 4;
                for (int e = threadIdx.x; e < C::MR * 16 * D4; e += NCONS * 32) {
                    const int j = e / (16 * D4), row = (e / D4) % 16, d4 = e % D4;
                    const int mt = mt0 + j;
                    const int m = mt * 16 + row;
                    if (mt >= mtiles || m >= mrows) continue;
                    const int i = i0 + m / G, gg = m % G;
                    const int p = ctx + i;
                    const int nw = min(nsub, (p - kbeg) / SUB + 1);   // sub-tiles whose first key is visible
                    const uint8_t *pb0 = smem + C::PART_OFF + (j * NCONS) * C::PART;
                    float mmax = -INFINITY;
                    for (int ww = 0; ww < nw; ++ww)
                        mmax = fmaxf(mmax, reinterpret_cast<const float2 *>(pb0 + ww * C::PART + 16 * C::OSTR * 4)[row].x);
                    float l = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int ww = 0; ww < nw; ++ww) {
                        const uint8_t *pb = pb0 + ww * C::PART;
                        const float2 ml = reinterpret_cast<const float2 *>(pb + 16 * C::OSTR * 4)[row];
                        const float sc = exp2f(ml.x - mmax);
                        l = fmaf(ml.y, sc, l);
                        const float4 ov = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(pb) +
                                                                            row * C::OSTR + 4 * d4);
                        acc.x = fmaf(ov.x, sc, acc.x);
                        acc.y = fmaf(ov.y, sc, acc.y);
                        acc.z = fmaf(ov.z, sc, acc.z);
                        acc.w = fmaf(ov.w, sc, acc.w);
                    }
                    const size_t pidx = ((size_t)(r0 + i) * Hq + kvh * G + gg) * nc_max + c;
                    *reinterpret_cast<float4 *>(part_o + pidx * D + 4 * d4) = acc;
                    if (d4 == 0) part_ml[pidx] = make_float2(mmax, l);
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(NCONS * 32) : "memory");
        }
        // a warp without a sub-tile in this item (or after an error) still releases once
        if (!karrived) {
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&freeb[bk]);
        }
        if (!varrived) {
            dev::fence_proxy_async();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&freeb[bv]);
        }
    }
}

// K3: out = (sum_c o_c 2^(m_c - m)) / (sum_c l_c 2^(m_c - m)), c ascending.
// One warp per (row, head, 32-value block of the head dimension), one value
// per lane: the chunk partials of 32 chunks are requested at once (the combine
// is a chain of dependent loads otherwise), then added in ascending chunk
// order.
template <int D, bool OUT_BF16, bool SHORT>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const int32_t *__restrict__ ctx_start, const int32_t *__restrict__ cu_rows, int S, int R, int Hq,
                    int nc_max, const float2 *__restrict__ part_ml, const float *__restrict__ part_o, void *out,
                    int max_kv_len, int kv_cap, uint8_t *__restrict__ xpk) {
    dev::pdl_wait();
    dev::pdl_launch_dependents();
    constexpr int QB = D / 32;   // 32-value blocks of a head
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= R * Hq * QB) return;
    const int qb = wid % QB, rh = wid / QB;
    const int r = rh / Hq, h = rh % Hq;
    const int d = qb * 32 + lane;
    // SHORT (every row within 32 chunks): chunk 0's partial, which every row
    // that is combined has, is requested together with the row's position
    float2 ml0 = make_float2(0.f, 0.f);
    float ov0 = 0.f;
    if constexpr (SHORT) {
        ml0 = part_ml[(size_t)rh * nc_max];
        ov0 = part_o[(size_t)rh * nc_max * D + d];
    }
    const int lo = dev::warp_seq_of_row(cu_rows, S, r);   // sequence of row r
    const int r0 = cu_rows[lo], rows = cu_rows[lo + 1] - r0, ctx = ctx_start[lo];
    const int p = ctx + (r - r0);
    const long long len = (long long)ctx + rows;
    // the partial kernel's rejections (layout or length), which leave no partials
    const bool rejected = rows <= 0 || ctx < 0 || r0 < 0 || r0 + rows > R || len > max_kv_len || len > kv_cap;
    float acc = 0.f;
    if (rejected || p < 0 || p >= max_kv_len) {
        // a rejected sequence (reported by the partial kernel): emit zeros
    } else if constexpr (SHORT) {
        const int nc = p / CHUNK + 1;   // at most 32
        if (nc == 1) {
            // one chunk: the general path's operations with c = 0 alone (the
            // other lanes' maxima are -inf, so m = fmaxf(-inf, m_0))
            const float m = fmaxf(-INFINITY, ml0.x);
            const float w = exp2f(ml0.x - m);
            const float l = fmaf(ml0.y, w, 0.f);
            acc = fmaf(ov0, w, 0.f);
            acc *= 1.0f / l;
        } else {
            // one chunk per lane: the general path's operations (a single group,
            // c0 = 0), with the (m, l) pairs and the values requested together
            // instead of the pairs first for the maximum
            const float2 *ml = part_ml + (size_t)rh * nc_max;
            const float *ob = part_o + (size_t)rh * nc_max * D + d;
            const float2 mlv = lane < nc ? ml[lane] : make_float2(-INFINITY, 0.f);
            float ov[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = j < nc ? ob[(size_t)j * D] : 0.f;
            float m = lane < nc ? fmaxf(-INFINITY, mlv.x) : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float wl = lane < nc ? exp2f(mlv.x - m) : 0.f;
            float l = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float w = __shfl_sync(0xffffffffu, wl, j);
                const float lc = __shfl_sync(0xffffffffu, mlv.y, j);
                if (j < nc) {
                    l = fmaf(lc, w, l);
                    acc = fmaf(ov[j], w, acc);
                }
            }
            acc *= 1.0f / l;
        }
    } else {
        const int nc = p / CHUNK + 1;
        const float2 *ml = part_ml + (size_t)rh * nc_max;
        const float *ob = part_o + (size_t)rh * nc_max * D + d;
        // m: max over the chunks (exact, any order); lane j holds chunks j, j + 32, ...
        float m = -INFINITY;
        for (int c = lane; c < nc; c += 32) m = fmaxf(m, ml[c].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        // l and the weighted values in ascending chunk order, 32 chunks' loads at a time
        float l = 0.f;
        for (int c0 = 0; c0 < nc; c0 += 32) {
            const int cl = c0 + lane;
            const float2 mlv = cl < nc ? ml[cl] : make_float2(-INFINITY, 0.f);
            const float wl = cl < nc ? exp2f(mlv.x - m) : 0.f;
            const int cn = min(32, nc - c0);
            float ov[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = j < cn ? ob[(size_t)(c0 + j) * D] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float w = __shfl_sync(0xffffffffu, wl, j);
                const float lc = __shfl_sync(0xffffffffu, mlv.y, j);
                if (j < cn) {
                    l = fmaf(lc, w, l);
                    acc = fmaf(ov[j], w, acc);
                }
            }
        }
        acc *= 1.0f / l;
    }
    const size_t oi = (size_t)rh * D + d;
    if (OUT_BF16) {
        reinterpret_cast<__nv_bfloat16 *>(out)[oi] = __float2bfloat16_rn(acc);
        if (xpk) {
            // row r is column r of an 80-column K1 pass (the o projection): pack this
            // 32-value block too, once the warp's stores are visible to it
            __syncwarp();
            if (lane == 0) {
                const int kb = h * D + 32 * qb;
                qmm::pack_wide_block(reinterpret_cast<const uint16_t *>(out) + (size_t)r * Hq * D + kb, kb, r, xpk);
            }
        }
    } else {
        reinterpret_cast<float *>(out)[oi] = acc;
    }
}

template <int D, bool BF16>
spec_status launch_partial(const CUtensorMap &tk, const CUtensorMap &tv, const void *q, int Hq, int Hkv, float scale,
                           int num_pages, const int32_t *bt, int max_blocks, const int32_t *ctx, const int32_t *cu,
                           int S, int R, int max_kv_len, int nc_max, float2 *ml, float *po, int32_t *dev_err,
                           cudaStream_t st) {
    using C = ACfg<D>;
    // Split a chunk's M-tiles over two items when sequences have more than one
    // M-tile on average.  The kernel halves only the chunks of sequences that
    // are short (SPLIT_CHUNKS chunks at most, decided from each sequence's own
    // length, since max_kv_len is only a bound): there the items alone leave
    // SMs idle, while long contexts are bound by each SM's copies, which a
    // split would double.
    const int G = Hq / Hkv;
    const bool split = S > 0 && (long long)R * G > 16ll * S;
    const int parts = split ? 2 : 1;
    auto kern = split ? attn_partial_kernel<D, BF16, true> : attn_partial_kernel<D, BF16, false>;
    static spec::SmemOptIn opt_in[2];
    spec_status so = spec::smem_opt_in(kern, C::SMEM, opt_in[split ? 1 : 0], "cudaFuncSetAttribute(attn smem)");
    if (so != SPEC_OK) return so;
    // a resident grid: at most one CTA per SM (the shared memory of one), CTA b taking items b, b + grid, ...
    const long long items = (long long)nc_max * Hkv * S * parts;
    const int sms = spec::num_sms() > 0 ? spec::num_sms() : 148;
    const int grid = (int)(items < sms ? items : sms);
    // With items for three or more rounds of the grid (at the bound), long
    // sequences' chunks are halved too: the finer items balance the CTAs'
    // loads better than whole ones (16384 keys, one sequence, widths 4 and 8:
    // 5 % faster), while with fewer items the doubled copies cost more
    // (4096 keys at width 8, 8 % slower).
    const bool split_long = split && (long long)nc_max * Hkv * S >= 3ll * grid;
    cudaError_t le = spec::launch_pdl(kern, dim3(grid), dim3(THREADS), C::SMEM, st, tk, tv,
                                      reinterpret_cast<const uint16_t *>(q), Hq, Hkv, scale * LOG2E, num_pages, bt,
                                      max_blocks, ctx, cu, S, R, max_kv_len, nc_max, ml, po, dev_err,
                                      split_long ? 1 : 0);
    return spec::cuda_status(le, "attn partial launch");
}

}  // namespace

namespace spec {
size_t attn_workspace_bytes(int R, int Hq, int D, int max_kv_len) {
    const size_t nc = (size_t)((max_kv_len + CHUNK - 1) / CHUNK);
    const size_t pairs = (size_t)R * Hq * nc;
    size_t ml = pairs * sizeof(float2);
    ml = (ml + 255) & ~size_t(255);
    return ml + pairs * D * sizeof(float);
}

// Launch K2 and K3; the caller has validated every argument.
spec_status attn_run(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, float scale, const void *k_cache,
                     const void *v_cache, int num_pages, const int32_t *block_table, int max_blocks,
                     const int32_t *ctx_start, const int32_t *cu_rows, int S, int R, int max_kv_len, void *out,
                     spec_dtype out_dt, void *workspace, int32_t *dev_err, cudaStream_t stream,
                     uint8_t *xpk = nullptr) {
    const int nc_max = (max_kv_len + CHUNK - 1) / CHUNK;
    const size_t pairs = (size_t)R * Hq * nc_max;
    size_t mlb = (pairs * sizeof(float2) + 255) & ~size_t(255);
    float2 *ml = reinterpret_cast<float2 *>(workspace);
    float *po = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + mlb);

    // The caches seen as (d within a 64-wide half, key, half, head, page): one box
    // is a page's 16 keys of one head, both halves (128-byte rows for the swizzle)
    CUtensorMap tk, tv;
    const uint64_t halves = (uint64_t)D / 64;
    uint64_t dims[5] = {64, (uint64_t)PAGE, halves, (uint64_t)Hkv, (uint64_t)num_pages};
    uint64_t strides[4] = {(uint64_t)D * 2, 128, (uint64_t)PAGE * D * 2, (uint64_t)Hkv * PAGE * D * 2};
    uint32_t box[5] = {64, PAGE, (uint32_t)halves, 1, 1};
    if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, k_cache, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, v_cache, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPEC_ERR_CUDA;
    const bool bf = (qkv_dt == SPEC_BF16);
    spec_status st;
    if (D == 128)
        st = bf ? launch_partial<128, true>(tk, tv, q, Hq, Hkv, scale, num_pages, block_table, max_blocks, ctx_start,
                                            cu_rows, S, R, max_kv_len, nc_max, ml, po, dev_err, stream)
                : launch_partial<128, false>(tk, tv, q, Hq, Hkv, scale, num_pages, block_table, max_blocks,
                                             ctx_start, cu_rows, S, R, max_kv_len, nc_max, ml, po, dev_err, stream);
    else
        st = bf ? launch_partial<64, true>(tk, tv, q, Hq, Hkv, scale, num_pages, block_table, max_blocks, ctx_start,
                                           cu_rows, S, R, max_kv_len, nc_max, ml, po, dev_err, stream)
                : launch_partial<64, false>(tk, tv, q, Hq, Hkv, scale, num_pages, block_table, max_blocks, ctx_start,
                                            cu_rows, S, R, max_kv_len, nc_max, ml, po, dev_err, stream);
    if (st != SPEC_OK) return st;
    const int warps = R * Hq * (D / 32);
    dim3 grid((warps + 3) / 4);
    const int kv_cap = (int)std::min<long long>((long long)max_blocks * PAGE, INT_MAX);
    const bool obf = (out_dt == SPEC_BF16);
    // every row within 32 chunks (the bound says so): the short-row instance
    const bool short_rows = max_kv_len <= 32 * CHUNK;
    auto launch_combine = [&](auto kern) {
        return launch_pdl(kern, grid, dim3(128), 0, stream, ctx_start, cu_rows, S, R, Hq, nc_max, (const float2 *)ml,
                          (const float *)po, out, max_kv_len, kv_cap, xpk);
    };
    cudaError_t le;
    if (D == 128) {
        if (obf)
            le = short_rows ? launch_combine(attn_combine_kernel<128, true, true>)
                            : launch_combine(attn_combine_kernel<128, true, false>);
        else
            le = short_rows ? launch_combine(attn_combine_kernel<128, false, true>)
                            : launch_combine(attn_combine_kernel<128, false, false>);
    } else {
        if (obf)
            le = short_rows ? launch_combine(attn_combine_kernel<64, true, true>)
                            : launch_combine(attn_combine_kernel<64, true, false>);
        else
            le = short_rows ? launch_combine(attn_combine_kernel<64, false, true>)
                            : launch_combine(attn_combine_kernel<64, false, false>);
    }
    return cuda_status(le, "attn combine launch");
}

spec_status attn_check(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, const void *k_cache,
                       const void *v_cache, int num_pages, const int32_t *block_table, int max_blocks,
                       const int32_t *ctx_start, const int32_t *cu_rows, int S, int R, int max_kv_len, const void *out,
                       spec_dtype out_dt) {
    SPEC_CHECK_ARG(qkv_dt == SPEC_F16 || qkv_dt == SPEC_BF16, "flash_decode: qkv_dt must be SPEC_F16 or SPEC_BF16");
    SPEC_CHECK_ARG(out_dt == SPEC_F32 || out_dt == SPEC_BF16, "flash_decode: out_dt must be SPEC_F32 or SPEC_BF16");
    SPEC_CHECK_ARG(D == 64 || D == 128, "flash_decode: D must be 64 or 128 (D=%d)", D);
    SPEC_CHECK_ARG(Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && Hq / Hkv <= 16,
                   "flash_decode: need Hq %% Hkv == 0 and Hq / Hkv <= 16 (Hq=%d Hkv=%d)", Hq, Hkv);
    SPEC_CHECK_ARG(S >= 0 && R >= 0 && num_pages >= 1 && max_blocks >= 1 && max_kv_len >= 1,
                   "flash_decode: bad sizes (S=%d R=%d num_pages=%d max_blocks=%d max_kv_len=%d)", S, R, num_pages,
                   max_blocks, max_kv_len);
    SPEC_CHECK_ARG(S <= 65535 && Hkv <= 65535, "flash_decode: S and Hkv must be <= 65535");
    SPEC_CHECK_ARG(q && k_cache && v_cache && block_table && ctx_start && cu_rows && out, "flash_decode: NULL pointer");
    SPEC_CHECK_ARG(aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
                   "flash_decode: q, k_cache and v_cache must be 16-byte aligned");
    return SPEC_OK;
}
}  // namespace spec

extern "C" size_t spec_flash_decode_workspace(int R, int Hq, int D, int max_kv_len) {
    if (R <= 0 || Hq <= 0 || D <= 0 || max_kv_len <= 0) return 0;
    return spec::attn_workspace_bytes(R, Hq, D, max_kv_len);
}

extern "C" spec_status spec_flash_decode(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, float scale,
                                         const void *k_cache, const void *v_cache, int num_pages,
                                         const int32_t *block_table, int max_blocks, const int32_t *ctx_start,
                                         const int32_t *cu_rows, int S, int R, int max_kv_len, void *out,
                                         spec_dtype out_dt, void *workspace, size_t ws_bytes, int32_t *dev_err,
                                         spec_stream_t stream) {
    spec_status st = spec::attn_check(q, qkv_dt, Hq, Hkv, D, k_cache, v_cache, num_pages, block_table, max_blocks,
                                      ctx_start, cu_rows, S, R, max_kv_len, out, out_dt);
    if (st != SPEC_OK) return st;
    if (S == 0 || R == 0) return SPEC_OK;
    const size_t need = spec::attn_workspace_bytes(R, Hq, D, max_kv_len);
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "flash_decode: workspace needs %zu bytes (16-byte aligned), got %zu",
                          need, ws_bytes);
    return spec::attn_run(q, qkv_dt, Hq, Hkv, D, scale, k_cache, v_cache, num_pages, block_table, max_blocks,
                          ctx_start, cu_rows, S, R, max_kv_len, out, out_dt, workspace, dev_err,
                          (cudaStream_t)stream);
}

extern "C" spec_status spec_flash_decode_packed(const void *q, spec_dtype qkv_dt, int Hq, int Hkv, int D, float scale,
                                                const void *k_cache, const void *v_cache, int num_pages,
                                                const int32_t *block_table, int max_blocks, const int32_t *ctx_start,
                                                const int32_t *cu_rows, int S, int R, int max_kv_len, void *out,
                                                void *workspace, size_t ws_bytes, void *xpk, int32_t *dev_err,
                                                spec_stream_t stream) {
    spec_status st = spec::attn_check(q, qkv_dt, Hq, Hkv, D, k_cache, v_cache, num_pages, block_table, max_blocks,
                                      ctx_start, cu_rows, S, R, max_kv_len, out, SPEC_BF16);
    if (st != SPEC_OK) return st;
    SPEC_CHECK_ARG(R <= qmm::WIDE_COLS && (Hq * D) % 256 == 0,
                   "flash_decode_packed: need R <= 80 and Hq * D a multiple of 256 (R=%d Hq*D=%d)", R, Hq * D);
    SPEC_CHECK_ARG(xpk && spec::aligned16(xpk) && spec::aligned16(out),
                   "flash_decode_packed: xpk and out must be non-NULL and 16-byte aligned");
    if (S == 0 || R == 0) return SPEC_OK;
    const size_t need = spec::attn_workspace_bytes(R, Hq, D, max_kv_len);
    if (!workspace || ws_bytes < need || !spec::aligned16(workspace))
        return spec::fail(SPEC_ERR_WORKSPACE, "flash_decode_packed: workspace needs %zu bytes (16-byte aligned), got %zu",
                          need, ws_bytes);
    return spec::attn_run(q, qkv_dt, Hq, Hkv, D, scale, k_cache, v_cache, num_pages, block_table, max_blocks,
                          ctx_start, cu_rows, S, R, max_kv_len, out, SPEC_BF16, workspace, dev_err,
                          (cudaStream_t)stream, reinterpret_cast<uint8_t *>(xpk));
}
