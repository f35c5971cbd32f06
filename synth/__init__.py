"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module only *makes inputs*: random draws, encodings of those draws into the
storage formats the library consumes (bf16 / fp16 bit patterns, int4 block-32
weights, paged KV caches with shuffled block tables) and data with a known,
constructed answer (logit rows whose top index is planted).  It implements
none of the verified computation: no matmul, no attention, no argmax, no
acceptance rule, no compaction, no drafting.  Both the CUDA path and the CPU
oracle consume exactly the same bytes from here.

Workload recipes (seeded with ``numpy.random.default_rng``):

* int4 block-32 weights: w ~ N(0, 0.02), one fp16 scale per 32 consecutive
  weights of a row, d = fp16(max|w| / 7), q = clamp(rint(w / d), -8, 7),
  stored as the nibble q + 8 with even k in the low nibble.  The pages name
  block quantisation but define no format; this symmetric round-to-nearest
  format is the stand-in.
* activations: bf16 ~ N(0, 1).
* attention: paged K/V cache [pages][Hkv][16][D], pages handed out in shuffled
  order, unused cache slots filled with NaN bit patterns so that a kernel that
  reads past a sequence's length shows it.
* verify: logits ~ N(0, sigma) with a planted top index per row, a fraction of
  rows with a planted runner-up (1e-6 below in fp32; one bf16 ulp below or an
  exact tie at a higher index in bf16), drafts that copy the planted top with
  probability 0.7 and are otherwise uniform.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE = 16  # tokens per KV page

DT_F32, DT_F16, DT_BF16 = 0, 1, 2


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# storage encodings
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_f16_bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32).astype(np.float16)).view(np.uint16)


def f16_bits_to_f32(h) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(h, dtype=np.uint16)).view(np.float16).astype(np.float32)


def quantize_q4b32(w) -> tuple[np.ndarray, np.ndarray]:
    """Encode a float32 [N][K] matrix as int4 block-32 weights.

    Returns (wq uint8 [N][K/2], ws uint16 fp16 bits [N][K/32]).
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 32 == 0
    blocks = w.reshape(N, K // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    d16 = (amax / np.float32(7.0)).astype(np.float16)
    d = d16.astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    q = np.rint(blocks / safe[:, :, None])
    q = np.clip(q, -8, 7)
    q[d == 0] = 0
    nib = (q.astype(np.int32) + 8).astype(np.uint8).reshape(N, K)
    wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(wq), np.ascontiguousarray(d16.view(np.uint16))


def pack_q4(q, scales_f32) -> tuple[np.ndarray, np.ndarray]:
    """Pack explicit integer codes q in [-8, 7] ([N][K]) and per-block scales ([N][K/32])."""
    q = np.asarray(q, dtype=np.int32)
    assert q.min() >= -8 and q.max() <= 7
    N, K = q.shape
    nib = (q + 8).astype(np.uint8)
    wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    ws = f32_to_f16_bits(np.asarray(scales_f32, dtype=np.float32).reshape(N, K // 32))
    return np.ascontiguousarray(wq), ws


# ---------------------------------------------------------------------------
# quantised matmul inputs
# ---------------------------------------------------------------------------
@dataclass
class QMatmulCase:
    N: int
    K: int
    wq: np.ndarray  # uint8 [N][K/2]
    ws: np.ndarray  # uint16 [N][K/32]
    x: np.ndarray   # uint16 bf16 bits [n_cols][ldx]
    n_cols: int
    ldx: int


def qmatmul_weights(seed: int, N: int, K: int, std: float = 0.02):
    g = rng(seed)
    w = g.normal(0.0, std, size=(N, K)).astype(np.float32)
    return quantize_q4b32(w)


def activations_bf16(seed: int, n_cols: int, K: int, ldx: int | None = None, std: float = 1.0):
    g = rng(seed)
    ldx = K if ldx is None else ldx
    x = np.zeros((n_cols, ldx), dtype=np.float32)
    x[:, :K] = g.normal(0.0, std, size=(n_cols, K)).astype(np.float32)
    return f32_to_bf16_bits(x)


def pack_sb_records(s, D16) -> np.ndarray:
    """Pack 6-bit block scales s ([N][K/32], 0..63) and fp16 super-scales D16 (uint16 bits,
    [N][K/256]) into the super-block record layout: per row ceil(K/512) pairs of 8-byte
    little-endian words, s_j at bits 6j, D at bits 48..63, the unused last record zero."""
    s = np.asarray(s, dtype=np.uint64)
    D16 = np.asarray(D16, dtype=np.uint16)
    N, nb = s.shape
    nsb = nb // 8
    assert D16.shape == (N, nsb) and s.max(initial=0) <= 63
    words = np.zeros((N, (nsb + 1) // 2 * 2), dtype=np.uint64)
    sj = s.reshape(N, nsb, 8)
    for j in range(8):
        words[:, :nsb] |= sj[:, :, j] << np.uint64(6 * j)
    words[:, :nsb] |= D16.astype(np.uint64) << np.uint64(48)
    return np.ascontiguousarray(words.astype("<u8").view(np.uint8))


def quantize_q4_superblock(w) -> tuple[np.ndarray, np.ndarray]:
    """Encode float32 [N][K] (K % 256 == 0) as 4-bit codes with two-level scales: per 256-k
    super-block an fp16 D = max block scale / 63, per 32-k block s = round(block scale / D)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 256 == 0
    blocks = w.reshape(N, K // 32, 32)
    want = np.abs(blocks).max(axis=2) / np.float32(7.0)               # ideal block scales
    D16 = (want.reshape(N, K // 256, 8).max(axis=2) / np.float32(63.0)).astype(np.float16)
    D = np.repeat(D16.astype(np.float32), 8, axis=1)
    s = np.where(D > 0, np.clip(np.rint(want / np.where(D > 0, D, 1)), 0, 63), 0).astype(np.int64)
    d = D * s
    safe = np.where(d == 0, np.float32(1.0), d)
    q = np.clip(np.rint(blocks / safe[:, :, None]), -8, 7)
    q[d == 0] = 0
    nib = (q.astype(np.int32) + 8).astype(np.uint8).reshape(N, K)
    wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(wq), pack_sb_records(s, D16.view(np.uint16))


def qmatmul_sb_case(seed: int, N: int, K: int, n_cols: int, ldx: int | None = None) -> QMatmulCase:
    """A QMatmulCase whose ``ws`` holds super-block scale records (uint8 [N][ceil(K/512)*16])."""
    g = rng(seed)
    wq, sbr = quantize_q4_superblock(g.normal(0.0, 0.02, size=(N, K)).astype(np.float32))
    x = activations_bf16(seed + 7919, n_cols, K, ldx)
    return QMatmulCase(N, K, wq, sbr, x, n_cols, x.shape[1])


def qmatmul_case(seed: int, N: int, K: int, n_cols: int, ldx: int | None = None) -> QMatmulCase:
    wq, ws = qmatmul_weights(seed, N, K)
    x = activations_bf16(seed + 7919, n_cols, K, ldx)
    return QMatmulCase(N, K, wq, ws, x, n_cols, x.shape[1])


# ---------------------------------------------------------------------------
# paged attention inputs
# ---------------------------------------------------------------------------
@dataclass
class AttentionCase:
    Hq: int
    Hkv: int
    D: int
    dt: int                 # DT_F16 or DT_BF16
    q: np.ndarray           # uint16 [R][Hq][D]
    k_cache: np.ndarray     # uint16 [pages][Hkv][16][D]
    v_cache: np.ndarray
    block_table: np.ndarray  # int32 [S][max_blocks], -1 where unused
    ctx_start: np.ndarray   # int32 [S]
    cu_rows: np.ndarray     # int32 [S+1]
    scale: float

    @property
    def S(self):
        return len(self.ctx_start)

    @property
    def R(self):
        return int(self.cu_rows[-1])

    @property
    def max_blocks(self):
        return self.block_table.shape[1]

    @property
    def max_kv_len(self):
        return int(max(self.ctx_start + np.diff(self.cu_rows)))


def _encode(vals, dt):
    return f32_to_f16_bits(vals) if dt == DT_F16 else f32_to_bf16_bits(vals)


def paged_layout(g: np.random.Generator, lens, extra_pages: int = 3, max_blocks: int | None = None):
    """Shuffled page assignment for sequences of the given lengths (tokens)."""
    need = [(int(L) + PAGE - 1) // PAGE for L in lens]
    total = sum(need) + extra_pages
    perm = g.permutation(total).astype(np.int32)
    mb = max(need) if max_blocks is None else max_blocks
    assert mb >= max(need)
    bt = np.full((len(lens), mb), -1, dtype=np.int32)
    o = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[o:o + n]
        o += n
    return bt, total


def attention_case(seed: int, rows, ctx, Hq: int, Hkv: int, D: int, dt: int = DT_BF16,
                   q_std: float = 1.0, scale: float | None = None, poison: bool = True) -> AttentionCase:
    """rows[s] query rows of sequence s sit at positions ctx[s] .. ctx[s]+rows[s]-1.

    The cache holds keys for positions 0 .. ctx[s]+rows[s]-1 (the block's own
    keys already appended).  Slots past a sequence's length hold NaN.
    """
    g = rng(seed)
    rows = np.asarray(rows, dtype=np.int32)
    ctx = np.asarray(ctx, dtype=np.int32)
    lens = ctx + rows
    bt, pages = paged_layout(g, lens)
    kc = g.normal(0.0, 1.0, size=(pages, Hkv, PAGE, D)).astype(np.float32)
    vc = g.normal(0.0, 1.0, size=(pages, Hkv, PAGE, D)).astype(np.float32)
    if poison:
        used = np.zeros((pages, PAGE), dtype=bool)
        for s, L in enumerate(lens):
            for j in range(int(L)):
                used[bt[s, j // PAGE], j % PAGE] = True
        kc[~used[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)] = np.nan
        vc[~used[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)] = np.nan
    R = int(rows.sum())
    q = (g.normal(0.0, 1.0, size=(R, Hq, D)) * q_std).astype(np.float32)
    cu = np.zeros(len(rows) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(rows)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return AttentionCase(Hq, Hkv, D, dt, _encode(q, dt), _encode(kc, dt), _encode(vc, dt),
                         bt, ctx, cu, float(scale))


# ---------------------------------------------------------------------------
# greedy verify inputs
# ---------------------------------------------------------------------------
@dataclass
class VerifyCase:
    V: int
    dt: int                 # DT_F32 or DT_BF16
    logits: np.ndarray      # float32 [R][V] or uint16 bf16 bits [R][V]
    cu_rows: np.ndarray     # int32 [S+1]
    drafts: np.ndarray      # int32 [R - S]
    ctx_start: np.ndarray   # int32 [S]
    planted_top: np.ndarray  # int32 [R] index planted as the row maximum
    tie_rows: np.ndarray    # bool [R]

    @property
    def S(self):
        return len(self.ctx_start)

    @property
    def R(self):
        return int(self.cu_rows[-1])


def verify_case(seed: int, draft_lens, V: int, dt: int = DT_F32, sigma: float = 1.0,
                tie_frac: float = 0.1, p_match: float = 0.7, ctx_range=(256, 8192)) -> VerifyCase:
    """Sequence s has draft_lens[s] drafts and draft_lens[s]+1 verify rows."""
    g = rng(seed)
    L = np.asarray(draft_lens, dtype=np.int32)
    S = len(L)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(L + 1)
    R = int(cu[-1])
    vals = g.normal(0.0, sigma, size=(R, V)).astype(np.float32)
    top = g.integers(0, V, size=R).astype(np.int32)
    ties = g.random(R) < tie_frac
    # planted top: strictly above every other entry of the row
    rowmax = vals.max(axis=1)
    vals[np.arange(R), top] = rowmax + np.float32(0.25 * sigma) + np.abs(g.normal(0.0, 0.5 * sigma, size=R)).astype(np.float32)
    if dt == DT_BF16:
        bits = f32_to_bf16_bits(vals)
        # rounding can only merge values; re-plant the top one bf16 ulp above the row's rounded max
        for r in range(R):
            row = bf16_bits_to_f32(bits[r])
            others = np.delete(row, top[r])
            m = others.max()
            if row[top[r]] <= m:
                bits[r, top[r]] = _bf16_next_up(f32_to_bf16_bits(np.array([m]))[0])
        for r in np.nonzero(ties)[0]:
            t = int(top[r])
            if t == V - 1:
                continue
            u = int(g.integers(t + 1, V))
            if r % 2 == 0:
                bits[r, u] = _bf16_next_down(bits[r, t])      # one bf16 ulp below
            else:
                bits[r, u] = bits[r, t]                       # exact tie at a higher index
        logits = bits
    else:
        for r in np.nonzero(ties)[0]:
            t = int(top[r])
            if t == V - 1:
                continue
            u = int(g.integers(t + 1, V))
            vals[r, u] = np.float32(vals[r, t] - np.float32(1e-6))
        logits = vals
    drafts = np.zeros(R - S, dtype=np.int32)
    for s in range(S):
        for i in range(int(L[s])):
            row = cu[s] + i
            if g.random() < p_match:
                drafts[cu[s] - s + i] = top[row]
            else:
                drafts[cu[s] - s + i] = int(g.integers(0, V))
    ctx = g.integers(ctx_range[0], ctx_range[1] + 1, size=S).astype(np.int32)
    return VerifyCase(V, dt, np.ascontiguousarray(logits), cu, drafts, ctx, top, ties)


def verify_case_natural(seed: int, draft_lens, V: int, sigma: float = 2.0, tie_frac: float = 0.01,
                        edges=(), ctx_range=(256, 8192)) -> VerifyCase:
    """bf16 logits whose row maxima are decided by the raw N(0, sigma) draws (no
    planted top), with planted competitors on a tie_frac share of the rows.  A
    planted row copies its largest value v (first occurrence at p) to another
    index t, chosen in turn as: an exact tie at a lower index t < p; the same at
    the element just before one of `edges` (a scan-split boundary of the
    consumer) with p moved to just after it; a value one bf16 ulp below v at a
    lower index; an exact tie at a higher index.  `planted_top` is -1 (the
    answer is left to the oracle) and the drafts are uniform random tokens
    (tests derive matching drafts from the oracle's answer)."""
    g = rng(seed)
    L = np.asarray(draft_lens, dtype=np.int32)
    S = len(L)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(L + 1)
    R = int(cu[-1])
    bits = f32_to_bf16_bits(g.normal(0.0, sigma, size=(R, V)).astype(np.float32))
    ties = g.random(R) < tie_frac
    edges = [int(e) for e in edges if 0 < int(e) < V]
    kind = 0
    for r in np.nonzero(ties)[0]:
        row = bf16_bits_to_f32(bits[r])
        p = int(np.argmax(row))            # first occurrence of the row's largest value
        top = bits[r, p]
        k = kind % 4
        kind += 1
        if k == 1 and edges:
            e = edges[(kind // 4) % len(edges)]
            # move the maximum to just after the boundary, its exact copy to just before it
            bits[r, p] = bits[r, e]
            bits[r, e] = top
            bits[r, e - 1] = top
        elif k == 0 or k == 1:
            if p > 0:
                bits[r, int(g.integers(0, p))] = top
        elif k == 2:
            if p > 0:
                bits[r, int(g.integers(0, p))] = _bf16_next_down(top)
        else:
            if p < V - 1:
                bits[r, int(g.integers(p + 1, V))] = top
    drafts = g.integers(0, V, size=R - S).astype(np.int32)
    ctx = g.integers(ctx_range[0], ctx_range[1] + 1, size=S).astype(np.int32)
    return VerifyCase(V, DT_BF16, np.ascontiguousarray(bits), cu, drafts, ctx, np.full(R, -1, np.int32), ties)


def _bf16_next_down(b):
    b = int(b)
    if b & 0x8000:
        return np.uint16(b + 1)
    if b == 0:
        return np.uint16(0x8001)
    return np.uint16(b - 1)


def _bf16_next_up(b):
    b = int(b)
    if b & 0x8000:
        return np.uint16(b - 1) if b != 0x8000 else np.uint16(1)
    return np.uint16(b + 1)


# ---------------------------------------------------------------------------
# KV compaction inputs
# ---------------------------------------------------------------------------
@dataclass
class CompactCase:
    Hkv: int
    D: int
    k_stage: np.ndarray     # uint16 [R][Hkv][D]
    v_stage: np.ndarray
    k_cache: np.ndarray     # uint16 [pages][Hkv][16][D]
    v_cache: np.ndarray
    block_table: np.ndarray  # int32 [S][max_blocks]
    ctx_start: np.ndarray   # int32 [S]
    accepted: np.ndarray    # int32 [S]
    cu_rows: np.ndarray     # int32 [S+1]

    @property
    def S(self):
        return len(self.ctx_start)

    @property
    def R(self):
        return int(self.cu_rows[-1])


def compact_case(seed: int, draft_lens, Hkv: int, D: int, ctx_range=(256, 8192),
                 accepted=None) -> CompactCase:
    g = rng(seed)
    L = np.asarray(draft_lens, dtype=np.int32)
    S = len(L)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(L + 1)
    R = int(cu[-1])
    ctx = g.integers(ctx_range[0], ctx_range[1] + 1, size=S).astype(np.int32)
    if accepted is None:
        acc = np.array([int(g.integers(0, int(l) + 1)) for l in L], dtype=np.int32)
    else:
        acc = np.asarray(accepted, dtype=np.int32)
    bt, pages = paged_layout(g, ctx + L + 1)
    ks = f32_to_bf16_bits(g.normal(0.0, 1.0, size=(R, Hkv, D)).astype(np.float32))
    vs = f32_to_bf16_bits(g.normal(0.0, 1.0, size=(R, Hkv, D)).astype(np.float32))
    kc = f32_to_bf16_bits(g.normal(0.0, 1.0, size=(pages, Hkv, PAGE, D)).astype(np.float32))
    vc = f32_to_bf16_bits(g.normal(0.0, 1.0, size=(pages, Hkv, PAGE, D)).astype(np.float32))
    return CompactCase(Hkv, D, ks, vs, kc, vc, bt, ctx, acc, cu)


# ---------------------------------------------------------------------------
# decoder (random init) for the end-to-end greedy generation workload
# ---------------------------------------------------------------------------
@dataclass
class DecoderConfig:
    layers: int = 8
    hidden: int = 2048
    heads: int = 16
    kv_heads: int = 4
    head_dim: int = 128
    ffn: int = 5632
    vocab: int = 32000
    eps: float = 1e-5
    rope_theta: float = 10000.0


TINY_DECODER = DecoderConfig(layers=2, hidden=64, heads=4, kv_heads=2, head_dim=16, ffn=128, vocab=97)
E2E_DECODER = DecoderConfig()


@dataclass
class DecoderWeights:
    cfg: DecoderConfig
    emb: np.ndarray                       # uint16 bf16 [V][H]
    layers: list = field(default_factory=list)  # dicts of (wq, ws) pairs: qkv, o, gu, down; norm weights
    lm: tuple = None                      # (wq, ws) [V][H]
    final_norm: np.ndarray = None         # float32 [H]


def decoder_weights(seed: int, cfg: DecoderConfig, std: float = 0.02) -> DecoderWeights:
    """Random-init weights.  qkv rows are [q (Hq*D) | k (Hkv*D) | v (Hkv*D)],
    gate/up rows are [gate (F) | up (F)]; every linear is int4 block-32."""
    g = rng(seed)
    H, D = cfg.hidden, cfg.head_dim
    emb = f32_to_bf16_bits(g.normal(0.0, std, size=(cfg.vocab, H)).astype(np.float32))
    layers = []
    for _ in range(cfg.layers):
        nq = (cfg.heads + 2 * cfg.kv_heads) * D
        lay = {
            "qkv": quantize_q4b32(g.normal(0.0, std, size=(nq, H)).astype(np.float32)),
            "o": quantize_q4b32(g.normal(0.0, std, size=(H, cfg.heads * D)).astype(np.float32)),
            "gu": quantize_q4b32(g.normal(0.0, std, size=(2 * cfg.ffn, H)).astype(np.float32)),
            "down": quantize_q4b32(g.normal(0.0, std, size=(H, cfg.ffn)).astype(np.float32)),
            "norm1": np.ones(H, dtype=np.float32),
            "norm2": np.ones(H, dtype=np.float32),
        }
        layers.append(lay)
    lm = quantize_q4b32(g.normal(0.0, std, size=(cfg.vocab, H)).astype(np.float32))
    return DecoderWeights(cfg, emb, layers, lm, np.ones(H, dtype=np.float32))


def prompts(seed: int, n_seqs: int, length: int, vocab: int) -> np.ndarray:
    return rng(seed).integers(0, vocab, size=(n_seqs, length)).astype(np.int32)


def pad_tokens(seed: int, n_seqs: int, n_steps: int, width: int, vocab: int) -> np.ndarray:
    """Random filler tokens for draft slots the n-gram lookup leaves empty."""
    return rng(seed).integers(0, vocab, size=(n_seqs, n_steps, width)).astype(np.int32)
