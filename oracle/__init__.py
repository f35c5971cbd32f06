"""CPU oracle (test infrastructure only).

A ctypes front end to ``oracle.c``: the plain, slow, single-threaded,
double-precision definition of every step of the verification hot path.
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library and
never imports it.

Functions take and return numpy arrays in the same storage formats the
library consumes (bf16 / fp16 as uint16 bit patterns, int4 block-32 weights).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

DT_F32, DT_F16, DT_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no FMA contraction) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-Wall", "-shared",
                               "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            c = _lib
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            c.oracle_qmatmul.argtypes = [vp, vp, i32, i32, vp, i32, i32, vp]
            c.oracle_qmatmul_sb.argtypes = [vp, vp, i32, i32, vp, i32, i32, vp]
            c.oracle_margin_gate.argtypes = [vp, i32, i32, vp, vp, vp, vp]
            c.oracle_margin_gate.restype = i32
            c.oracle_sb_record.argtypes = [vp, vp, vp]
            c.oracle_attention.argtypes = [vp, i32, i32, i32, i32, dbl, vp, vp, vp, i32, vp, vp, i32, vp, vp]
            c.oracle_verify_greedy.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp]
            c.oracle_verify_greedy.restype = i32
            u32, f32 = ctypes.c_uint32, ctypes.c_float
            c.oracle_philox4x32_10.argtypes = [vp, vp, vp]
            c.oracle_verify_sample.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, f32, u32, u32, vp, vp, vp, vp, vp]
            c.oracle_verify_sample.restype = i32
            c.oracle_kv_compact.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, vp, vp, vp, i32, vp, vp, vp]
            c.oracle_rmsnorm.argtypes = [vp, i32, vp, dbl, vp]
            c.oracle_rope.argtypes = [vp, i32, i32, dbl]
            c.oracle_silu_mul.argtypes = [dbl, dbl]
            c.oracle_silu_mul.restype = dbl
            c.oracle_decoder_layer.argtypes = ([vp, i32, i32, i32, i32, i32, i32, dbl, dbl] + [vp] * 10
                                               + [vp, vp, vp, i32, vp, vp, i32])
            c.oracle_embed.argtypes = [vp, i32, vp, i32, vp]
            c.oracle_lm_head.argtypes = [vp, i32, i32, vp, dbl, vp, vp, i32, vp]
            c.oracle_ngram_draft.argtypes = [vp, i32, i32, vp, vp]
            c.oracle_ngram_draft.restype = i32
            c.or_bf16_to_double.argtypes = [ctypes.c_uint16]
            c.or_bf16_to_double.restype = dbl
            c.or_f16_to_double.argtypes = [ctypes.c_uint16]
            c.or_f16_to_double.restype = dbl
            c.or_double_to_bf16.argtypes = [dbl]
            c.or_double_to_bf16.restype = ctypes.c_uint16
        return _lib


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


# ---------------------------------------------------------------------------
def f16_to_double(h: int) -> float:
    return lib().or_f16_to_double(int(h))


def bf16_to_double(b: int) -> float:
    return lib().or_bf16_to_double(int(b))


def double_to_bf16(x: float) -> int:
    return int(lib().or_double_to_bf16(float(x)))


def qmatmul(wq, ws, x, N: int, K: int, n_cols: int | None = None, ldx: int | None = None) -> np.ndarray:
    """y[j][n] = sum_k x[j][k] d[n][k/32] q[n][k]; returns float64 [n_cols][N]."""
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint16)
    x = _c(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    n_cols = x.shape[0] if n_cols is None else n_cols
    ldx = x.shape[1] if ldx is None else ldx
    y = np.zeros((n_cols, N), dtype=np.float64)
    lib().oracle_qmatmul(_p(wq), _p(ws), N, K, _p(x), n_cols, ldx, _p(y))
    return y


def sb_pitch(K: int) -> int:
    """Bytes of super-block scale records per weight row: ceil(K/512) pairs of 8-byte records."""
    return (K + 511) // 512 * 16


def sb_record(rec) -> tuple[list[int], float]:
    """Decode one 8-byte super-block record into its eight 6-bit block scales and its fp16 super-scale."""
    rec = _c(np.frombuffer(bytes(rec), dtype=np.uint8), np.uint8)
    assert rec.size == 8
    s = np.zeros(8, dtype=np.int32)
    D = np.zeros(1, dtype=np.float64)
    lib().oracle_sb_record(_p(rec), _p(s), _p(D))
    return [int(v) for v in s], float(D[0])


def qmatmul_sb(wq, sbr, x, N: int, K: int, n_cols: int | None = None, ldx: int | None = None) -> np.ndarray:
    """y[j][n] = sum_k x[j][k] D[n][k/256] s[n][k/32] q[n][k] (two-level scales); float64 [n_cols][N]."""
    wq = _c(wq, np.uint8)
    sbr = _c(sbr, np.uint8)
    x = _c(x, np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    n_cols = x.shape[0] if n_cols is None else n_cols
    ldx = x.shape[1] if ldx is None else ldx
    y = np.zeros((n_cols, N), dtype=np.float64)
    lib().oracle_qmatmul_sb(_p(wq), _p(sbr), N, K, _p(x), n_cols, ldx, _p(y))
    return y


def qmatmul_sb_rows(wq, sbr, x, K: int, rows) -> np.ndarray:
    """qmatmul_sb restricted to output features ``rows``."""
    rows = np.asarray(rows, dtype=np.int64)
    wq_s = _c(np.asarray(wq).reshape(-1, K // 2)[rows], np.uint8)
    sb_s = _c(np.asarray(sbr).reshape(-1, sb_pitch(K))[rows], np.uint8)
    return qmatmul_sb(wq_s, sb_s, x, len(rows), K)


def qmatmul_rows(wq, ws, x, K: int, rows) -> np.ndarray:
    """The same product restricted to output features ``rows`` (rows are independent)."""
    rows = np.asarray(rows, dtype=np.int64)
    wq_s = _c(np.asarray(wq).reshape(-1, K // 2)[rows], np.uint8)
    ws_s = _c(np.asarray(ws).reshape(-1, K // 32)[rows], np.uint16)
    return qmatmul(wq_s, ws_s, x, len(rows), K)


def attention(case=None, *, q=None, dt=None, Hq=None, Hkv=None, D=None, scale=None, k_cache=None,
              v_cache=None, block_table=None, ctx_start=None, cu_rows=None, want=None) -> np.ndarray:
    """Causal softmax attention over the paged cache; returns float64 [R][Hq][D]."""
    if case is not None:
        q, dt, Hq, Hkv, D, scale = case.q, case.dt, case.Hq, case.Hkv, case.D, case.scale
        k_cache, v_cache, block_table = case.k_cache, case.v_cache, case.block_table
        ctx_start, cu_rows = case.ctx_start, case.cu_rows
    bt = _c(block_table, np.int32)
    cu = _c(cu_rows, np.int32)
    ctx = _c(ctx_start, np.int32)
    S = len(ctx)
    R = int(cu[-1])
    qa = _c(q, np.float32 if dt == DT_F32 else np.uint16)
    kc = _c(k_cache, np.float32 if dt == DT_F32 else np.uint16)
    vc = _c(v_cache, np.float32 if dt == DT_F32 else np.uint16)
    w = None if want is None else _c(want, np.uint8)
    out = np.zeros((R, Hq, D), dtype=np.float64)
    lib().oracle_attention(_p(qa), dt, Hq, Hkv, D, float(scale), _p(kc), _p(vc), _p(bt), bt.shape[1],
                           _p(ctx), _p(cu), S, _p(w), _p(out))
    return out


def verify_greedy(logits, dt: int, V: int, cu_rows, drafts, ctx_start):
    """Returns dict(argmax, accepted, correction, ctx_new, nans)."""
    lg = _c(logits, np.float32 if dt == DT_F32 else np.uint16)
    cu = _c(cu_rows, np.int32)
    dr = _c(drafts, np.int32)
    ctx = _c(ctx_start, np.int32)
    S = len(ctx)
    R = int(cu[-1])
    am = np.zeros(R, np.int32)
    acc = np.zeros(S, np.int32)
    cor = np.zeros(S, np.int32)
    cn = np.zeros(S, np.int32)
    if dr.size == 0:
        dr = np.zeros(1, np.int32)
    nans = lib().oracle_verify_greedy(_p(lg), dt, V, _p(cu), S, _p(dr), _p(ctx), _p(am), _p(acc), _p(cor), _p(cn))
    return dict(argmax=am, accepted=acc, correction=cor, ctx_new=cn, nans=int(nans))


def philox4x32_10(counter, key):
    """Philox4x32-10 of four 32-bit counter words and two key words -> four words."""
    ctr = np.asarray(counter, np.uint32).copy()
    k = np.asarray(key, np.uint32).copy()
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(ctr), _p(k), _p(out))
    return out


def verify_sample(logits, dt: int, V: int, cu_rows, drafts, ctx_start, inv_temp: float, seed: int, seq_id=None):
    """Temperature-sampling verification (Gumbel-max with Philox draws keyed by
    sequence and position).  Returns dict(token, accepted, correction, ctx_new,
    top2_gap, nans); top2_gap is each row's winning margin in fp32 scores."""
    lg = _c(logits, np.float32 if dt == DT_F32 else np.uint16)
    cu = _c(cu_rows, np.int32)
    dr = _c(drafts, np.int32)
    ctx = _c(ctx_start, np.int32)
    S = len(ctx)
    R = int(cu[-1])
    tok = np.zeros(R, np.int32)
    acc = np.zeros(S, np.int32)
    cor = np.zeros(S, np.int32)
    cn = np.zeros(S, np.int32)
    gap = np.zeros(R, np.float32)
    if dr.size == 0:
        dr = np.zeros(1, np.int32)
    sid = None if seq_id is None else _c(seq_id, np.int32)
    nans = lib().oracle_verify_sample(_p(lg), dt, V, _p(cu), S, _p(dr), _p(ctx), _p(sid), float(inv_temp),
                                      seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF,
                                      _p(tok), _p(acc), _p(cor), _p(cn), _p(gap))
    return dict(token=tok, accepted=acc, correction=cor, ctx_new=cn, top2_gap=gap, nans=int(nans))


def margin_gate(logits, err):
    """Top-2 margin gate over fp32 logits [R][V] with per-row error bounds err[R]:
    returns (top index [R], margin [R], recheck flags [R] as bool)."""
    lg = _c(logits, np.float32)
    R, V = lg.shape
    e = _c(np.broadcast_to(np.asarray(err, np.float64), (R,)), np.float64)
    top = np.zeros(R, np.int32)
    margin = np.zeros(R, np.float64)
    flag = np.zeros(R, np.uint8)
    lib().oracle_margin_gate(_p(lg), R, V, _p(e), _p(top), _p(margin), _p(flag))
    return top, margin, flag.astype(bool)


def kv_compact(k_stage, v_stage, k_cache, v_cache, Hkv, D, block_table, ctx_start, accepted, cu_rows):
    """Returns (k_cache', v_cache', cu_kept, kept_src, dst_slot); caches are copied, not modified."""
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    ks = None if k_stage is None else _c(k_stage, np.uint16)
    vs = None if v_stage is None else _c(v_stage, np.uint16)
    bt = _c(block_table, np.int32)
    ctx = _c(ctx_start, np.int32)
    acc = _c(accepted, np.int32)
    cu = _c(cu_rows, np.int32)
    S = len(ctx)
    n_kept = int((acc + 1).sum())
    cuk = np.zeros(S + 1, np.int32)
    src = np.zeros(max(n_kept, 1), np.int32)
    dst = np.zeros(max(n_kept, 1), np.int64)
    lib().oracle_kv_compact(_p(ks), _p(vs), _p(kc), _p(vc), Hkv, D, _p(bt), bt.shape[1], _p(ctx), _p(acc),
                            _p(cu), S, _p(cuk), _p(src), _p(dst))
    return kc, vc, cuk, src[:n_kept], dst[:n_kept]


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _c(x, np.float64)
    w = _c(w, np.float32)
    y = np.zeros_like(x)
    lib().oracle_rmsnorm(_p(x), x.size, _p(w), float(eps), _p(y))
    return y


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True, order="C")
    lib().oracle_rope(_p(v), v.size, int(pos), float(theta))
    return v


def silu_mul(g: float, u: float) -> float:
    return lib().oracle_silu_mul(float(g), float(u))


def ngram_draft(hist, W: int, pad):
    """Returns (proposed tokens [W], matched n-gram length)."""
    h = _c(hist, np.int32)
    pd = _c(pad, np.int32)
    out = np.zeros(W, np.int32)
    n = lib().oracle_ngram_draft(_p(h) if h.size else _p(np.zeros(1, np.int32)), h.size, W, _p(pd), _p(out))
    return out, int(n)


# ---------------------------------------------------------------------------
# decoder (random-init) built from the pieces above
# ---------------------------------------------------------------------------
class Decoder:
    """Single-threaded CPU decoder over a paged bf16 KV cache.

    Holds its own cache; ``forward`` appends the block rows' K/V at their
    positions and returns fp32 logits for every row.
    """

    def __init__(self, weights, n_seqs: int, max_len: int):
        self.w = weights
        cfg = weights.cfg
        self.cfg = cfg
        self.max_blocks = (max_len + 15) // 16
        pages = n_seqs * self.max_blocks
        self.block_table = np.arange(pages, dtype=np.int32).reshape(n_seqs, self.max_blocks)
        self.k_cache = [np.zeros((pages, cfg.kv_heads, 16, cfg.head_dim), np.uint16) for _ in range(cfg.layers)]
        self.v_cache = [np.zeros((pages, cfg.kv_heads, 16, cfg.head_dim), np.uint16) for _ in range(cfg.layers)]

    def layer(self, li: int, h: np.ndarray, ctx_start, cu_rows, seqs=None) -> np.ndarray:
        """Apply decoder layer ``li`` in place to h (float32 [R][H]).  ``seqs`` maps
        batch sequence index -> cache row (defaults to identity)."""
        cfg, lay = self.cfg, self.w.layers[li]
        bt = self.block_table if seqs is None else _c(self.block_table[np.asarray(seqs)], np.int32)
        ctx = _c(ctx_start, np.int32)
        cu = _c(cu_rows, np.int32)
        h = np.ascontiguousarray(h, dtype=np.float32)
        ptrs = [lay["qkv"][0], lay["qkv"][1], lay["o"][0], lay["o"][1], lay["gu"][0], lay["gu"][1],
                lay["down"][0], lay["down"][1], lay["norm1"], lay["norm2"]]
        ptrs = [np.ascontiguousarray(p) for p in ptrs]
        lib().oracle_decoder_layer(_p(h), h.shape[0], cfg.hidden, cfg.heads, cfg.kv_heads, cfg.head_dim, cfg.ffn,
                                   cfg.eps, cfg.rope_theta, *[_p(p) for p in ptrs],
                                   _p(self.k_cache[li]), _p(self.v_cache[li]), _p(bt), bt.shape[1],
                                   _p(ctx), _p(cu), len(ctx))
        return h

    def embed(self, tokens) -> np.ndarray:
        t = _c(tokens, np.int32)
        h = np.zeros((t.size, self.cfg.hidden), np.float32)
        lib().oracle_embed(_p(self.w.emb), self.cfg.hidden, _p(t), t.size, _p(h))
        return h

    def lm_head(self, h) -> np.ndarray:
        h = _c(h, np.float32)
        R = h.shape[0]
        logits = np.zeros((R, self.cfg.vocab), np.float32)
        lm_q, lm_s = self.w.lm
        lib().oracle_lm_head(_p(h), R, self.cfg.hidden, _p(self.w.final_norm), self.cfg.eps,
                             _p(lm_q), _p(lm_s), self.cfg.vocab, _p(logits))
        return logits

    def forward(self, tokens, ctx_start, cu_rows, seqs=None) -> np.ndarray:
        h = self.embed(tokens)
        for li in range(self.cfg.layers):
            h = self.layer(li, h, ctx_start, cu_rows, seqs)
        return self.lm_head(h)


def generate(weights, prompts_arr, n_new: int, draft_width: int, pads, inv_temp: float = 0.0, seed: int = 0):
    """Greedy generation with the oracle decoder (inv_temp > 0: temperature
    sampling through verify_sample, draws keyed by sequence and position).

    draft_width == 0: ordinary decoding, one row per sequence per step.
    draft_width  > 0: speculative decoding; each step verifies the last token
    plus draft_width n-gram drafts per sequence and keeps the accepted prefix
    and the correction token, truncated at n_new tokens.
    Returns (tokens [S][n_new], steps, accepted_total).
    """
    S, P = prompts_arr.shape
    dec = Decoder(weights, S, P + n_new + draft_width + 1)
    V = weights.cfg.vocab
    hist = [list(map(int, prompts_arr[s])) for s in range(S)]
    # prefill all but the last prompt token; the last one opens the first verify block
    cu = np.arange(S + 1, dtype=np.int32) * (P - 1)
    dec.forward(prompts_arr[:, :P - 1].reshape(-1), np.zeros(S, np.int32), cu)
    ctx = np.full(S, P - 1, np.int32)
    out = [[] for _ in range(S)]
    steps = 0
    acc_total = 0
    while min(len(o) for o in out) < n_new:
        live = [s for s in range(S) if len(out[s]) < n_new]
        toks, rows, drafts = [], [], []
        for s in live:
            block = [hist[s][-1]]
            if draft_width:
                d, _ = ngram_draft(hist[s], draft_width, pads[s, steps % pads.shape[1]])
                block += list(map(int, d))
                drafts += list(map(int, d))
            toks += block
            rows.append(len(block))
        cu = np.zeros(len(live) + 1, np.int32)
        cu[1:] = np.cumsum(rows)
        lg = dec.forward(np.array(toks, np.int32), ctx[live], cu, seqs=live)
        if inv_temp > 0:
            res = verify_sample(lg, DT_F32, V, cu, np.array(drafts, np.int32), ctx[live], inv_temp, seed,
                                seq_id=np.array(live, np.int32))
        else:
            res = verify_greedy(lg, DT_F32, V, cu, np.array(drafts, np.int32), ctx[live])
        for k, s in enumerate(live):
            a = int(res["accepted"][k])
            acc_total += a
            new = drafts[k * draft_width:k * draft_width + a] if draft_width else []
            new = list(new) + [int(res["correction"][k])]
            new = new[:n_new - len(out[s])]
            out[s] += new
            hist[s] += new
            ctx[s] = int(res["ctx_new"][k])
        steps += 1
    return np.array(out, np.int32), steps, acc_total
