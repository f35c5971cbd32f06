"""End-to-end greedy generation on a random-init decoder, driven entirely by
libspec kernels: the target forward (int4 linears, RMSNorm, RoPE, paged
attention, SwiGLU), greedy verification, KV realignment, n-gram drafting and
the history update all run on the device; one speculative step needs no host
round trip and is captured in a CUDA graph.

The model is the workload's stand-in: the pages run real decoders with real
weights, which are out of reach here (ramgpt.org, "When Lossless Speculation
Stops Being Lossless on Blackwell", section "Why Tiny Numerical Differences Can
Change Entire Answers": byte-identical speculative vs non-speculative output is
the user-facing test).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _lib as L


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a.copy()).to(device)


def margin_gate_coef(scales, K: int) -> float:
    """The margin gate's summation-order bound per unit ||x||_1 for an int4 block-32
    matrix with fp16 scales `scales` (raw bits) and K inputs: two fp32 evaluations
    of its n = K/32 block terms differ by at most 2 gamma_(2n) sum |t_b|, and
    |t_b| <= 9 max|d| ||x_b||_1 (|q| <= 8, plus the rounding of the block partial)."""
    n_blk = K // 32
    u = 2.0 ** -24
    gamma = 2 * n_blk * u / (1 - 2 * n_blk * u)
    d_max = float(np.abs(np.asarray(scales, np.uint16).view(np.float16).astype(np.float64)).max())
    return 2 * gamma * 9 * d_max


class Decoder:
    """Device-resident decoder: weights, paged KV cache, activation buffers.

    ``weights`` is a ``synth.DecoderWeights``-like object (cfg, emb, layers, lm,
    final_norm) in storage formats.  Each sequence owns max_len / 16 private
    pages; the block table is contiguous per sequence.
    """

    def __init__(self, weights, n_seqs: int, max_len: int, max_rows: int, device="cuda"):
        cfg = weights.cfg
        self.cfg, self.S, self.device = cfg, n_seqs, device
        self.H, self.Hq, self.Hkv, self.D, self.F, self.V = (cfg.hidden, cfg.heads, cfg.kv_heads, cfg.head_dim,
                                                             cfg.ffn, cfg.vocab)
        self.nqkv = (self.Hq + 2 * self.Hkv) * self.D
        self.max_len = max_len
        self.max_blocks = (max_len + 15) // 16
        self.pages = n_seqs * self.max_blocks
        self.emb = _dev(weights.emb, device)
        self.layers = []
        for lay in weights.layers:
            self.layers.append({k: (tuple(_dev(a, device) for a in v) if isinstance(v, tuple) else _dev(v, device))
                                for k, v in lay.items()})
        # the gate/up rows interleaved for spec_qmatmul_swiglu: per group of 8
        # features its 8 gate rows, then their 8 up rows
        F = self.F
        if F % 8 == 0:
            g = torch.arange(F // 8, device=device).view(-1, 1) * 8 + torch.arange(8, device=device).view(1, -1)
            perm = torch.cat([g, g + F], dim=1).reshape(-1)
            for lay in self.layers:
                wq, ws = lay["gu"]
                lay["gu_il"] = (wq.index_select(0, perm).contiguous(), ws.index_select(0, perm).contiguous())
        self.lm = tuple(_dev(a, device) for a in weights.lm)
        self.final_norm = _dev(weights.final_norm, device)
        self.block_table = torch.arange(self.pages, dtype=torch.int32, device=device).view(n_seqs, self.max_blocks)
        shape = (self.pages, self.Hkv, 16, self.D)
        self.k_cache = [torch.zeros(shape, dtype=torch.int16, device=device) for _ in range(cfg.layers)]
        self.v_cache = [torch.zeros(shape, dtype=torch.int16, device=device) for _ in range(cfg.layers)]
        self.gate_coef = margin_gate_coef(weights.lm[1], cfg.hidden)
        self.gate = None
        self.rope = torch.empty((max_len, self.D // 2, 2), dtype=torch.float32, device=device)
        L.spec_rope_table(self.rope, max_len, self.D, cfg.rope_theta)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self._alloc(max_rows)

    def _alloc(self, R):
        d, H, F = self.device, self.H, self.F
        self.max_rows = R
        self.h = torch.zeros((R, H), dtype=torch.float32, device=d)
        self.a = torch.zeros((R, H), dtype=torch.int16, device=d)       # normed rows entering a matmul
        self.act = torch.zeros((R, F), dtype=torch.int16, device=d)     # SwiGLU output rows
        self.qkv = torch.zeros((R, self.nqkv), dtype=torch.float32, device=d)
        self.q = torch.zeros((R, self.Hq, self.D), dtype=torch.int16, device=d)
        self.attn = torch.zeros((R, self.Hq * self.D), dtype=torch.int16, device=d)
        self.gu = torch.zeros((R, 2 * F), dtype=torch.float32, device=d)
        self.logits = torch.zeros((R, self.V), dtype=torch.float32, device=d)
        self.ws_bytes = L.spec_flash_decode_workspace(R, self.Hq, self.D, self.max_len)
        self.attn_ws = torch.empty(self.ws_bytes // 4 + 64, dtype=torch.float32, device=d)
        shapes = [(self.nqkv, H), (H, self.Hq * self.D), (2 * F, H), (H, F), (self.V, H)]
        self.qws_bytes = max(L.spec_qmatmul_workspace(N, K, R) for N, K in shapes)
        self.qws = torch.zeros(self.qws_bytes // 4 + 64, dtype=torch.int32, device=d)   # zero once; calls keep it so
        # an 80-column K1 pass's activations, packed by the producing kernel (RMSNorm, SwiGLU)
        xpk_bytes = max(L.spec_packed_activation_bytes(k) for k in (H, F, self.Hq * self.D))
        self.xpk = torch.empty(xpk_bytes // 4 + 16, dtype=torch.int32, device=d)
        self._plans = {}   # (N, K, rows) -> the 80-column pass is the plan (spec_qmatmul_plan)

    @staticmethod
    def _packed(R):
        """Rows that make one 80-column K1 pass: their producers write the packed form."""
        return 16 < R <= 80

    # ------------------------------------------------------------------
    def embed(self, tokens, R):
        L.spec_embed(self.emb, self.V, self.H, tokens, R, self.h, self.dev_err)

    def layer(self, li, R, cu_rows, ctx, S, max_kv_len=None, trace=None):
        """Decoder layer li over R rows.  ``trace(name)``, if given, is called after
        each step (norm1, qkv, rope, attn, o, norm2, gu, swiglu, down) so a caller
        can read the step's output buffer; it launches nothing itself."""
        lay, H, F, D = self.layers[li], self.H, self.F, self.D
        max_kv_len = max_kv_len or self.max_len
        tr = trace or (lambda name: None)
        pk = self._packed(R)
        # which matmuls run the 80-column pass from packed activations (spec_qmatmul_plan)
        pk_qkv = pk and self._plan80(self.nqkv, H, R)
        pk_o = pk and self._plan80(H, self.Hq * D, R)
        pk_gu = pk and self._plan80(2 * F, H, R)
        pk_down = pk and self._plan80(H, F, R)
        self._norm(lay["norm1"], R, pk_qkv)
        tr("norm1")
        self._matmul(lay["qkv"], self.nqkv, H, self.a, R, self.qkv, 0, pk_qkv)
        tr("qkv")
        L.spec_rope_append(self.qkv, R, self.Hq, self.Hkv, D, self.rope, self.max_len, cu_rows, ctx, S, self.q,
                           self.k_cache[li], self.v_cache[li], self.pages, self.block_table, self.max_blocks,
                           None, None, self.dev_err)
        tr("rope")
        if pk_o:
            L.spec_flash_decode_packed(self.q, L.SPEC_BF16, self.Hq, self.Hkv, D, 1.0 / math.sqrt(D),
                                       self.k_cache[li], self.v_cache[li], self.pages, self.block_table,
                                       self.max_blocks, ctx, cu_rows, S, R, max_kv_len, self.attn, self.attn_ws,
                                       self.ws_bytes, self.xpk, self.dev_err)
        else:
            L.spec_flash_decode(self.q, L.SPEC_BF16, self.Hq, self.Hkv, D, 1.0 / math.sqrt(D), self.k_cache[li],
                                self.v_cache[li], self.pages, self.block_table, self.max_blocks, ctx, cu_rows, S, R,
                                max_kv_len, self.attn, L.SPEC_BF16, self.attn_ws, self.ws_bytes, self.dev_err)
        tr("attn")
        self._matmul(lay["o"], H, self.Hq * D, self.attn, R, self.h, 1, pk_o)
        tr("o")
        self._norm(lay["norm2"], R, pk_gu)
        tr("norm2")
        if trace is None and not pk_down and "gu_il" in lay:
            # gate/up product and SwiGLU in one launch (the same bits as the two calls)
            wq, ws = lay["gu_il"]
            L.spec_qmatmul_swiglu(wq, ws, F, H, self.a, self.xpk if pk_gu else None, R, H, self.act, F, self.qws,
                                  self.qws_bytes, self.dev_err)
        else:
            self._matmul(lay["gu"], 2 * F, H, self.a, R, self.gu, 0, pk_gu)
            tr("gu")
            if pk_down:
                L.spec_swiglu_packed(self.gu, R, F, self.act, self.xpk)
            else:
                L.spec_swiglu(self.gu, R, F, self.act)
        tr("swiglu")
        self._matmul(lay["down"], H, F, self.act, R, self.h, 1, pk_down)
        tr("down")

    def _norm(self, w, R, pk):
        """self.a = RMSNorm(self.h) * w (and its packed form when pk)."""
        if pk:
            L.spec_add_rmsnorm_packed(self.h, None, w, R, self.H, self.cfg.eps, self.a, self.xpk)
        else:
            L.spec_add_rmsnorm(self.h, None, w, R, self.H, self.cfg.eps, self.a)

    def _plan80(self, N, K, R):
        """True when the 80-column pass from packed activations is the faster plan
        for an N x K matrix over R rows (every plan gives the same bits)."""
        key = (N, K, R)
        if key not in self._plans:
            self._plans[key] = L.spec_qmatmul_plan(N, K, R, True) == 80
        return self._plans[key]

    def _matmul(self, wts, N, K, x, R, y, accumulate, pk):
        """y (+)= W x over R rows; from the packed activations when pk."""
        if pk:
            L.spec_qmatmul_packed(wts[0], wts[1], N, K, self.xpk, R, y, L.SPEC_F32, N, accumulate, self.qws,
                                  self.qws_bytes, self.dev_err)
        else:
            L.spec_qmatmul(wts[0], wts[1], N, K, x, R, K, y, L.SPEC_F32, N, accumulate, self.qws, self.qws_bytes,
                           self.dev_err)

    def enable_gate(self, capacity: int = 16):
        """Evaluate the LM head through the margin gate (tokenstrom.com, "'Lossless,'
        but not quite", sections "Why the math checks out and the text still flips"
        and "What the big servers offer and what it costs"): fast non-invariant
        logits, then an invariant re-evaluation of only the rows whose top-2 margin
        is within twice the summation-order bound (all rows when more than
        `capacity` are).  Every row's argmax equals the invariant argmax."""
        d, R, H, V = self.device, self.max_rows, self.H, self.V
        cap = max(1, min(capacity, R))
        g = {"cap": cap}
        g["ws_bytes"] = L.spec_margin_gate_workspace(R, V)
        g["ws"] = torch.empty(g["ws_bytes"] // 4 + 16, dtype=torch.float32, device=d)
        g["top"] = torch.zeros(R, dtype=torch.int32, device=d)
        g["rows"] = torch.zeros(cap, dtype=torch.int32, device=d)
        g["count"] = torch.zeros(1, dtype=torch.int32, device=d)
        g["overflow"] = torch.zeros(1, dtype=torch.int32, device=d)
        g["xg"] = torch.zeros((cap, H), dtype=torch.int16, device=d)
        g["yg"] = torch.zeros((cap, V), dtype=torch.float32, device=d)
        self.gate = g

    def head(self, R, trace=None):
        pk = self._packed(R) and self.gate is None and self._plan80(self.V, self.H, R)
        self._norm(self.final_norm, R, pk)
        if trace:
            trace("final_norm")
        if self.gate is None:
            self._matmul(self.lm, self.V, self.H, self.a, R, self.logits, 0, pk)
            return
        g, H, V = self.gate, self.H, self.V
        L.spec_qmatmul_noninvariant(self.lm[0], self.lm[1], V, H, self.a, R, H, self.logits, V, 0, self.qws,
                                    self.qws_bytes)
        L.spec_margin_gate(self.logits, V, R, self.a, H, H, self.gate_coef, g["top"], g["rows"], g["count"],
                           g["overflow"], g["cap"], g["xg"], g["ws"], g["ws_bytes"], self.dev_err)
        L.spec_qmatmul_devcols(self.lm[0], self.lm[1], V, H, g["xg"], g["cap"], H, g["yg"], L.SPEC_F32, V, 0,
                               g["count"], 1, self.qws, self.qws_bytes, self.dev_err)
        L.spec_gate_scatter(g["yg"], V, g["rows"], g["count"], g["cap"], self.logits)
        L.spec_qmatmul_devcols(self.lm[0], self.lm[1], V, H, self.a, R, H, self.logits, L.SPEC_F32, V, 0,
                               g["overflow"], 1, self.qws, self.qws_bytes, self.dev_err)

    def forward(self, tokens, cu_rows, ctx, S, R, max_kv_len=None):
        """Logits (fp32 [R][V], in self.logits) for a ragged verify batch whose rows
        sit at positions ctx[s] + i; writes the rows' K/V into the cache."""
        assert R <= self.max_rows
        self.embed(tokens, R)
        for li in range(self.cfg.layers):
            self.layer(li, R, cu_rows, ctx, S, max_kv_len)
        self.head(R)
        return self.logits[:R]


def max_len_for(P: int, n_new: int, W: int) -> int:
    """KV positions a Generator needs for prompts of P tokens, n_new new tokens and W drafts."""
    return P + (n_new + 1) * (W + 1) + 2 * W + 16


class Generator:
    """Greedy generation for S sequences, W drafts per step (W = 0: ordinary
    width-1 decoding).  All per-step state lives on the device.  With
    inv_temp > 0 tokens are sampled at temperature 1 / inv_temp instead
    (spec_verify_sample; draws keyed by seed, sequence index and position)."""

    def __init__(self, dec: Decoder, prompts: np.ndarray, W: int, pads: np.ndarray, n_new: int,
                 inv_temp: float = 0.0, seed: int = 0):
        self.dec, self.W = dec, W
        self.inv_temp, self.seed = float(inv_temp), int(seed)
        S, P = prompts.shape
        assert S == dec.S
        d = dec.device
        self.S, self.P, self.n_new = S, P, n_new
        # a sequence may gain W + 1 tokens per step while the slowest gains one
        self.cap = P + (n_new + 1) * (W + 1) + 8
        assert dec.max_len >= self.cap + W + 1, "decoder max_len too small for this generation"
        self.R = S * (W + 1)
        hist = np.zeros((S, self.cap), np.int32)
        hist[:, :P] = prompts
        self.hist = torch.from_numpy(hist).to(d)
        self.hist_len = torch.full((S,), P, dtype=torch.int32, device=d)
        self.ctx = torch.full((S,), P - 1, dtype=torch.int32, device=d)
        self.ctx_new = torch.zeros(S, dtype=torch.int32, device=d)
        self.cu = torch.arange(0, self.R + 1, W + 1, dtype=torch.int32, device=d)
        self.block = torch.zeros(self.R, dtype=torch.int32, device=d)
        self.drafts = torch.zeros(max(S * W, 1), dtype=torch.int32, device=d)
        self.argmax = torch.zeros(self.R, dtype=torch.int32, device=d)
        self.accepted = torch.zeros(S, dtype=torch.int32, device=d)
        self.correction = torch.zeros(S, dtype=torch.int32, device=d)
        self.cu_kept = torch.zeros(S + 1, dtype=torch.int32, device=d)
        self.kept_src = torch.zeros(self.R, dtype=torch.int32, device=d)
        self.dst_slot = torch.zeros(self.R, dtype=torch.int64, device=d)
        self.vws_bytes = L.spec_verify_greedy_workspace(self.R, dec.V)
        self.vws = torch.empty(self.vws_bytes // 8 + 2, dtype=torch.int64, device=d)
        self.pads = torch.from_numpy(np.ascontiguousarray(pads, np.int32)).to(d)   # [n_pad][S][W]
        self.pad_step = torch.zeros((S, max(W, 1)), dtype=torch.int32, device=d)
        self.steps = 0
        self.graph = None
        # prefill the first P-1 prompt tokens of every sequence (same kernels, one ragged batch)
        pre = torch.from_numpy(np.ascontiguousarray(prompts[:, :P - 1].reshape(-1), np.int32)).to(d)
        cu = torch.arange(0, S * (P - 1) + 1, P - 1, dtype=torch.int32, device=d)
        zero = torch.zeros(S, dtype=torch.int32, device=d)
        dec.forward(pre, cu, zero, S, S * (P - 1))

    def _step_body(self):
        dec, W, S, R = self.dec, self.W, self.S, self.R
        L.spec_ngram_draft(self.hist, self.cap, self.hist_len, S, W, self.pad_step, self.drafts, None, self.block)
        logits = dec.forward(self.block, self.cu, self.ctx, S, R)
        if self.inv_temp > 0:
            L.spec_verify_sample(logits, L.SPEC_F32, dec.V, self.cu, S, R, self.drafts if W else None, self.ctx,
                                 None, self.inv_temp, self.seed, self.argmax, self.accepted, self.correction,
                                 self.ctx_new, self.vws, self.vws_bytes, dec.dev_err)
        else:
            L.spec_verify_greedy(logits, L.SPEC_F32, dec.V, self.cu, S, R, self.drafts if W else None, self.ctx,
                                 self.argmax, self.accepted, self.correction, self.ctx_new, self.vws, self.vws_bytes,
                                 dec.dev_err)
        # the block's K/V were written into the cache in place: realignment is index-only
        L.spec_kv_compact(None, None, None, None, dec.Hkv, dec.D, dec.pages, dec.block_table, dec.max_blocks,
                          self.ctx, self.accepted, self.cu, S, R, self.cu_kept, self.kept_src, self.dst_slot,
                          dec.dev_err)
        L.spec_commit_accepted(self.hist, self.cap, self.hist_len, self.drafts, W, self.accepted, self.correction,
                               self.ctx_new, self.ctx, S, dec.dev_err)

    def set_pads(self, step):
        if self.W:
            self.pad_step.copy_(self.pads[step % self.pads.shape[0]])

    def step(self, use_graph=False):
        self.set_pads(self.steps)
        if use_graph and self.steps > 0:
            # the first step runs eagerly, so every kernel is configured before capture
            if self.graph is None:
                self._capture()
            self.graph.replay()
        else:
            self._step_body()
        self.steps += 1

    def _capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        # every call in the step is capture-safe: no allocation, no synchronisation
        with torch.cuda.graph(g, stream=s):
            self._step_body()
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g

    def done(self) -> bool:
        return int(self.hist_len.min().item()) >= self.P + self.n_new

    def run(self, use_graph=False, max_steps=None):
        max_steps = max_steps or (self.n_new + 1)
        while not self.done() and self.steps < max_steps:
            self.step(use_graph)
        torch.cuda.synchronize()
        return self.tokens()

    def tokens(self) -> np.ndarray:
        h = self.hist.cpu().numpy()
        return h[:, self.P:self.P + self.n_new]
