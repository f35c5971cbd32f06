"""End-to-end: speculative greedy generation must produce the same bytes as
width-1 greedy generation (ramgpt.org, "When Lossless Speculation Stops Being
Lossless on Blackwell", sections "Why Tiny Numerical Differences Can Change
Entire Answers" and "A Better Backend Test Matrix"), and each decoder layer
must agree with the oracle's layer within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, bf16_rounding_ok, bf16_rounding_report, bits_to_f64, host, rel_err_rows

pytestmark = pytest.mark.gpu

SMALL = synth.DecoderConfig(layers=2, hidden=256, heads=4, kv_heads=2, head_dim=64, ffn=512, vocab=1024)


def generate(weights, prompts, W, n_new, pads, use_graph=False):
    from invariant_speculative_verification_gb300.decoder import Decoder, Generator, max_len_for
    S, P = prompts.shape
    max_len = max_len_for(P, n_new, W)
    dec = Decoder(weights, S, max_len, max_rows=max(S * (P - 1), S * (W + 1)))
    gen = Generator(dec, prompts, W, pads, n_new)
    toks = gen.run(use_graph=use_graph)
    assert int(dec.dev_err.item()) == 0
    return toks, gen.steps


@pytest.mark.parametrize("use_graph", [False, True])
def test_speculative_equals_width1_small_decoder(use_graph):
    w = synth.decoder_weights(1005, SMALL)
    pr = synth.prompts(1006, 8, 32, SMALL.vocab)
    pads = synth.pad_tokens(1007, 8, 256, 4, SMALL.vocab).transpose(1, 0, 2).copy()
    base, s1 = generate(w, pr, 0, 96, pads, use_graph)
    spec, s4 = generate(w, pr, 4, 96, pads, use_graph)
    assert np.array_equal(base, spec)
    assert s4 < s1


@pytest.mark.parametrize("cfg,P,layers", [(SMALL, 20, None), (synth.E2E_DECODER, 16, 2)],
                         ids=["small", "full_size_2_layers"])
def test_layer_steps_and_logits_match_oracle(cfg, P, layers):
    """Every step of each decoder layer and of the LM head against the oracle's
    piece for that step, fed the GPU's own input to the step (so each comparison
    carries only that step's error):
      * fp32 results (the int4 matmuls and their residual adds) within TOL of
        the row's max-abs, the fixed parity bound;
      * bf16 results that round a short fp32 computation (RMSNorm, RoPE and the
        K/V cache entries, SwiGLU) equal the oracle's value rounded to bf16, except
        where that value lies within the fp32 computation's error of a rounding
        midpoint, where either neighbour is right;
      * the attention output, an fp32 result rounded to bf16, within TOL + 2^-9
        (half a bf16 ulp relative to the element) of the row's max-abs.
    At full size the int4 matmuls split tiles across CTAs and calls of 24 to 250
    tiles share one workspace, in the decoder's own call order."""
    from invariant_speculative_verification_gb300.decoder import Decoder
    w = synth.decoder_weights(2024, cfg)
    toks = synth.prompts(2025, 1, P, cfg.vocab)[0]
    dec = Decoder(w, 1, 64, max_rows=P)
    H, F, D, Hq, Hkv = cfg.hidden, cfg.ffn, cfg.head_dim, cfg.heads, cfg.kv_heads
    d = "cuda"
    t = torch.from_numpy(toks).to(d)
    cu = torch.tensor([0, P], dtype=torch.int32, device=d)
    ctx = torch.zeros(1, dtype=torch.int32, device=d)
    dec.embed(t, P)
    torch.cuda.synchronize()
    assert np.array_equal(host(dec.h[:P]), oracle.Decoder(w, 1, 64).embed(toks))
    bf = lambda buf: host(buf[:P], np.uint16)            # noqa: E731
    f64 = lambda buf: host(buf[:P]).astype(np.float64)   # noqa: E731
    for li in range(layers or cfg.layers):
        lay = w.layers[li]
        snap = {"in": f64(dec.h)}

        def trace(name):
            torch.cuda.synchronize()
            if name in ("norm1", "norm2"):
                snap[name] = bf(dec.a)
            elif name == "qkv":
                snap[name] = f64(dec.qkv)
            elif name == "rope":
                snap["q"] = host(dec.q[:P], np.uint16)
                snap["k"] = host(dec.k_cache[li], np.uint16).copy()
                snap["v"] = host(dec.v_cache[li], np.uint16).copy()
            elif name == "attn":
                snap[name] = bf(dec.attn)
            elif name in ("o", "down"):
                snap[name] = f64(dec.h)
            elif name == "gu":
                snap[name] = f64(dec.gu)
            elif name == "swiglu":
                snap[name] = bf(dec.act)

        dec.layer(li, P, cu, ctx, 1, trace=trace)
        # RMSNorm (fp32 sum of squares and rsqrt: relative error well below 1e-6)
        for nm, h_src in (("norm1", snap["in"]), ("norm2", snap["o"])):
            ref = np.stack([oracle.rmsnorm(h_src[r], lay[nm], cfg.eps) for r in range(P)])
            assert bf16_rounding_ok(snap[nm], ref, 1e-6 * np.abs(ref) + 1e-30), (li, nm)
        # qkv projection
        ref = oracle.qmatmul(lay["qkv"][0], lay["qkv"][1], snap["norm1"], dec.nqkv, H)
        assert rel_err_rows(snap["qkv"], ref) <= TOL, (li, "qkv")
        # RoPE on q and k at positions 0..P-1 (fp32 table and arithmetic), V copied;
        # page p of the one sequence is cache page p
        qkv = snap["qkv"]
        for r in range(P):
            for hh in range(Hq + Hkv):
                v = qkv[r, hh * D:(hh + 1) * D]
                ref = oracle.rope(v, r, cfg.rope_theta)
                slack = 1e-6 * (np.abs(v) + np.abs(np.roll(v, D // 2))) + 1e-30
                got = snap["q"][r, hh] if hh < Hq else snap["k"][r // 16, hh - Hq, r % 16]
                assert bf16_rounding_ok(got, ref, slack), (li, "rope", r, hh, bf16_rounding_report(got, ref, slack))
            vv = qkv[r, (Hq + Hkv) * D:]
            for kh in range(Hkv):
                assert bf16_rounding_ok(snap["v"][r // 16, kh, r % 16], vv[kh * D:(kh + 1) * D], 0.0), (li, "v", r)
        # attention over the GPU's own bf16 q and cache
        ref = oracle.attention(q=snap["q"], dt=synth.DT_BF16, Hq=Hq, Hkv=Hkv, D=D, scale=1.0 / np.sqrt(D),
                               k_cache=snap["k"], v_cache=snap["v"], block_table=host(dec.block_table),
                               ctx_start=np.zeros(1, np.int32), cu_rows=np.array([0, P], np.int32))
        assert rel_err_rows(bits_to_f64(snap["attn"]).reshape(P, Hq, D), ref) <= TOL + 2 ** -9, (li, "attn")
        # o projection added to the residual stream
        y = oracle.qmatmul(lay["o"][0], lay["o"][1], snap["attn"], H, Hq * D)
        assert rel_err_rows(snap["o"] - snap["in"], y) <= TOL, (li, "o")
        # gate/up, SwiGLU (fp32 silu: relative error well below 1e-6), down added to the residual
        ref = oracle.qmatmul(lay["gu"][0], lay["gu"][1], snap["norm2"], 2 * F, H)
        assert rel_err_rows(snap["gu"], ref) <= TOL, (li, "gu")
        gu = snap["gu"]
        ref = np.array([[oracle.silu_mul(gu[r, i], gu[r, F + i]) for i in range(F)] for r in range(P)])
        assert bf16_rounding_ok(snap["swiglu"], ref, 1e-6 * np.abs(ref) + 1e-30), (li, "swiglu")
        y = oracle.qmatmul(lay["down"][0], lay["down"][1], snap["swiglu"], H, F)
        assert rel_err_rows(snap["down"] - snap["o"], y) <= TOL, (li, "down")
    hs = {}

    def trace_head(name):
        torch.cuda.synchronize()
        hs[name] = bf(dec.a)

    h_last = f64(dec.h)
    dec.head(P, trace=trace_head)
    torch.cuda.synchronize()
    ref = np.stack([oracle.rmsnorm(h_last[r], w.final_norm, cfg.eps) for r in range(P)])
    assert bf16_rounding_ok(hs["final_norm"], ref, 1e-6 * np.abs(ref) + 1e-30), "final_norm"
    ref = oracle.qmatmul(w.lm[0], w.lm[1], hs["final_norm"], cfg.vocab, H)
    assert rel_err_rows(host(dec.logits[:P]), ref) <= TOL, "lm_head"


def test_full_size_decoder_speculative_equals_width1():
    """8 layers, hidden 2048, 16/4 heads of 128, FFN 5632, vocab 32000; 16 prompts
    of 128 tokens; here 128 generated tokens (the benchmark runs 1024)."""
    cfg = synth.E2E_DECODER
    w = synth.decoder_weights(1005, cfg)
    pr = synth.prompts(1006, 16, 128, cfg.vocab)
    pads = synth.pad_tokens(1007, 16, 512, 4, cfg.vocab).transpose(1, 0, 2).copy()
    base, s1 = generate(w, pr, 0, 128, pads, use_graph=True)
    spec, s4 = generate(w, pr, 4, 128, pads, use_graph=True)
    assert np.array_equal(base, spec)
