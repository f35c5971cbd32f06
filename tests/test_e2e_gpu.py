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
from tests.gpu_util import TOL, host, rel_err_rows

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
def test_layers_and_logits_match_oracle(cfg, P, layers):
    """Each layer's update and the logits vs the oracle, the layer fed the GPU's own
    input.  At full size the int4 matmuls split tiles across CTAs and calls of 24 to
    250 tiles share one workspace, in the decoder's own call order."""
    from invariant_speculative_verification_gb300.decoder import Decoder
    w = synth.decoder_weights(2024, cfg)
    toks = synth.prompts(2025, 1, P, cfg.vocab)[0]
    dec = Decoder(w, 1, 64, max_rows=P)
    od = oracle.Decoder(w, 1, 64)
    d = "cuda"
    t = torch.from_numpy(toks).to(d)
    cu = torch.tensor([0, P], dtype=torch.int32, device=d)
    ctx = torch.zeros(1, dtype=torch.int32, device=d)
    dec.embed(t, P)
    assert np.array_equal(host(dec.h[:P]), od.embed(toks))
    for li in range(layers or cfg.layers):
        h_in = host(dec.h[:P]).copy()
        for c_gpu, c_or in ((dec.k_cache[li], od.k_cache[li]), (dec.v_cache[li], od.v_cache[li])):
            c_or[...] = host(c_gpu, np.uint16)
        dec.layer(li, P, cu, ctx, 1)
        torch.cuda.synchronize()
        ref = od.layer(li, h_in.copy(), np.array([0], np.int32), np.array([0, P], np.int32))
        got = host(dec.h[:P])
        assert rel_err_rows(got - h_in, ref - h_in) <= 4 * TOL, li   # the layer's update, row by row
        kg = synth.bf16_bits_to_f32(host(dec.k_cache[li], np.uint16))
        ko = synth.bf16_bits_to_f32(od.k_cache[li])
        assert np.allclose(kg, ko, rtol=1e-2, atol=1e-2)
    dec.head(P)
    torch.cuda.synchronize()
    ref = od.lm_head(host(dec.h[:P]))
    assert rel_err_rows(host(dec.logits[:P]), ref) <= TOL


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
