"""Prefill / micro-batch / prefix-cache invariance: a prompt evaluated in one
pass, in micro-batches of any size, or as a cached prefix plus the rest leaves
bit-identical K/V in the cache and bit-identical logits for every row.

The pages list these as further ways the same tokens reach the target in
different batch shapes (ramgpt.org, "When Lossless Speculation Stops Being
Lossless on Blackwell", section "A Better Backend Test Matrix": prefill
chunking, micro-batch size and prompt-cache reuse).  Here they hold by
construction -- every row's reduction order is fixed by K and by its own
position -- and this test checks it through the whole decoder.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

CFG = synth.DecoderConfig(layers=2, hidden=256, heads=4, kv_heads=2, head_dim=64, ffn=512, vocab=1024)


def run_chunks(weights, prompts, splits):
    """Feed each sequence's prompt in the given chunk lengths (splits[s]); every
    call evaluates one chunk of every sequence that still has tokens, as one
    ragged batch.  Returns (logits per sequence [P][V], the decoder)."""
    from invariant_speculative_verification_gb300.decoder import Decoder
    S, P = prompts.shape
    dec = Decoder(weights, S, max_len=P + 32, max_rows=S * P)
    done = [0] * S
    out = [np.zeros((P, CFG.vocab), np.float32) for _ in range(S)]
    step = 0
    while any(d < P for d in done):
        toks, cu, ctx, who = [], [0], [], []
        for s in range(S):
            if done[s] >= P:
                n = 0
            else:
                n = min(splits[s][step % len(splits[s])], P - done[s])
            toks.extend(prompts[s, done[s]:done[s] + n])
            cu.append(cu[-1] + n)
            ctx.append(done[s])
            who.append(n)
        R = cu[-1]
        d = dec.device
        logits = dec.forward(torch.tensor(toks, dtype=torch.int32, device=d),
                             torch.tensor(cu, dtype=torch.int32, device=d),
                             torch.tensor(ctx, dtype=torch.int32, device=d), S, R).cpu().numpy()
        for s in range(S):
            out[s][done[s]:done[s] + who[s]] = logits[cu[s]:cu[s + 1]]
            done[s] += who[s]
        step += 1
    torch.cuda.synchronize()
    assert int(dec.dev_err.item()) == 0
    return out, dec


def test_prefill_chunking_and_prefix_reuse_are_bit_invariant():
    w = synth.decoder_weights(3030, CFG)
    S, P = 3, 70
    prompts = synth.prompts(3031, S, P, CFG.vocab)
    whole, d0 = run_chunks(w, prompts, [[P]] * S)
    variants = [
        [[1], [1], [1]],                      # token by token (width-1 decoding of the prompt)
        [[16], [5], [37]],                    # a different micro-batch size per sequence
        [[64, 6], [3, 40, 27], [69, 1]],      # a long cached prefix, then the rest
    ]
    for splits in variants:
        got, d1 = run_chunks(w, prompts, splits)
        for s in range(S):
            assert np.array_equal(got[s].view(np.uint32), whole[s].view(np.uint32)), (splits, s)
        pages = (P + 15) // 16
        for li in range(CFG.layers):
            for s in range(S):
                blocks = d0.block_table[s, :pages].long()
                assert torch.equal(d1.k_cache[li][blocks], d0.k_cache[li][blocks]), (splits, li, s)
                assert torch.equal(d1.v_cache[li][blocks], d0.v_cache[li][blocks]), (splits, li, s)
