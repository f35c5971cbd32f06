"""Pins of the oracle's temperature-sampling verification (CPU).

The generator is pinned to the published known-answer vectors of
Philox4x32-10; the sampler to the distribution it must draw from (Gumbel-max
gives an exact sample of softmax(logit / T)), its zero-temperature limit (the
greedy argmax) and its independence from the batch it is evaluated in; the
method to its invariant (speculative sampling output == width-1 sampling
output on a tiny decoder).
"""
import os

import numpy as np

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answer_vectors():
    n = 0
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        assert list(oracle.philox4x32_10(w[0:4], w[4:6])) == w[6:10]
        n += 1
    assert n == 3


def _draws(logits, inv_temp, seed, n_pos):
    """Tokens drawn for one logit row at positions 0 .. n_pos-1 (one row per position)."""
    V = logits.shape[0]
    lg = np.tile(logits.astype(np.float32), (n_pos, 1))
    cu = np.arange(n_pos + 1, dtype=np.int32)            # n_pos sequences of one row each
    ctx = np.zeros(n_pos, np.int32)
    sid = np.zeros(n_pos, np.int32)                        # the same sequence ...
    ctx[:] = np.arange(n_pos)                              # ... at positions 0 .. n_pos-1
    return oracle.verify_sample(lg, oracle.DT_F32, V, cu, np.zeros(0, np.int32), ctx, inv_temp, seed,
                                seq_id=sid)["token"]


def test_draws_follow_softmax_of_logits_over_temperature():
    logits = np.array([0.0, 1.0, 2.0, 3.0, -1.0])
    n = 40000
    for T in (1.0, 2.5):
        tok = _draws(logits, 1.0 / T, 12345, n)
        freq = np.bincount(tok, minlength=5) / n
        p = np.exp(logits / T - (logits / T).max())
        p /= p.sum()
        # 5 standard errors of a binomial proportion
        assert np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / n) + 1e-4), (T, freq, p)


def test_zero_temperature_limit_is_the_argmax():
    g = np.random.default_rng(4)
    lg = g.normal(0, 1, (50, 300)).astype(np.float32)
    cu = np.arange(51, dtype=np.int32)
    res = oracle.verify_sample(lg, oracle.DT_F32, 300, cu, np.zeros(0, np.int32), np.arange(50, dtype=np.int32),
                               1e5, 99)
    assert np.array_equal(res["token"], lg.argmax(axis=1))


def test_draws_depend_on_sequence_and_position_not_on_the_batch():
    g = np.random.default_rng(8)
    V = 200
    rows = [3, 1, 4]
    lg = g.normal(0, 2, (sum(rows), V)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    ctx = np.array([10, 0, 57], np.int32)
    sid = np.array([2, 0, 5], np.int32)
    full = oracle.verify_sample(lg, oracle.DT_F32, V, cu, np.zeros(sum(rows) - 3, np.int32), ctx, 0.7, 42,
                                seq_id=sid)["token"]
    for s in range(3):
        for i in range(rows[s]):
            r = cu[s] + i
            one = oracle.verify_sample(lg[r:r + 1], oracle.DT_F32, V, np.array([0, 1], np.int32),
                                       np.zeros(0, np.int32), np.array([ctx[s] + i], np.int32), 0.7, 42,
                                       seq_id=np.array([sid[s]], np.int32))["token"][0]
            assert one == full[r], (s, i)
    # another seed or another sequence identity draws differently somewhere
    other = oracle.verify_sample(lg, oracle.DT_F32, V, cu, np.zeros(sum(rows) - 3, np.int32), ctx, 0.7, 43,
                                 seq_id=sid)["token"]
    assert not np.array_equal(other, full)


def test_acceptance_follows_the_sampled_tokens():
    g = np.random.default_rng(9)
    V = 64
    lg = g.normal(0, 1, (5, V)).astype(np.float32)
    cu = np.array([0, 5], np.int32)
    ctx = np.array([20], np.int32)
    t = oracle.verify_sample(lg, oracle.DT_F32, V, cu, np.zeros(4, np.int32), ctx, 1.0, 5)["token"]
    # all drafts equal to the drawn tokens: all accepted, the last row's token corrects
    r = oracle.verify_sample(lg, oracle.DT_F32, V, cu, t[:4], ctx, 1.0, 5)
    assert r["accepted"][0] == 4 and r["correction"][0] == t[4] and r["ctx_new"][0] == 25
    # the second draft differs: one accepted, correction = the drawn token of row 1
    d = t[:4].copy()
    d[1] = (d[1] + 1) % V
    r = oracle.verify_sample(lg, oracle.DT_F32, V, cu, d, ctx, 1.0, 5)
    assert r["accepted"][0] == 1 and r["correction"][0] == t[1]


def test_speculative_sampling_equals_width1_sampling_tiny_decoder():
    w = synth.decoder_weights(77, synth.TINY_DECODER)
    prompts = synth.prompts(78, 3, 12, synth.TINY_DECODER.vocab)
    pads = synth.pad_tokens(79, 3, 64, 4, synth.TINY_DECODER.vocab).transpose(1, 0, 2).copy()
    base, _, _ = oracle.generate(w, prompts, 24, 0, pads, inv_temp=1.0 / 0.8, seed=2024)
    spec, _, acc = oracle.generate(w, prompts, 24, 4, pads, inv_temp=1.0 / 0.8, seed=2024)
    assert np.array_equal(base, spec)
    greedy, _, _ = oracle.generate(w, prompts, 24, 0, pads)
    assert not np.array_equal(greedy, base)   # sampling at T = 0.8 does change the text
