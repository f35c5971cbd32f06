"""Pins of the oracle's decoder composition by a hand-worked one-layer case.

The case (tests/golden/decoder_layer_hand_case.txt) is built from one-hot int4
weights so that every intermediate value of the layer and the LM head is a
closed form.  The expected values below are those closed forms for this case
only (no loop over heads, rows or features, nothing shared with the oracle);
each misreading the case is built against -- gate and up swapped, attention
scale 1, RoPE on V or missing on Q or K, interleaved RoPE pairs, a norm
skipped, the norm weight ignored -- moves at least one checked value far
outside the tolerance, which the second test shows by evaluating those
misreadings' own closed forms.

Source: ramgpt.org, "When Lossless Speculation Stops Being Lossless on
Blackwell", section "Why Tiny Numerical Differences Can Change Entire
Answers" (byte identity is a property of the decoder's output).
"""
import math

import numpy as np
import pytest

import oracle
import synth

H, HQ, HKV, D, F, V = 32, 2, 1, 16, 32, 8
THETA = 4.0 / math.pi ** 2   # rotary pair 4 turns by theta^(-4/8) = pi/2 at position 1
CFG = synth.DecoderConfig(layers=1, hidden=H, heads=HQ, kv_heads=HKV, head_dim=D, ffn=F, vocab=V, eps=0.0,
                          rope_theta=THETA)


def B(x: float) -> float:
    """x rounded to bfloat16 (8 significant bits, ties to even)."""
    if x == 0.0:
        return 0.0
    m, e = math.frexp(x)
    return math.ldexp(round(m * 256), e - 8)


def silu(x: float) -> float:
    return x / (1.0 + math.exp(-x))


def linear(N: int, K: int, entries, scales=()):
    """int4 block-32 weights: code 8 (q = 0) and scale 1.0 everywhere except the
    listed (row, k, q) entries and (row, block, scale) scales."""
    codes = np.full((N, K), 8, np.int64)
    d = np.ones((N, K // 32), np.float64)
    for n, k, q in entries:
        codes[n, k] = q + 8
    for n, b, s in scales:
        d[n, b] = s
    wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return wq, d.astype(np.float16).view(np.uint16)


def weights():
    qkv = linear((HQ + 2 * HKV) * D, H,
                 [(4, 0, 1), (20, 2, -1), (36, 0, 1), (44, 1, 1), (48, 1, 2), (49, 2, 2), (52, 0, 1), (60, 2, 1)],
                 [(44, 0, 0.5)])
    o = linear(H, HQ * D, [(8, 0, 1), (9, 1, 1), (10, 4, 1), (11, 12, 1), (12, 16, 1), (13, 28, 1)])
    gu = linear(2 * F, H, [(0, 8, 1), (F + 0, 10, 1)])
    down = linear(H, F, [(20, 0, 1)])
    lm = linear(V, H, [(0, 20, 1), (1, 8, 1), (2, 0, -3), (3, 12, 2)], [(3, 0, 0.5)])
    lay = {"qkv": qkv, "o": o, "gu": gu, "down": down, "norm1": np.ones(H, np.float32),
           "norm2": np.ones(H, np.float32)}
    fnorm = np.ones(H, np.float32)
    fnorm[20] = 0.5
    emb = np.zeros((V, H), np.uint16)
    return synth.DecoderWeights(CFG, emb, [lay], lm, fnorm)


def h_in() -> np.ndarray:
    h = np.zeros((2, H), np.float32)
    h[0, 0] = h[0, 1] = 0.5
    h[1, 0] = h[1, 2] = 0.5
    return h


def expected(swap_gate_up=False, att_scale=0.25, rope_v=False, rope_q=True, rope_k=True, interleaved=False,
             skip_norm1=False, skip_norm2=False, skip_final_norm=False, ignore_norm_weight=False):
    """Closed forms of this case: (h_out rows as dicts, logits rows, cached K at position 1)."""
    a = 0.5 if skip_norm1 else 4.0   # norm1 output at the two nonzero entries of each row (rms 0.125)
    # q, k, v per row before RoPE (sparse: component -> value)
    q0 = [{4: a}, {4: a}]
    q1 = [{}, {4: -a}]
    k = [{4: a, 12: 0.5 * a}, {4: a}]
    v = [{0: 2 * a, 4: a}, {1: 2 * a, 4: a, 12: a}]

    def rot(vec):
        """Position 1.  Rotate-half: pair (4, 12) turns by pi/2.  Interleaved pairs
        would instead turn (4, 5) by theta^(-4/16) and (12, 13) by theta^(-12/16)."""
        out = {c: x for c, x in vec.items() if c not in (4, 5, 12, 13)}
        if interleaved:
            for c, i in ((4, 2), (12, 6)):
                t = THETA ** (-2.0 * i / D)
                x, y = vec.get(c, 0.0), vec.get(c + 1, 0.0)
                out[c], out[c + 1] = B(x * math.cos(t) - y * math.sin(t)), B(y * math.cos(t) + x * math.sin(t))
        else:
            out[4], out[12] = -vec.get(12, 0.0), vec.get(4, 0.0)
        return {c: x for c, x in out.items() if x != 0.0}

    if rope_q:
        q0[1], q1[1] = rot(q0[1]), rot(q1[1])
    if rope_k:
        k[1] = rot(k[1])
    if rope_v:
        v[1] = rot(v[1])

    def dot(x, y):
        return sum(t * y.get(c, 0.0) for c, t in x.items())

    def attend(q, row):
        s = [att_scale * dot(q, k[j]) for j in range(row + 1)]
        m = max(s)
        p = [math.exp(t - m) for t in s]
        z = sum(p)
        out = {}
        for j in range(row + 1):
            for c, t in v[j].items():
                out[c] = out.get(c, 0.0) + p[j] / z * t
        return {c: B(t) for c, t in out.items()}

    hs, logits = [], []
    for row in range(2):
        h = {c: float(t) for c, t in enumerate(h_in()[row]) if t != 0.0}
        a0, a1 = attend(q0[row], row), attend(q1[row], row)
        for dst, src in ((8, a0.get(0, 0.0)), (9, a0.get(1, 0.0)), (10, a0.get(4, 0.0)), (11, a0.get(12, 0.0)),
                         (12, a1.get(0, 0.0)), (13, a1.get(12, 0.0))):
            if src:
                h[dst] = h.get(dst, 0.0) + src
        rms = 1.0 if skip_norm2 else math.sqrt(sum(t * t for t in h.values()) / H)
        g, u = B(h.get(8, 0.0) / rms), B(h.get(10, 0.0) / rms)
        act = B(silu(u) * g) if swap_gate_up else B(silu(g) * u)
        if act:
            h[20] = h.get(20, 0.0) + act
        hs.append(h)
        rf = 1.0 if skip_final_norm else math.sqrt(sum(t * t for t in h.values()) / H)
        w20 = 1.0 if ignore_norm_weight else 0.5
        af = {c: B(t * (w20 if c == 20 else 1.0) / rf) for c, t in h.items()}
        lg = np.zeros(V)
        lg[0] = af.get(20, 0.0)
        lg[1] = af.get(8, 0.0)
        lg[2] = -3.0 * af.get(0, 0.0)
        lg[3] = 2.0 * 0.5 * af.get(12, 0.0)
        logits.append(lg)
    return hs, np.array(logits), k[1]


def run_oracle():
    w = weights()
    dec = oracle.Decoder(w, 1, 16)
    h = dec.layer(0, h_in(), np.array([0], np.int32), np.array([0, 2], np.int32))
    return dec, h, dec.lm_head(h)


def dense(hrow):
    out = np.zeros(H)
    for c, x in hrow.items():
        out[c] = x
    return out


def test_hand_worked_decoder_layer_and_lm_head():
    dec, h, logits = run_oracle()
    hs, lg, k1 = expected()
    for row in range(2):
        np.testing.assert_allclose(h[row], dense(hs[row]), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(logits, lg, rtol=1e-6, atol=1e-7)
    # the worked values written out in the golden file (row 0)
    assert h[0, 8] == 8.0 and h[0, 10] == 4.0 and h[0, 12] == 8.0
    assert h[0, 20] == pytest.approx(B(silu(3.765625) * 1.8828125), abs=0) == 6.9375
    np.testing.assert_allclose(logits[0, :4], [1.4140625, 3.265625, -0.6123047, 3.265625], rtol=1e-6)
    np.testing.assert_allclose(h[1, 8:14], [0.953125, 7.03125, 4, 3.515625, 7.03125, 0.4765625], rtol=1e-6)
    np.testing.assert_allclose(logits[1, :4], [0.14453125, 0.47460938, -0.7470703, 3.5], rtol=1e-6)
    # cached K and V (page 0, kv head 0): K rotated at position 1, V never rotated
    kc = synth.bf16_bits_to_f32(dec.k_cache[0][0, 0])
    vc = synth.bf16_bits_to_f32(dec.v_cache[0][0, 0])
    # (cos(pi/2) is 6e-17 in double, so the rotated-away component is ~1e-16, not 0)
    assert kc[0, 4] == 4.0 and kc[0, 12] == 2.0 and abs(kc[1, 4]) < 1e-12 and kc[1, 12] == 4.0
    assert dense(k1)[12] == 4.0
    assert vc[1, 1] == 8.0 and vc[1, 4] == 4.0 and vc[1, 12] == 4.0 and vc[0, 0] == 8.0
    assert np.count_nonzero(kc[2:]) == 0 and np.count_nonzero(vc[2:]) == 0


@pytest.mark.parametrize("misreading", [
    {"swap_gate_up": True}, {"att_scale": 1.0}, {"rope_v": True}, {"rope_q": False}, {"rope_k": False},
    {"interleaved": True}, {"skip_norm1": True}, {"skip_norm2": True}, {"skip_final_norm": True}, {"ignore_norm_weight": True}])
def test_each_misreading_moves_a_checked_value(misreading):
    """The case discriminates: under each misreading some checked value lies far
    outside the 1e-6 tolerance the test above uses."""
    hs, lg, _ = expected()
    hs2, lg2, _ = expected(**misreading)
    gap = max(max(np.abs(dense(a) - dense(b)).max() for a, b in zip(hs, hs2)), np.abs(lg - lg2).max())
    assert gap > 1e-2, misreading
