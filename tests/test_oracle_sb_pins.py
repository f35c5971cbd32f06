"""Pins of the oracle's two-level (super-block) scale format, independent of the oracle itself:
hand-encoded records, equality with the pinned single-level product wherever D * s is an exact fp16
scale, a closed form, and the record padding when K / 256 is odd."""
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def golden_records():
    out = []
    for line in open(os.path.join(HERE, "golden", "sb_records.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, s, d = (f.strip() for f in line.split("|"))
        out.append((bytes(int(h, 16) for h in b.split()), [int(v) for v in s.split()], float(d)))
    return out


@pytest.mark.parametrize("rec,s,D", golden_records())
def test_record_decode_matches_hand_encoded_fixture(rec, s, D):
    got_s, got_D = oracle.sb_record(rec)
    assert got_s == s and got_D == D


@pytest.mark.parametrize("K", [256, 768, 2048])
def test_equals_single_level_product_when_block_scales_are_exact_fp16(K):
    """D a power of two and s <= 63 make D * s an exact fp16 value: the two-level
    product must then equal the single-level product with d_b = D * s_b."""
    g = np.random.default_rng(K)
    N, n = 37, 3
    codes = g.integers(0, 16, size=(N, K))
    wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    e = g.integers(-12, 2, size=(N, K // 256))
    D = np.ldexp(1.0, e).astype(np.float16)
    s = g.integers(0, 64, size=(N, K // 32))
    sbr = synth.pack_sb_records(s, D.view(np.uint16))
    d = (np.repeat(D.astype(np.float64), 8, axis=1) * s).astype(np.float16)
    assert np.array_equal(d.astype(np.float64), np.repeat(D.astype(np.float64), 8, axis=1) * s)
    x = synth.activations_bf16(K + 1, n, K)
    y_sb = oracle.qmatmul_sb(wq, sbr, x, N, K)
    y_1 = oracle.qmatmul(wq, d.view(np.uint16), x, N, K)
    assert np.array_equal(y_sb, y_1)


def test_closed_form_constant_code_and_unit_activations():
    """All codes 9 (q = 1), x = 1: y[n] = 32 * sum over super-blocks of D * sum_j s_j."""
    N, K = 5, 512
    wq = np.full((N, K // 2), 0x99, np.uint8)
    g = np.random.default_rng(7)
    s = g.integers(0, 64, size=(N, K // 32))
    D = np.array([[0.25, 2.0]] * N, dtype=np.float16)
    sbr = synth.pack_sb_records(s, D.view(np.uint16))
    x = np.full((1, K), 0x3F80, np.uint16)                   # bf16 1.0
    want = 32.0 * (D.astype(np.float64) * s.reshape(N, 2, 8).sum(axis=2)).sum(axis=1)
    assert np.array_equal(oracle.qmatmul_sb(wq, sbr, x, N, K)[0], want)


def test_padding_record_is_ignored_and_pitch_is_16_byte_pairs():
    N, K = 4, 768                                           # three super-blocks, two record pairs
    assert oracle.sb_pitch(K) == 32
    c = synth.qmatmul_sb_case(11, N, K, 2)
    y = oracle.qmatmul_sb(c.wq, c.ws, c.x, N, K)
    junk = c.ws.copy()
    junk[:, 24:32] = 0xA5                                   # the fourth (padding) record
    assert np.array_equal(oracle.qmatmul_sb(c.wq, junk, c.x, N, K), y)
    junk[:, 16:24] ^= 0x01                                  # the third record is used
    assert not np.array_equal(oracle.qmatmul_sb(c.wq, junk, c.x, N, K), y)


def test_quantizer_round_trip_is_close():
    """The seeded generator's encoding reproduces its float matrix to within half a step."""
    g = np.random.default_rng(3)
    w = g.normal(0, 0.02, size=(8, 512)).astype(np.float32)
    wq, sbr = synth.quantize_q4_superblock(w)
    x = np.eye(512, dtype=np.float32)
    back = oracle.qmatmul_sb(wq, sbr, synth.f32_to_bf16_bits(x), 8, 512).T   # column k of W
    step = np.abs(w).reshape(8, 16, 32).max(axis=2) / 7.0
    err = np.abs(back - w).reshape(8, 16, 32).max(axis=2)
    assert float((err / np.maximum(step, 1e-30)).max()) <= 0.75
