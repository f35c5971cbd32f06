"""Decoder glue and device n-gram drafting against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu


def _L():
    import invariant_speculative_verification_gb300 as L
    return L


def test_add_rmsnorm_matches_oracle_and_is_row_invariant():
    L = _L()
    g = np.random.default_rng(1)
    R, H = 37, 2048
    h = g.normal(0, 1, (R, H)).astype(np.float32)
    d = g.normal(0, 1, (R, H)).astype(np.float32)
    w = g.normal(1, 0.1, H).astype(np.float32)
    hd, dd = dev(h), dev(d)
    out = torch.zeros((R, H), dtype=torch.int16, device="cuda")
    L.spec_add_rmsnorm(hd, dd, dev(w), R, H, 1e-5, out)
    torch.cuda.synchronize()
    hs = h + d
    assert np.array_equal(host(hd), hs)
    got = synth.bf16_bits_to_f32(host(out, np.uint16))
    ref = np.stack([oracle.rmsnorm(hs[r].astype(np.float64), w, 1e-5) for r in range(R)])
    assert rel_err_rows(got, ref) <= 2 ** -7                       # one bf16 rounding
    one = torch.zeros((1, H), dtype=torch.int16, device="cuda")
    L.spec_add_rmsnorm(dev(hs[5:6]), None, dev(w), 1, H, 1e-5, one)
    torch.cuda.synchronize()
    assert torch.equal(one[0], out[5])


def test_rope_append_and_cache_write():
    L = _L()
    g = np.random.default_rng(2)
    Hq, Hkv, D, S = 4, 2, 64, 3
    rows = np.array([2, 1, 3], np.int32)
    ctx = np.array([5, 0, 30], np.int32)
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(cu[-1])
    qkv = g.normal(0, 1, (R, (Hq + 2 * Hkv) * D)).astype(np.float32)
    max_pos, pages, mb = 64, 16, 4
    tab = torch.empty((max_pos, D // 2, 2), dtype=torch.float32, device="cuda")
    L.spec_rope_table(tab, max_pos, D, 10000.0)
    bt = np.arange(S * mb, dtype=np.int32).reshape(S, mb)[:, ::-1].copy()
    kc = torch.zeros((pages, Hkv, 16, D), dtype=torch.int16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.zeros((R, Hq, D), dtype=torch.int16, device="cuda")
    L.spec_rope_append(dev(qkv), R, Hq, Hkv, D, tab, max_pos, dev(cu), dev(ctx), S, q, kc, vc, pages, dev(bt), mb)
    torch.cuda.synchronize()
    qg = synth.bf16_bits_to_f32(host(q, np.uint16))
    kg = synth.bf16_bits_to_f32(host(kc, np.uint16))
    vg = synth.bf16_bits_to_f32(host(vc, np.uint16))
    for s in range(S):
        for i in range(rows[s]):
            r, pos = cu[s] + i, ctx[s] + i
            for hh in range(Hq):
                ref = oracle.rope(qkv[r, hh * D:(hh + 1) * D].astype(np.float64), pos, 10000.0)
                assert np.allclose(qg[r, hh], ref, rtol=2 ** -7, atol=1e-6)
            page, slot = bt[s, pos // 16], pos % 16
            for kh in range(Hkv):
                ref = oracle.rope(qkv[r, (Hq + kh) * D:(Hq + kh + 1) * D].astype(np.float64), pos, 10000.0)
                assert np.allclose(kg[page, kh, slot], ref, rtol=2 ** -7, atol=1e-6)
                vref = qkv[r, (Hq + Hkv + kh) * D:(Hq + Hkv + kh + 1) * D]
                assert np.array_equal(vg[page, kh, slot], synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vref)))


def test_swiglu_embed_and_cast():
    L = _L()
    g = np.random.default_rng(3)
    R, F = 9, 640
    gu = g.normal(0, 2, (R, 2 * F)).astype(np.float32)
    out = torch.zeros((R, F), dtype=torch.int16, device="cuda")
    L.spec_swiglu(dev(gu), R, F, out)
    torch.cuda.synchronize()
    got = synth.bf16_bits_to_f32(host(out, np.uint16))
    ref = np.array([[oracle.silu_mul(gu[r, i], gu[r, F + i]) for i in range(F)] for r in range(R)])
    assert rel_err_rows(got, ref) <= 2 ** -7
    # the 16-byte path (aligned, F % 4 == 0) and the element path give the same bits
    buf = torch.zeros(R * 2 * F + 1, dtype=torch.float32, device="cuda")
    buf[1:] = dev(gu).reshape(-1)
    out2 = torch.zeros((R, F), dtype=torch.int16, device="cuda")
    L.spec_swiglu(buf[1:], R, F, out2)   # misaligned by 4 bytes: element path
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    F3 = 643
    gu3 = g.normal(0, 2, (3, 2 * F3)).astype(np.float32)
    out3 = torch.zeros((3, F3), dtype=torch.int16, device="cuda")
    L.spec_swiglu(dev(gu3), 3, F3, out3)
    torch.cuda.synchronize()
    ref3 = np.array([[oracle.silu_mul(gu3[r, i], gu3[r, F3 + i]) for i in range(F3)] for r in range(3)])
    assert rel_err_rows(synth.bf16_bits_to_f32(host(out3, np.uint16)), ref3) <= 2 ** -7
    x = g.normal(0, 3, 1000).astype(np.float32)
    o = torch.zeros(1000, dtype=torch.int16, device="cuda")
    L.spec_cast_bf16(dev(x), 1000, o)
    torch.cuda.synchronize()
    assert np.array_equal(host(o, np.uint16), synth.f32_to_bf16_bits(x))
    emb = synth.f32_to_bf16_bits(g.normal(0, 0.02, (50, 64)).astype(np.float32))
    toks = np.array([3, 49, 0, 7], np.int32)
    h = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_embed(dev(emb), 50, 64, dev(toks), 4, h, err)
    torch.cuda.synchronize()
    assert np.array_equal(host(h), synth.bf16_bits_to_f32(emb[toks])) and int(err.item()) == 0


def test_ngram_draft_matches_oracle_exactly():
    L = _L()
    g = np.random.default_rng(4)
    S, cap, W = 64, 400, 4
    hist = np.zeros((S, cap), np.int32)
    lens = g.integers(0, cap, S).astype(np.int32)
    for s in range(S):
        vocab = int(g.choice([3, 8, 50, 1000]))
        hist[s, :lens[s]] = g.integers(0, vocab, lens[s])
    pad = g.integers(0, 1000, (S, W)).astype(np.int32)
    dr = torch.zeros((S, W), dtype=torch.int32, device="cuda")
    mn = torch.zeros(S, dtype=torch.int32, device="cuda")
    blk = torch.zeros((S, W + 1), dtype=torch.int32, device="cuda")
    L.spec_ngram_draft(dev(hist), cap, dev(lens), S, W, dev(pad), dr, mn, blk)
    torch.cuda.synchronize()
    drh, mnh, bh = host(dr), host(mn), host(blk)
    for s in range(S):
        ref, n = oracle.ngram_draft(hist[s, :lens[s]], W, pad[s])
        assert np.array_equal(drh[s], ref) and mnh[s] == n, s
        assert bh[s, 0] == (hist[s, lens[s] - 1] if lens[s] else 0) and np.array_equal(bh[s, 1:], ref)
