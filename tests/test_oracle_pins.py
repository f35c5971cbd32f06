"""Pins for the CPU oracle: closed forms, exact brute force, invariants and the
pages' worked examples.  None of these re-types the oracle's own formula in the
oracle's arithmetic; each is chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from synth import DT_BF16, DT_F16, DT_F32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------
def test_f16_decode_matches_ieee_binary16_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_known_values():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F80: math.inf, 0xC2F7: -123.5, 0x0000: 0.0}
    for b, v in cases.items():
        assert oracle.bf16_to_double(b) == v


def test_bf16_rounding_ties_to_even_and_matches_generator_encoding():
    # halfway cases: 1 + 2^-8 lies between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 lies between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.double_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == 0xBF82
    g = np.random.default_rng(5)
    x = np.concatenate([g.normal(0, 1, 3000), g.normal(0, 1e-3, 1000), g.normal(0, 1e4, 1000)]).astype(np.float32)
    got = np.array([oracle.double_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, synth.f32_to_bf16_bits(x))


def test_golden_float_nonassociativity():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "float_nonassociativity.txt")) if not l.startswith("#")]
    for a, b, c, left, right in rows:
        a, b, c = float(a), float(b), float(c)
        for t in (np.float32, np.float64):
            assert float((t(a) + t(b)) - t(c)) == float(left)
            assert float(t(a) + (t(b) - t(c))) == pytest.approx(float(right), rel=1e-6)


# ---------------------------------------------------------------------------
# quantised matmul
# ---------------------------------------------------------------------------
def _frac_bf16(b):
    return Fraction(float(synth.bf16_bits_to_f32(np.array([b], np.uint16))[0]))


def _frac_f16(h):
    return Fraction(float(np.array([h], np.uint16).view(np.float16)[0]))


def test_qmatmul_exact_rational_brute_force():
    N, K, C = 5, 96, 3
    case = synth.qmatmul_case(11, N, K, C)
    y = oracle.qmatmul(case.wq, case.ws, case.x, N, K)
    for j in range(C):
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                byte = int(case.wq[n, k // 2])
                nib = (byte >> (4 * (k & 1))) & 15
                exact += _frac_bf16(case.x[j, k]) * _frac_f16(case.ws[n, k // 32]) * (nib - 8)
            assert abs(Fraction(y[j, n]) - exact) <= abs(exact) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 18)


def test_qmatmul_one_hot_selects_the_dequantised_weight():
    g = np.random.default_rng(3)
    N, K = 4, 64
    q = g.integers(-8, 8, size=(N, K))
    d = (g.random((N, K // 32)) * 0.1 + 0.01).astype(np.float32)
    wq, ws = synth.pack_q4(q, d)
    dq = synth.f16_bits_to_f32(ws).astype(np.float64)
    for k in [0, 1, 2, 31, 32, 33, 63]:
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y = oracle.qmatmul(wq, ws, synth.f32_to_bf16_bits(x), N, K)
        assert np.array_equal(y[0], dq[:, k // 32] * q[:, k])


def test_qmatmul_nibble_order_even_low_odd_high():
    q = np.zeros((1, 32), np.int64)
    q[0, 6], q[0, 7] = -3, 5
    wq, ws = synth.pack_q4(q, np.ones((1, 1), np.float32))
    assert wq[0, 3] == ((-3 + 8) | ((5 + 8) << 4))
    for k, want in [(6, -3.0), (7, 5.0)]:
        x = np.zeros((1, 32), np.float32)
        x[0, k] = 1.0
        assert oracle.qmatmul(wq, ws, synth.f32_to_bf16_bits(x), 1, 32)[0, 0] == want


def test_qmatmul_all_sevens_closed_form():
    N, K = 3, 128
    d = np.array([[0.5, 0.25, 0.125, 1.0], [2.0, 2.0, 2.0, 2.0], [0.0, 1.0, 0.0, 1.0]], np.float32)
    wq, ws = synth.pack_q4(np.full((N, K), 7), d)
    x = synth.f32_to_bf16_bits(np.ones((1, K), np.float32))
    y = oracle.qmatmul(wq, ws, x, N, K)
    assert np.array_equal(y[0], 7 * 32 * d.astype(np.float64).sum(axis=1))


def test_qmatmul_scaling_by_two_and_padding_of_ldx():
    case = synth.qmatmul_case(4, 16, 64, 2)
    y = oracle.qmatmul(case.wq, case.ws, case.x, 16, 64)
    x2 = synth.f32_to_bf16_bits(2 * synth.bf16_bits_to_f32(case.x))
    assert np.array_equal(oracle.qmatmul(case.wq, case.ws, x2, 16, 64), 2 * y)
    padded = np.full((2, 80), 0x7FC0, np.uint16)   # NaN in the padding must not be read
    padded[:, :64] = case.x
    assert np.array_equal(oracle.qmatmul(case.wq, case.ws, padded, 16, 64, ldx=80), y)
    rows = [3, 0, 15]
    assert np.array_equal(oracle.qmatmul_rows(case.wq, case.ws, case.x, 64, rows), y[:, rows])


def test_quantizer_round_trip_bound():
    g = np.random.default_rng(9)
    w = g.normal(0, 0.02, size=(16, 256)).astype(np.float32)
    wq, ws = synth.quantize_q4b32(w)
    d = synth.f16_bits_to_f32(ws).astype(np.float64)
    nib = np.stack([wq & 15, wq >> 4], axis=-1).reshape(16, 256).astype(np.int64)
    deq = (nib - 8) * np.repeat(d, 32, axis=1)
    err = np.abs(w - deq)
    assert np.all(err <= np.repeat(d, 32, axis=1) * 0.5 * (1 + 1e-3) + 1e-12)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _att(q, k, v, ctx, rows, Hq, Hkv, D, scale, dt=DT_F32, perm=None):
    """Build a contiguous-page cache from per-position K/V ([S][len][Hkv][D]) and call the oracle."""
    S = len(ctx)
    lens = [c + r for c, r in zip(ctx, rows)]
    mb = max((L + 15) // 16 for L in lens)
    pages = S * mb
    order = np.arange(pages) if perm is None else perm
    kc = np.zeros((pages, Hkv, 16, D), np.float32)
    vc = np.zeros((pages, Hkv, 16, D), np.float32)
    bt = np.zeros((S, mb), np.int32)
    for s in range(S):
        for b in range(mb):
            bt[s, b] = order[s * mb + b]
        for j in range(lens[s]):
            kc[bt[s, j // 16], :, j % 16] = k[s][j]
            vc[bt[s, j // 16], :, j % 16] = v[s][j]
    cu = np.zeros(S + 1, np.int32)
    cu[1:] = np.cumsum(rows)
    return oracle.attention(q=np.asarray(q, np.float32), dt=dt, Hq=Hq, Hkv=Hkv, D=D, scale=scale,
                            k_cache=kc, v_cache=vc, block_table=bt, ctx_start=np.array(ctx, np.int32),
                            cu_rows=cu)


def test_attention_single_key_returns_its_value():
    g = np.random.default_rng(1)
    D = 8
    k = [g.normal(size=(1, 1, D))]
    v = [g.normal(size=(1, 1, D)).astype(np.float32)]
    out = _att(g.normal(size=(1, 1, D)), k, v, [0], [1], 1, 1, D, 0.3)
    assert np.array_equal(out[0, 0], v[0][0, 0].astype(np.float64))


def test_attention_two_keys_closed_form_weights():
    # scores ln 3 and 0 -> weights 3/4 and 1/4
    D = 4
    q = np.array([[[1, 0, 0, 0]]], np.float32)
    k = [np.array([[[1, 0, 0, 0]], [[0, 0, 0, 0]]], np.float32)]
    v = [np.array([[[4, 8, -4, 1]], [[0, 4, 4, 1]]], np.float32)]
    out = _att(q, k, v, [1], [1], 1, 1, D, math.log(3.0))
    np.testing.assert_allclose(out[0, 0], [3.0, 7.0, -2.0, 1.0], rtol=0, atol=1e-14)


def test_attention_equal_keys_give_the_mean_and_unit_values_give_one():
    g = np.random.default_rng(2)
    D, L = 16, 37
    kv = g.normal(size=(1, 1, D))
    k = [np.repeat(kv[None], L, axis=0).reshape(L, 1, D)]
    v = [g.normal(size=(L, 1, D)).astype(np.float32)]
    out = _att(g.normal(size=(3, 1, D)), k, v, [L - 3], [3], 1, 1, D, 0.7)
    for i in range(3):
        p = L - 3 + i
        np.testing.assert_allclose(out[i, 0], v[0][:p + 1, 0].astype(np.float64).mean(axis=0), atol=1e-13)
    ones = [np.ones((L, 1, D), np.float32)]
    out = _att(g.normal(size=(3, 1, D)), [g.normal(size=(L, 1, D))], ones, [L - 3], [3], 1, 1, D, 0.7)
    np.testing.assert_allclose(out, 1.0, atol=1e-14)


def test_attention_dominating_score_selects_that_value():
    g = np.random.default_rng(3)
    D, L = 8, 20
    k = g.normal(size=(L, 1, D)).astype(np.float32) * 0.01
    k[7, 0, 0] = 100.0
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 100.0
    v = g.normal(size=(L, 1, D)).astype(np.float32)
    out = _att(q, [k], [v], [L - 1], [1], 1, 1, D, 1.0)
    assert np.array_equal(out[0, 0], v[7, 0].astype(np.float64))


def test_attention_causal_mask_inside_the_verify_block():
    # K = 0 -> uniform weights over exactly the visible keys; V = one-hot rows
    D, ctx, n = 32, 9, 6
    L = ctx + n
    k = [np.zeros((L, 1, D), np.float32)]
    v = [np.eye(L, D, dtype=np.float32).reshape(L, 1, D)]
    out = _att(np.ones((n, 1, D)), k, v, [ctx], [n], 1, 1, D, 1.0)
    for i in range(n):
        p = ctx + i
        want = np.zeros(D)
        want[:p + 1] = 1.0 / (p + 1)
        np.testing.assert_allclose(out[i, 0], want, atol=1e-15)
        assert np.all(out[i, 0, p + 1:] == 0)


def test_attention_grouped_heads_map_to_contiguous_kv_groups():
    D, L = 8, 5
    g = np.random.default_rng(4)
    k = g.normal(size=(L, 2, D)).astype(np.float32)
    v = np.zeros((L, 2, D), np.float32)
    v[:, 0] = 1.0
    v[:, 1] = 2.0
    out = _att(g.normal(size=(1, 4, D)), [k], [v], [L - 1], [1], 4, 2, D, 0.5)
    np.testing.assert_allclose(out[0, :2], 1.0, atol=1e-14)
    np.testing.assert_allclose(out[0, 2:], 2.0, atol=1e-14)


def test_attention_score_shift_invariance_and_page_permutation():
    g = np.random.default_rng(6)
    D, L, n = 8, 45, 4
    q = g.integers(-3, 4, size=(n, 1, D)).astype(np.float32)
    k = g.integers(-3, 4, size=(L, 1, D)).astype(np.float32)
    v = g.normal(size=(L, 1, D)).astype(np.float32)
    base = _att(q, [k], [v], [L - n], [n], 1, 1, D, 0.25)
    # adding u to every key adds q.u to every score of a row: the softmax is unchanged
    u = g.integers(-2, 3, size=(1, 1, D)).astype(np.float32)
    shifted = _att(q, [k + u], [v], [L - n], [n], 1, 1, D, 0.25)
    np.testing.assert_allclose(shifted, base, atol=1e-12)
    perm = g.permutation(3)
    assert np.array_equal(_att(q, [k], [v], [L - n], [n], 1, 1, D, 0.25, perm=perm), base)


def test_attention_row_head_subset_and_ragged_sequences():
    case = synth.attention_case(7, rows=[3, 1, 5], ctx=[20, 0, 33], Hq=4, Hkv=2, D=16, dt=DT_BF16)
    full = oracle.attention(case)
    assert np.all(np.isfinite(full))          # NaN-poisoned unused slots are never read
    want = np.zeros((case.R, 4), np.uint8)
    want[[0, 4, 8], [1, 3, 0]] = 1
    sub = oracle.attention(case, want=want)
    for r, h in [(0, 1), (4, 3), (8, 0)]:
        assert np.array_equal(sub[r, h], full[r, h])
    # the second sequence has a single row at position 0: its output is V_0 of its kv head
    s = 1
    r = int(case.cu_rows[s])
    page = case.block_table[s, 0]
    for h in range(4):
        v0 = synth.bf16_bits_to_f32(case.v_cache[page, h // 2, 0]).astype(np.float64)
        assert np.array_equal(full[r, h], v0)


# ---------------------------------------------------------------------------
# greedy verification
# ---------------------------------------------------------------------------
def _brute_verify(rows_vals, drafts):
    """Independent statement: argmax = lowest index holding the maximum; accepted =
    the longest prefix of drafts equal to the row argmaxes."""
    am = [min(i for i, x in enumerate(r) if x == max(r)) for r in rows_vals]
    L = len(drafts)
    a = max(a for a in range(L + 1) if all(drafts[i] == am[i] for i in range(a)))
    return am, a, am[a]


def test_verify_brute_force_enumeration_small_vocab():
    g = np.random.default_rng(12)
    V = 3
    logits, cu, drafts, expect = [], [0], [], []
    for _ in range(3000):
        L = int(g.integers(0, 4))
        rows = g.integers(0, 3, size=(L + 1, V)).astype(np.float32)
        d = g.integers(0, V, size=L)
        am, a, c = _brute_verify(rows.tolist(), d.tolist())
        logits.append(rows)
        drafts += d.tolist()
        cu.append(cu[-1] + L + 1)
        expect.append((am, a, c))
    lg = np.concatenate(logits)
    ctx = g.integers(0, 100, size=len(expect)).astype(np.int32)
    res = oracle.verify_greedy(lg, DT_F32, V, np.array(cu, np.int32), np.array(drafts, np.int32), ctx)
    for s, (am, a, c) in enumerate(expect):
        assert list(res["argmax"][cu[s]:cu[s + 1]]) == am
        assert res["accepted"][s] == a
        assert res["correction"][s] == c
        assert res["ctx_new"][s] == ctx[s] + a + 1


@pytest.mark.parametrize("dt", [DT_F32, DT_BF16])
def test_verify_planted_tops_near_ties_and_invariants(dt):
    if dt == DT_F32:
        case = synth.verify_case(1001, [4, 4], 1000, DT_F32, sigma=1.0, tie_frac=0.1)
    else:
        case = synth.verify_case(1004, list(np.random.default_rng(1).integers(1, 8, size=12)), 4096, DT_BF16,
                                 sigma=2.0, tie_frac=0.5)
    res = oracle.verify_greedy(case.logits, dt, case.V, case.cu_rows, case.drafts, case.ctx_start)
    assert np.array_equal(res["argmax"], case.planted_top)
    L = np.diff(case.cu_rows) - 1
    assert np.all((res["accepted"] >= 0) & (res["accepted"] <= L))
    assert np.all((res["correction"] >= 0) & (res["correction"] < case.V))
    assert np.array_equal(res["ctx_new"], case.ctx_start + res["accepted"] + 1)
    # all drafts right -> everything accepted; first draft wrong -> nothing accepted
    good = np.concatenate([case.planted_top[case.cu_rows[s]:case.cu_rows[s + 1] - 1] for s in range(case.S)])
    r = oracle.verify_greedy(case.logits, dt, case.V, case.cu_rows, good, case.ctx_start)
    assert np.array_equal(r["accepted"], L)
    assert np.array_equal(r["correction"], case.planted_top[case.cu_rows[1:] - 1])
    bad = good.copy()
    bad[case.cu_rows[:-1] - np.arange(case.S)] = (good[case.cu_rows[:-1] - np.arange(case.S)] + 1) % case.V
    r = oracle.verify_greedy(case.logits, dt, case.V, case.cu_rows, bad, case.ctx_start)
    assert np.all(r["accepted"] == 0)
    assert np.array_equal(r["correction"], case.planted_top[case.cu_rows[:-1]])


def test_verify_exact_tie_goes_to_lowest_index_and_nans_are_counted():
    lg = np.array([[0.5, 2.0, 1.0, 2.0], [-1.0, -1.0, -1.0, -1.0], [np.nan, 1.0, 3.0, 0.0]], np.float32)
    res = oracle.verify_greedy(lg, DT_F32, 4, np.array([0, 3], np.int32), np.array([1, 0], np.int32),
                               np.array([10], np.int32))
    assert list(res["argmax"]) == [1, 0, 2]
    assert res["accepted"][0] == 2 and res["correction"][0] == 2 and res["nans"] == 1


def test_golden_ragged_acceptance():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "ragged_acceptance.txt")) if not l.startswith("#")]
    V = 10
    rows, cu, drafts, ctx, expect = [], [0], [], [], []
    for t in lines:
        i_d, i_t, i_e = t.index("drafts"), t.index("targets"), t.index("expect")
        d = list(map(int, t[i_d + 1:i_t]))
        tg = list(map(int, t[i_t + 1:i_e]))
        for tok in tg:
            r = np.zeros(V, np.float32)
            r[tok] = 1.0
            rows.append(r)
        drafts += d
        cu.append(cu[-1] + len(tg))
        ctx.append(int(t[3]))
        expect.append(list(map(int, t[i_e + 1:])))
    res = oracle.verify_greedy(np.array(rows), DT_F32, V, np.array(cu, np.int32), np.array(drafts, np.int32),
                               np.array(ctx, np.int32))
    for s, (a, c, n) in enumerate(expect):
        assert (res["accepted"][s], res["correction"][s], res["ctx_new"][s]) == (a, c, n)


# ---------------------------------------------------------------------------
# KV compaction
# ---------------------------------------------------------------------------
def _slot(bt, s, pos):
    return bt[s, pos // 16], pos % 16


def test_kv_compact_full_acceptance_round_trips_every_staged_row():
    L = [3, 1, 6, 2]
    case = synth.compact_case(21, L, Hkv=2, D=8, ctx_range=(0, 60), accepted=L)
    kc, vc, cuk, src, dst = oracle.kv_compact(case.k_stage, case.v_stage, case.k_cache, case.v_cache, 2, 8,
                                              case.block_table, case.ctx_start, case.accepted, case.cu_rows)
    assert np.array_equal(cuk, np.concatenate([[0], np.cumsum(np.array(L) + 1)]))
    for s in range(4):
        for i in range(L[s] + 1):
            page, off = _slot(case.block_table, s, case.ctx_start[s] + i)
            r = case.cu_rows[s] + i
            assert np.array_equal(kc[page, :, off], case.k_stage[r])
            assert np.array_equal(vc[page, :, off], case.v_stage[r])
            j = cuk[s] + i
            assert src[j] == r and dst[j] == page * 16 + off


def test_kv_compact_rejected_rows_never_reach_the_cache():
    L = [5, 7, 2, 4, 1]
    case = synth.compact_case(22, L, Hkv=3, D=16, ctx_range=(10, 200))
    ks, vs = case.k_stage.copy(), case.v_stage.copy()
    for s in range(case.S):
        ks[case.cu_rows[s] + case.accepted[s] + 1:case.cu_rows[s + 1]] = 0xFFFF
        vs[case.cu_rows[s] + case.accepted[s] + 1:case.cu_rows[s + 1]] = 0xFFFF
    kc, vc, cuk, src, dst = oracle.kv_compact(ks, vs, case.k_cache, case.v_cache, 3, 16, case.block_table,
                                              case.ctx_start, case.accepted, case.cu_rows)
    assert not np.any(kc == 0xFFFF) and not np.any(vc == 0xFFFF)
    changed = np.any(kc != case.k_cache, axis=(1, 3)) | np.any(vc != case.v_cache, axis=(1, 3))
    assert changed.sum() == int((case.accepted + 1).sum())
    # in-place mode: same indices, cache untouched
    kc2, vc2, cuk2, src2, dst2 = oracle.kv_compact(None, None, case.k_cache, case.v_cache, 3, 16, case.block_table,
                                                   case.ctx_start, case.accepted, case.cu_rows)
    assert np.array_equal(kc2, case.k_cache) and np.array_equal(vc2, case.v_cache)
    assert np.array_equal(cuk2, cuk) and np.array_equal(src2, src) and np.array_equal(dst2, dst)


# ---------------------------------------------------------------------------
# decoder pieces
# ---------------------------------------------------------------------------
def test_rmsnorm_closed_forms():
    eps = 1e-5
    y = oracle.rmsnorm([3.0, 4.0], [1.0, 2.0], eps)
    r = math.sqrt((9 + 16) / 2 + eps)
    np.testing.assert_allclose(y, [3 / r, 8 / r], rtol=1e-15)
    y = oracle.rmsnorm(np.full(64, -2.5), np.ones(64), eps)
    np.testing.assert_allclose(y, -2.5 / math.sqrt(6.25 + eps), rtol=1e-15)


def test_rope_closed_forms_and_group_property():
    D, theta = 16, 10000.0
    g = np.random.default_rng(8)
    v = g.normal(size=D)
    assert np.array_equal(oracle.rope(v, 0, theta), v)
    for i in [0, 3, 7]:
        e = np.zeros(D)
        e[i] = 1.0
        p = 37
        ang = p * theta ** (-2.0 * i / D)
        out = oracle.rope(e, p, theta)
        want = np.zeros(D)
        want[i], want[i + D // 2] = math.cos(ang), math.sin(ang)
        np.testing.assert_allclose(out, want, atol=1e-15)
    a = oracle.rope(oracle.rope(v, 5, theta), 11, theta)
    np.testing.assert_allclose(a, oracle.rope(v, 16, theta), atol=1e-12)
    pair_norm = lambda x: x[:D // 2] ** 2 + x[D // 2:] ** 2
    np.testing.assert_allclose(pair_norm(oracle.rope(v, 123, theta)), pair_norm(v), rtol=1e-12)


def test_silu_mul_closed_forms():
    assert oracle.silu_mul(0.0, 5.0) == 0.0
    assert oracle.silu_mul(1.0, 1.0) == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    assert oracle.silu_mul(40.0, 0.5) == pytest.approx(20.0, rel=1e-15)
    assert abs(oracle.silu_mul(-40.0, 1.0)) < 1e-15


def test_decoder_layer_with_zero_output_weights_is_identity_on_the_residual():
    cfg = synth.TINY_DECODER
    w = synth.decoder_weights(3, cfg)
    for lay in w.layers:
        for key in ("o", "down"):
            wq, ws = lay[key]
            lay[key] = (np.full_like(wq, 0x88), ws)     # every nibble encodes q = 0
    dec = oracle.Decoder(w, 2, 64)
    tokens = np.array([1, 2, 3, 4, 5], np.int32)
    h = dec.embed(tokens)
    h2 = dec.layer(0, h.copy(), np.array([0, 0], np.int32), np.array([0, 3, 5], np.int32))
    assert np.array_equal(h2, h)
    # the layer still wrote K/V for every block row at its position
    assert np.count_nonzero(np.any(dec.k_cache[0] != 0, axis=(1, 3))) == 5


def test_embedding_rows_are_the_table_rows():
    cfg = synth.TINY_DECODER
    w = synth.decoder_weights(3, cfg)
    dec = oracle.Decoder(w, 1, 16)
    h = dec.embed([5, 0, 96])
    assert np.array_equal(h, synth.bf16_bits_to_f32(w.emb[[5, 0, 96]]))


# ---------------------------------------------------------------------------
# n-gram drafting
# ---------------------------------------------------------------------------
def test_ngram_draft_hand_examples():
    pad = np.array([90, 91, 92, 93], np.int32)
    out, n = oracle.ngram_draft([1, 2, 3, 4, 1, 2, 3], 4, pad)
    assert list(out) == [4, 1, 2, 3] and n == 3
    out, n = oracle.ngram_draft([5, 6, 7, 5, 6], 4, pad)      # bigram [5, 6] at 0 -> 7 5 6
    assert list(out) == [7, 5, 6, 93] and n == 2
    out, n = oracle.ngram_draft([1, 9, 1, 8, 1], 4, pad)      # unigram, most recent earlier at 2 -> 8 1
    assert list(out) == [8, 1, 92, 93] and n == 1
    out, n = oracle.ngram_draft([4, 5, 6], 4, pad)            # nothing repeats
    assert list(out) == [90, 91, 92, 93] and n == 0
    out, n = oracle.ngram_draft([7], 4, pad)
    assert list(out) == [90, 91, 92, 93] and n == 0
    out, n = oracle.ngram_draft([2, 2, 2, 2, 2], 4, pad)      # most recent earlier trigram at 1 -> 2
    assert list(out) == [2, 91, 92, 93] and n == 3


# ---------------------------------------------------------------------------
# the method's invariant: speculative greedy output equals width-1 greedy output
# ---------------------------------------------------------------------------
def test_oracle_speculative_greedy_equals_width1_greedy_tiny_decoder():
    cfg = synth.TINY_DECODER
    w = synth.decoder_weights(1005, cfg)
    pr = synth.prompts(1006, 3, 12, cfg.vocab)
    pads = synth.pad_tokens(1007, 3, 64, 4, cfg.vocab)
    base, steps1, _ = oracle.generate(w, pr, 24, 0, pads)
    spec, steps4, acc = oracle.generate(w, pr, 24, 4, pads)
    assert np.array_equal(base, spec)
    assert steps1 == 24 and steps4 <= 24
