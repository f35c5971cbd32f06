"""Pins of the margin gate (tokenstrom.com, "'Lossless,' but not quite",
sections "Why the math checks out and the text still flips" and "What the big
servers offer and what it costs": only steps with a small top-2 margin can
flip, so only those need the expensive re-check).

* the oracle's gate against an independent sort-based formulation (brute
  force over small rows with ties);
* its boundary cases (margin exactly 2 err re-checked, exact ties re-checked,
  one-entry rows never);
* the theorem the gate rests on: when every fast logit lies within err of the
  invariant one and the margin exceeds 2 err, both argmaxes agree (Monte Carlo
  over planted near-ties and worst-case perturbations);
* the error bound's form: two fp32 evaluation orders of the same block sums
  (fused multiply-add chains cut into segments of different lengths, then
  the segments added in order) differ by at most 2 gamma_(n-1) sum |t_b|,
  gamma_k = k u / (1 - k u), u = 2^-24 -- checked on adversarial and random
  inputs with numpy's own float32 arithmetic."""
import numpy as np
import pytest

import oracle

U = 2.0 ** -24


def gamma(k):
    return k * U / (1 - k * U)


def test_gate_matches_a_sort_based_formulation():
    g = np.random.default_rng(3)
    for _ in range(3000):
        V = int(g.integers(1, 7))
        row = g.integers(-3, 4, size=V).astype(np.float32) * np.float32(0.5)
        err = float(g.choice([0.0, 0.1, 0.25, 0.5, 1.0]))
        top, margin, flag = oracle.margin_gate(row[None, :], [err])
        order = sorted(range(V), key=lambda v: (-float(row[v]), v))
        assert top[0] == order[0]
        exp_margin = np.inf if V == 1 else float(row[order[0]]) - float(row[order[1]])
        assert margin[0] == exp_margin
        assert flag[0] == (exp_margin <= 2 * err)


def test_gate_boundaries():
    lg = np.array([[1.0, 0.5, 0.0], [2.0, 2.0, 1.0], [0.0, 0.0, 7.0]], np.float32)
    top, margin, flag = oracle.margin_gate(lg, [0.25, 10.0, 3.5])
    assert list(top) == [0, 0, 2]
    assert list(margin) == [0.5, 0.0, 7.0]
    assert list(flag) == [True, True, True]           # 0.5 <= 0.5; a tie; 7 <= 7
    _, m1, f1 = oracle.margin_gate(np.array([[4.0]], np.float32), [100.0])
    assert m1[0] == np.inf and not f1[0]


def test_unflagged_rows_keep_the_invariant_argmax():
    g = np.random.default_rng(11)
    R, V = 400, 257
    inv = g.normal(0, 1, (R, V)).astype(np.float32)
    # planted near-ties: the runner-up a hair below (or equal to) the top
    for r in range(0, R, 3):
        t = int(np.argmax(inv[r]))
        u = int(g.integers(0, V))
        if u != t:
            inv[r, u] = inv[r, t] - np.float32(g.choice([0.0, 1e-4, 1e-3]))
    err = np.full(R, 1e-3)
    fast = inv + (g.uniform(-1, 1, (R, V)) * err[:, None]).astype(np.float32)
    # worst case too: push the runner-up up and the top down by err
    for r in range(1, R, 7):
        t = int(np.argmax(inv[r]))
        fast[r] = inv[r] + np.float32(err[r])
        fast[r, t] = inv[r, t] - np.float32(err[r])
    dev = np.abs(fast.astype(np.float64) - inv.astype(np.float64)).max(axis=1)
    err_eff = np.maximum(err, dev)           # fp32 rounding of the perturbation
    top, margin, flag = oracle.margin_gate(fast, err_eff)
    inv_top, _, _ = oracle.margin_gate(inv, np.zeros(R))
    assert np.all(top[~flag] == inv_top[~flag])
    assert flag.sum() > 0 and (~flag).sum() > 0


def _chain(t, seg):
    """fp32: fused multiply-add chains of the block terms (d, p) within segments of
    `seg` blocks from +0, then the segment sums added in order."""
    d, p = t
    total = None
    for s0 in range(0, len(d), seg):
        s = np.float32(0.0)
        for b in range(s0, min(s0 + seg, len(d))):
            s = np.float32(np.float64(d[b]) * np.float64(p[b]) + np.float64(s))   # one rounding, as fma
        total = s if total is None else np.float32(total + s)
    return float(total)


@pytest.mark.parametrize("n", [16, 64, 176])
def test_two_evaluation_orders_differ_by_at_most_the_bound(n):
    g = np.random.default_rng(n)
    for trial in range(200):
        d = (np.abs(g.normal(0, 0.01, n)) + 1e-4).astype(np.float32)
        if trial % 2:   # cancellation-heavy: alternating large terms
            p = (g.normal(0, 1, n) * 1e3 * np.where(np.arange(n) % 2, 1, -1)).astype(np.float32)
        else:
            p = g.normal(0, 5, n).astype(np.float32)
        exact = float(np.sum(np.float64(d) * np.float64(p)))
        bound = gamma(n - 1) * float(np.sum(np.abs(np.float64(d) * np.float64(p))))
        a, b = _chain((d, p), 16), _chain((d, p), 64)
        assert abs(a - exact) <= bound and abs(b - exact) <= bound
        assert abs(a - b) <= 2 * bound
