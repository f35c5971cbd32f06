"""Margin-gated re-check of the LM head on the GPU (tokenstrom.com, "'Lossless,'
but not quite", sections "Why the math checks out and the text still flips"
and "What the big servers offer and what it costs").

The fast logits come from spec_qmatmul_noninvariant (its K-segments differ
from the invariant ones), the gate flags the rows whose top-2 margin is within
twice the summation-order bound, the flagged rows are re-evaluated by the
invariant product and copied back.  Checked: the bound holds entry by entry;
the gate flags what the oracle's gate flags on the same logits; the gated
argmax of every row equals the invariant argmax (planted exact ties and near
ties included) and the oracle's wherever the oracle's own margin is clear of
the kernels' tolerance; and the overflow path."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, dev, host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def err_coef(ws_bits, K):
    """The summation-order bound per unit ||x||_1: two fp32 evaluations of the same
    K/32 block terms differ by at most 2 gamma_(2n) sum|t_b| (n = K/32 blocks, at most
    2n roundings on any term's path), and |t_b| = |d_b P_b| <= 9 max|d| ||x_b||_1."""
    n = K // 32
    gamma = 2 * n * U / (1 - 2 * n * U)
    dmax = float(np.abs(np.asarray(ws_bits, np.uint16).view(np.float16).astype(np.float64)).max())
    return 2 * gamma * 9 * dmax


def lm_case(seed, V, H, R, n_tie, n_near):
    """LM-head weights and R activation rows; rows 0..n_tie-1 aim at a vocabulary row
    that has an exact copy elsewhere, the next n_near at one with a one-code variant."""
    g = np.random.default_rng(seed)
    w = g.normal(0, 0.02, (V, H)).astype(np.float32)
    wq, ws = synth.quantize_q4b32(w)
    x = g.normal(0, 1, (R, H)).astype(np.float32)
    codes = np.stack([(wq & 15), (wq >> 4)], axis=-1).reshape(V, H).astype(np.int64) - 8
    deq = codes * np.repeat(ws.view(np.float16).astype(np.float32), 32, axis=1)
    for r in range(n_tie + n_near):
        t = int(g.integers(0, V))
        u = int(g.integers(0, V))
        while u == t:
            u = int(g.integers(0, V))
        wq[u], ws[u] = wq[t], ws[t]
        if r >= n_tie:
            # one code one step off in the block with the smallest scale: a near tie
            b = int(np.argmin(ws[t].view(np.float16)))
            byte = wq[u, 16 * b]
            lo = byte & 15
            wq[u, 16 * b] = (byte & 0xF0) | (lo + 1 if lo < 15 else lo - 1)
        # aim row r at t: large positive logit for t (and its copy)
        x[r] = np.sign(deq[t] + 1e-12) * np.abs(x[r])
    xb = synth.f32_to_bf16_bits(x)
    return wq, ws, xb


def run_gate(L, wq, ws, xb, V, H, R, capacity, noninv_seg=4):
    d = "cuda"
    wq_d, ws_d, x_d = dev(wq), dev(ws), dev(xb)
    wsb = max(L.spec_qmatmul_workspace(V, H, R), L.spec_qmatmul_workspace(V, H, capacity))
    wsp = torch.zeros(wsb // 4 + 64, dtype=torch.int32, device=d)
    inv = torch.zeros((R, V), dtype=torch.float32, device=d)
    fast = torch.zeros((R, V), dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    L.spec_qmatmul(wq_d, ws_d, V, H, x_d, R, H, inv, L.SPEC_F32, V, 0, wsp, wsb, err)
    L.spec_qmatmul_noninvariant(wq_d, ws_d, V, H, x_d, R, H, fast, V, noninv_seg, wsp, wsb)
    torch.cuda.synchronize()
    fast_host = host(fast).copy()
    coef = err_coef(ws, H)
    gwb = L.spec_margin_gate_workspace(R, V)
    gws = torch.empty(gwb // 4 + 16, dtype=torch.float32, device=d)
    top = torch.zeros(R, dtype=torch.int32, device=d)
    rows = torch.full((capacity,), -1, dtype=torch.int32, device=d)
    cnt = torch.zeros(1, dtype=torch.int32, device=d)
    ovf = torch.zeros(1, dtype=torch.int32, device=d)
    xg = torch.zeros((capacity, H), dtype=torch.int16, device=d)
    yg = torch.zeros((capacity, V), dtype=torch.float32, device=d)
    L.spec_margin_gate(fast, V, R, x_d, H, H, coef, top, rows, cnt, ovf, capacity, xg, gws, gwb, err)
    L.spec_qmatmul_devcols(wq_d, ws_d, V, H, xg, capacity, H, yg, L.SPEC_F32, V, 0, cnt, 1, wsp, wsb, err)
    L.spec_gate_scatter(yg, V, rows, cnt, capacity, fast)
    L.spec_qmatmul_devcols(wq_d, ws_d, V, H, x_d, R, H, fast, L.SPEC_F32, V, 0, ovf, 1, wsp, wsb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return dict(inv=host(inv), fast0=fast_host, gated=host(fast), top=host(top), rows=host(rows),
                count=int(cnt.item()), overflow=int(ovf.item()), coef=coef)


def first_argmax(a):
    return np.argmax(a, axis=1)   # numpy: first occurrence of the maximum


@pytest.mark.parametrize("R,capacity", [(80, 16), (80, 2)], ids=["fits", "overflow"])
def test_gate_gives_the_invariant_argmax(R, capacity):
    import invariant_speculative_verification_gb300 as L
    V, H = 32000, 2048
    wq, ws, xb = lm_case(77, V, H, R, n_tie=3, n_near=3)
    res = run_gate(L, wq, ws, xb, V, H, R, capacity)
    xnorm = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)).sum(axis=1)
    errs = res["coef"] * xnorm
    # the bound holds entry by entry
    diff = np.abs(res["fast0"].astype(np.float64) - res["inv"].astype(np.float64)).max(axis=1)
    assert np.all(diff <= errs), (diff / errs).max()
    assert diff.max() > 0          # the fast path really differs
    # the GPU gate flags what the oracle's gate flags (away from the threshold itself)
    otop, omargin, oflag = oracle.margin_gate(res["fast0"], errs)
    assert np.array_equal(res["top"], otop)
    clear = np.abs(omargin - 2 * errs) > 1e-2 * errs
    flagged = np.zeros(R, bool)
    if capacity < 3:
        assert res["count"] > capacity and res["overflow"] == R
    else:
        assert res["overflow"] == 0
        flagged[res["rows"][:res["count"]]] = True
        assert np.array_equal(flagged[clear], oflag[clear])
        assert list(res["rows"][:res["count"]]) == sorted(res["rows"][:res["count"]])
    assert res["count"] == int(oflag.sum()) or not np.all(clear)
    assert np.all(oflag[:3])       # planted exact ties are re-checked (3 > capacity 2: overflow)
    # every row's gated argmax is the invariant argmax; re-checked rows are bitwise invariant
    inv_top = first_argmax(res["inv"])
    assert np.array_equal(first_argmax(res["gated"]), inv_top)
    for r in np.nonzero(oflag)[0]:
        assert np.array_equal(res["gated"][r].view(np.int32), res["inv"][r].view(np.int32))
    # the oracle agrees wherever its own margin is clear of the kernels' tolerance
    ref = oracle.qmatmul(wq, ws, xb, V, H)
    o_sorted = np.sort(ref, axis=1)
    o_margin = o_sorted[:, -1] - o_sorted[:, -2]
    sure = o_margin > 2 * TOL * np.abs(ref).max(axis=1)
    assert np.array_equal(inv_top[sure], first_argmax(ref)[sure])
    # exact ties in the oracle: the lowest index wins on the GPU too
    for r in range(3):
        assert inv_top[r] == int(np.flatnonzero(ref[r] == ref[r].max())[0])


def test_gate_with_nothing_flagged_leaves_the_fast_logits():
    import invariant_speculative_verification_gb300 as L
    V, H, R = 4096, 1024, 8
    g = np.random.default_rng(5)
    wq, ws = synth.quantize_q4b32(g.normal(0, 0.02, (V, H)).astype(np.float32))
    xb = synth.f32_to_bf16_bits(g.normal(0, 1, (R, H)).astype(np.float32))
    res = run_gate(L, wq, ws, xb, V, H, R, 8)
    xnorm = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)).sum(axis=1)
    _, _, oflag = oracle.margin_gate(res["fast0"], res["coef"] * xnorm)
    keep = ~oflag
    assert np.array_equal(res["gated"][keep].view(np.int32), res["fast0"][keep].view(np.int32))
    assert np.array_equal(first_argmax(res["gated"]), first_argmax(res["inv"]))


@pytest.mark.parametrize("cfg_name", ["small", "full_size"])
def test_gated_speculative_generation_equals_invariant_width1(cfg_name):
    """Speculative decoding whose LM head runs through the margin gate produces the
    same bytes as ordinary width-1 decoding with the invariant LM head."""
    from invariant_speculative_verification_gb300.decoder import Decoder, Generator, max_len_for
    cfg = (synth.DecoderConfig(layers=2, hidden=256, heads=4, kv_heads=2, head_dim=64, ffn=512, vocab=1024)
           if cfg_name == "small" else synth.E2E_DECODER)
    S, P, n_new = (8, 32, 96) if cfg_name == "small" else (16, 128, 128)
    w = synth.decoder_weights(1005, cfg)
    pr = synth.prompts(1006, S, P, cfg.vocab)
    pads = synth.pad_tokens(1007, S, 512, 4, cfg.vocab).transpose(1, 0, 2).copy()

    def run(W, gated):
        dec = Decoder(w, S, max_len_for(P, n_new, W), max_rows=max(S * (P - 1), S * (W + 1)))
        if gated:
            dec.enable_gate(capacity=16)
        gen = Generator(dec, pr, W, pads, n_new)
        toks = gen.run(use_graph=True)
        assert int(dec.dev_err.item()) == 0
        return toks

    base = run(0, False)
    gated = run(4, True)
    assert np.array_equal(base, gated)
