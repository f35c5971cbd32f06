"""Activations packed by their producer for an 80-column K1 pass.

spec_add_rmsnorm_packed / spec_swiglu_packed write the rows they produce both
in the plain layout and in the packed stage layout of the 80-column pass;
spec_qmatmul_packed runs that pass from the packed form.  Only the delivery of
the activations changes (ramgpt.org, "When Lossless Speculation Stops Being
Lossless on Blackwell", section "Quantized Matrix Multiplication Shows the
Same Class of Failure"): the plain outputs and the products must equal the
plain calls' bit for bit, and the product must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, bits_equal, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu


def _L():
    import invariant_speculative_verification_gb300 as L
    return L


def _matmul_pair(L, wq, ws, N, K, x, R, xpk, accumulate=0, y0=None):
    """(plain spec_qmatmul, spec_qmatmul_packed) outputs [R][N] fp32."""
    wsb = L.spec_qmatmul_workspace(N, K, R)
    outs = []
    for packed in (False, True):
        wsp = torch.zeros(wsb // 4 + 64, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = y0.clone() if y0 is not None else torch.zeros((R, N), dtype=torch.float32, device="cuda")
        if packed:
            L.spec_qmatmul_packed(wq, ws, N, K, xpk, R, y, L.SPEC_F32, N, accumulate, wsp, wsb, err)
        else:
            L.spec_qmatmul(wq, ws, N, K, x, R, K, y, L.SPEC_F32, N, accumulate, wsp, wsb, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(y)
    return outs


@pytest.mark.parametrize("R", [17, 37, 80])
def test_rmsnorm_packed_feeds_the_wide_pass_bit_for_bit(R):
    L = _L()
    g = np.random.default_rng(40 + R)
    N, H = 3072, 2048
    h = g.normal(0, 1, (R, H)).astype(np.float32)
    w = g.normal(1, 0.1, H).astype(np.float32)
    wq, ws = synth.qmatmul_weights(900 + R, N, H)
    wqd, wsd = dev(wq), dev(ws)
    plain = torch.zeros((R, H), dtype=torch.int16, device="cuda")
    packed = torch.zeros((R, H), dtype=torch.int16, device="cuda")
    xpk = torch.full((L.spec_packed_activation_bytes(H) // 4 + 16,), -1, dtype=torch.int32, device="cuda")
    L.spec_add_rmsnorm(dev(h), None, dev(w), R, H, 1e-5, plain)
    L.spec_add_rmsnorm_packed(dev(h), None, dev(w), R, H, 1e-5, packed, xpk)
    torch.cuda.synchronize()
    assert bits_equal(plain, packed)
    y_plain, y_packed = _matmul_pair(L, wqd, wsd, N, H, plain, R, xpk)
    assert bits_equal(y_plain, y_packed)
    rows = [0, R // 2, R - 1]
    ref = oracle.qmatmul(wq, ws, host(plain, np.uint16)[rows], N, H)
    assert rel_err_rows(host(y_packed)[rows], ref) <= TOL


@pytest.mark.parametrize("R", [23, 80])
def test_swiglu_packed_feeds_the_wide_pass_bit_for_bit_with_accumulate(R):
    L = _L()
    g = np.random.default_rng(60 + R)
    N, F = 2048, 5632
    gu = g.normal(0, 2, (R, 2 * F)).astype(np.float32)
    wq, ws = synth.qmatmul_weights(950 + R, N, F)
    wqd, wsd = dev(wq), dev(ws)
    plain = torch.zeros((R, F), dtype=torch.int16, device="cuda")
    packed = torch.zeros((R, F), dtype=torch.int16, device="cuda")
    xpk = torch.full((L.spec_packed_activation_bytes(F) // 4 + 16,), -1, dtype=torch.int32, device="cuda")
    gud = dev(gu)
    L.spec_swiglu(gud, R, F, plain)
    L.spec_swiglu_packed(gud, R, F, packed, xpk)
    torch.cuda.synchronize()
    assert bits_equal(plain, packed)
    y0 = torch.from_numpy(g.normal(0, 1, (R, N)).astype(np.float32)).cuda()
    y_plain, y_packed = _matmul_pair(L, wqd, wsd, N, F, plain, R, xpk, accumulate=1, y0=y0)
    assert bits_equal(y_plain, y_packed)


def test_packed_arguments_are_checked():
    L = _L()
    xpk = torch.zeros(L.spec_packed_activation_bytes(2048) // 4 + 16, dtype=torch.int32, device="cuda")
    wq, ws = synth.qmatmul_weights(7, 512, 2048)
    y = torch.zeros((81, 512), dtype=torch.float32, device="cuda")
    wsb = L.spec_qmatmul_workspace(512, 2048, 81)
    wsp = torch.zeros(wsb // 4 + 64, dtype=torch.int32, device="cuda")
    assert L.spec_packed_activation_bytes(1000) == 0
    for n_cols in (16, 81):
        with pytest.raises(L.SpecError):
            L.spec_qmatmul_packed(dev(wq), dev(ws), 512, 2048, xpk, n_cols, y, L.SPEC_F32, 512, 0, wsp, wsb)
    out = torch.zeros((81, 2048), dtype=torch.int16, device="cuda")
    h = torch.zeros((81, 2048), dtype=torch.float32, device="cuda")
    w = torch.ones(2048, dtype=torch.float32, device="cuda")
    with pytest.raises(L.SpecError):
        L.spec_add_rmsnorm_packed(h, None, w, 81, 2048, 1e-5, out, xpk)


def test_attention_packed_feeds_the_o_projection_bit_for_bit():
    L = _L()
    Hq, Hkv, D, S, W = 16, 4, 128, 16, 5
    R = S * W
    g = np.random.default_rng(77)
    ctx = g.integers(100, 600, size=S).astype(np.int32)
    c = synth.attention_case(78, rows=[W] * S, ctx=list(ctx), Hq=Hq, Hkv=Hkv, D=D, dt=synth.DT_BF16,
                             q_std=1 / np.sqrt(D), scale=1.0)
    max_len = int((ctx + W).max())
    q, kc, vc, bt = dev(c.q), dev(c.k_cache), dev(c.v_cache), dev(c.block_table)
    cs, cu = dev(c.ctx_start), dev(c.cu_rows)
    wsb = L.spec_flash_decode_workspace(R, Hq, D, max_len)
    xpk = torch.full((L.spec_packed_activation_bytes(Hq * D) // 4 + 16,), -1, dtype=torch.int32, device="cuda")
    outs = []
    for packed in (False, True):
        ws = torch.empty(wsb // 4 + 64, dtype=torch.float32, device="cuda")
        out = torch.zeros((R, Hq * D), dtype=torch.int16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (q, L.SPEC_BF16, Hq, Hkv, D, 1.0, kc, vc, c.k_cache.shape[0], bt, c.block_table.shape[1], cs, cu, S, R,
                max_len, out)
        if packed:
            L.spec_flash_decode_packed(*args, ws, wsb, xpk, err)
        else:
            L.spec_flash_decode(*args, L.SPEC_BF16, ws, wsb, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(out)
    assert bits_equal(outs[0], outs[1])
    N, K = 2048, Hq * D
    wq, ws_ = synth.qmatmul_weights(79, N, K)
    y0 = torch.from_numpy(g.normal(0, 1, (R, N)).astype(np.float32)).cuda()
    y_plain, y_packed = _matmul_pair(L, dev(wq), dev(ws_), N, K, outs[0], R, xpk, accumulate=1, y0=y0)
    assert bits_equal(y_plain, y_packed)


def _interleave_gate_up(wq, ws, F):
    """Rows of a [gate; up] matrix reordered as spec_qmatmul_swiglu takes them:
    per group of 8 features its 8 gate rows, then their 8 up rows."""
    g = np.arange(F).reshape(-1, 8)
    perm = np.concatenate([g, g + F], axis=1).reshape(-1)
    return np.ascontiguousarray(wq[perm]), np.ascontiguousarray(ws[perm])


@pytest.mark.parametrize("F,K,R", [(5632, 2048, 80), (5632, 2048, 33), (5632, 2048, 16), (5632, 2048, 5),
                                   (40, 512, 23)])
def test_fused_swiglu_equals_matmul_then_swiglu_bit_for_bit(F, K, R):
    """spec_qmatmul_swiglu (interleaved gate/up rows) writes exactly what
    spec_qmatmul on the [gate; up] rows followed by spec_swiglu writes, from
    plain and (17-80 rows) from packed activations; sampled features agree with
    the oracle's SwiGLU of the oracle's products."""
    L = _L()
    g = np.random.default_rng(70 + F + R)
    h = g.normal(0, 1, (R, K)).astype(np.float32)
    w = g.normal(1, 0.1, K).astype(np.float32)
    wq, ws = synth.qmatmul_weights(950 + R, 2 * F, K)
    wqi, wsi = _interleave_gate_up(wq, ws, F)
    a = torch.zeros((R, K), dtype=torch.int16, device="cuda")
    xpk = torch.full((L.spec_packed_activation_bytes(K) // 4 + 16,), -1, dtype=torch.int32, device="cuda")
    L.spec_add_rmsnorm_packed(dev(h), None, dev(w), R, K, 1e-5, a, xpk)
    wsb = L.spec_qmatmul_workspace(2 * F, K, R)
    wsp = torch.zeros(wsb // 4 + 64, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gu = torch.zeros((R, 2 * F), dtype=torch.float32, device="cuda")
    L.spec_qmatmul(dev(wq), dev(ws), 2 * F, K, a, R, K, gu, L.SPEC_F32, 2 * F, 0, wsp, wsb, err)
    ref = torch.zeros((R, F), dtype=torch.int16, device="cuda")
    L.spec_swiglu(gu, R, F, ref)
    outs = []
    for use_pk in ((False, True) if 16 < R <= 80 else (False,)):
        act = torch.full((R, F), -1, dtype=torch.int16, device="cuda")
        L.spec_qmatmul_swiglu(dev(wqi), dev(wsi), F, K, a, xpk if use_pk else None, R, K, act, F, wsp, wsb, err)
        outs.append(act)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for act in outs:
        assert bits_equal(act, ref)
    assert int(wsp[:16384].abs().sum().item()) == 0
    rows = sorted({0, R // 2, R - 1})
    feats = sorted({0, 7, 8, F // 2, F - 1})
    xa = host(a, np.uint16)[rows]
    gate = oracle.qmatmul(wq[feats], ws[feats], xa, len(feats), K)
    up = oracle.qmatmul(wq[[F + f for f in feats]], ws[[F + f for f in feats]], xa, len(feats), K)
    want = np.array([[oracle.silu_mul(gate[i, j], up[i, j]) for j in range(len(feats))] for i in range(len(rows))])
    got = synth.bf16_bits_to_f32(host(outs[0], np.uint16))[np.ix_(rows, feats)]
    # bf16 rounding of the result plus the products' own tolerance; a swapped
    # gate/up pair or a wrong feature row is off by O(1)
    assert rel_err_rows(got, want) <= 2 ** -6


def test_fused_swiglu_arguments_are_checked():
    L = _L()
    x = torch.zeros((4, 512), dtype=torch.int16, device="cuda")
    w = torch.zeros(64 * 256, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64 * 16, dtype=torch.int16, device="cuda")
    act = torch.zeros((4, 32), dtype=torch.int16, device="cuda")
    wsp = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    with pytest.raises(L.SpecError, match="multiple of 8"):
        L.spec_qmatmul_swiglu(w, s, 30, 512, x, None, 4, 512, act, 32, wsp, wsp.numel() * 4)
    with pytest.raises(L.SpecError, match="ld_act"):
        L.spec_qmatmul_swiglu(w, s, 32, 512, x, None, 4, 512, act, 16, wsp, wsp.numel() * 4)
