"""K1 with two-level (super-block) scales (spec_qmatmul_sb): parity with the
oracle and the same bit-exact batch invariance as the single-level product.

The format is self-defined (the pages name Q4_K / Q6_K and IQ3_S / IQ4_XS in
tokenstrom.com, "'Lossless,' but not quite", section "Why the math checks out
and the text still flips", and ramgpt.org, "When Lossless Speculation Stops
Being Lossless on Blackwell", section "Quantized Matrix Multiplication Shows the
Same Class of Failure", but define none); the invariance test shape is that
section's: a batched product against a sequence of single-column products.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, bits_equal, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu

_WS = {}


def _lib():
    import invariant_speculative_verification_gb300 as L
    return L


def workspace(nbytes):
    if "ws" not in _WS or _WS["ws"].numel() * 4 < nbytes:
        _WS["ws"] = torch.zeros(nbytes // 4 + 1024, dtype=torch.int32, device="cuda")
    return _WS["ws"]


def run(w, x, n_cols, N, K, out_dt=0, y=None, accumulate=0, fmt="sb"):
    L = _lib()
    if y is None:
        y = torch.zeros((max(n_cols, 1), N), dtype=torch.float32 if out_dt == 0 else torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsp = workspace(L.spec_qmatmul_workspace(N, K, max(n_cols, 1)))
    f = L.spec_qmatmul_sb if fmt == "sb" else L.spec_qmatmul
    f(w[0], w[1], N, K, x, n_cols, K, y, out_dt, N, accumulate, wsp, wsp.numel() * 4, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return y


def upload(case):
    return (dev(case.wq), dev(case.ws)), dev(case.x)


@pytest.mark.parametrize("N,K,n", [(512, 512, 8), (200, 768, 5), (1000, 2048, 5), (96, 5120, 3), (130, 17408, 4)])
def test_parity_and_width_invariance(N, K, n):
    """Odd super-block counts (K = 768: a padding record), several K-segments, ragged N."""
    case = synth.qmatmul_sb_case(9100 + N + K, N, K, n)
    w, x = upload(case)
    y = run(w, x, n, N, K)
    assert rel_err_rows(host(y), oracle.qmatmul_sb(case.wq, case.ws, case.x, N, K)) <= TOL
    for j in range(n):
        assert bits_equal(run(w, x[j:j + 1], 1, N, K)[0], y[j]), j


@pytest.mark.parametrize("n", [16, 17, 80, 81])
def test_wide_passes_keep_every_column_bit_identical(n):
    """16 columns (narrow pass), 17 and 80 (one 80-column pass), 81 (two passes)."""
    N, K = 300, 1280
    case = synth.qmatmul_sb_case(9200 + n, N, K, n)
    w, x = upload(case)
    y = run(w, x, n, N, K)
    assert rel_err_rows(host(y), oracle.qmatmul_sb(case.wq, case.ws, case.x, N, K)) <= TOL
    for j in sorted({0, 7, n // 2, n - 1}):
        assert bits_equal(run(w, x[j:j + 1], 1, N, K)[0], y[j]), j


def test_equals_single_level_product_bit_for_bit_when_scales_coincide():
    """With D a power of two, D * s is an exact fp16 value: both formats then hand the
    kernel the same fp32 block scale, so the results must be identical bits."""
    N, K, n = 700, 2816, 9
    g = np.random.default_rng(4)
    codes = g.integers(0, 16, size=(N, K))
    wq = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    D = np.ldexp(1.0, g.integers(-14, -6, size=(N, K // 256))).astype(np.float16)
    s = g.integers(0, 64, size=(N, K // 32))
    sbr = synth.pack_sb_records(s, D.view(np.uint16))
    d = (np.repeat(D.astype(np.float64), 8, axis=1) * s).astype(np.float16)
    x = dev(synth.activations_bf16(5, n, K))
    y_sb = run((dev(wq), dev(sbr)), x, n, N, K)
    y_1 = run((dev(wq), dev(d.view(np.uint16))), x, n, N, K, fmt="block")
    assert bits_equal(y_sb, y_1)


def test_bf16_output_and_accumulate():
    N, K = 512, 1024
    case = synth.qmatmul_sb_case(9300, N, K, 4)
    w, x = upload(case)
    y32 = run(w, x, 4, N, K)
    assert torch.equal(run(w, x, 4, N, K, out_dt=2), y32.to(torch.bfloat16))
    base = torch.randn(4, N, device="cuda")
    acc = base.clone()
    run(w, x, 4, N, K, y=acc, accumulate=1)
    assert bits_equal(acc, base + y32)


def test_full_size_sampled_parity_and_invariance():
    """A 27B-class projection (17408 x 5120): widths 1-8 bitwise against width-1
    calls, parity on sampled output rows."""
    N, K = 17408, 5120
    case = synth.qmatmul_sb_case(9400, N, K, 8)
    w, x = upload(case)
    singles = torch.cat([run(w, x[j:j + 1], 1, N, K) for j in range(8)])
    for n in (2, 3, 5, 8):
        assert bits_equal(run(w, x, n, N, K)[:n], singles[:n]), n
    rows = np.random.default_rng(8).choice(N, 32, replace=False)
    ref = oracle.qmatmul_sb_rows(case.wq, case.ws, case.x, K, rows)
    got = host(singles)[:, rows]
    scale = np.abs(host(singles)).max(axis=1, keepdims=True)
    assert float((np.abs(got - ref) / scale).max()) <= TOL


def test_host_checks():
    L = _lib()
    case = synth.qmatmul_sb_case(9500, 128, 512, 1)
    w, x = upload(case)
    y = torch.zeros((1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul_sb(w[0], w[1], 128, 512, x, 1, 512, y, 0, 128, 0, workspace(1 << 20), 16)
    assert e.value.status == 3
    with pytest.raises(L.SpecError):
        L.spec_qmatmul_sb(w[0], w[1], 128, 500, x, 1, 512, y, 0, 128, 0, workspace(1 << 20), 1 << 20)
