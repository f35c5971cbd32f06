"""K1 (spec_qmatmul): parity with the oracle and bit-exact batch invariance.

Batch invariance test shape from ramgpt.org, "When Lossless Speculation Stops
Being Lossless on Blackwell", sections "Quantized Matrix Multiplication Shows
the Same Class of Failure" (batched product vs a sequence of single-column
products) and "A Better Backend Test Matrix" (widths 2, 3, 4, 5 and 8).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, bits_equal, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu

WIDTHS = [1, 2, 3, 4, 5, 8]


def _lib():
    import invariant_speculative_verification_gb300 as L
    return L


_WS = {}


def workspace(nbytes):
    """A zero-filled workspace shared by the calls of this module (calls leave it zeroed)."""
    key = "ws"
    if key not in _WS or _WS[key].numel() * 4 < nbytes:
        _WS[key] = torch.zeros(nbytes // 4 + 1024, dtype=torch.int32, device="cuda")
    return _WS[key]


def run(case_or_w, x_dev, n_cols, N, K, ldx=None, out_dt=0, y=None, accumulate=0, ldy=None):
    L = _lib()
    wq, ws = case_or_w
    ldx = K if ldx is None else ldx
    ldy = N if ldy is None else ldy
    if y is None:
        y = torch.zeros((max(n_cols, 1), ldy), dtype=torch.float32 if out_dt == 0 else torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = L.spec_qmatmul_workspace(N, K, max(n_cols, 1))
    wsp = workspace(need)
    L.spec_qmatmul(wq, ws, N, K, x_dev, n_cols, ldx, y, out_dt, ldy, accumulate, wsp, wsp.numel() * 4, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return y


def debug_nt_ws(N, K, nt):
    tiles = (N + 127) // 128
    ncg = 1
    if nt == 12:      # 16-column passes, up to five column groups in one launch
        nt, ncg = 2, 5
    elif nt == 13:    # 8-column passes, up to ten column groups in one launch
        nt, ncg = 1, 10
    packed = (K // 256) * 43520 if nt >= 10 else 0   # the 80-column pass's packed activations
    nt = min(nt, 10)
    t = tiles * ncg
    return ((t * 4 + 255) // 256) * 256 + t * (1 + (K + 511) // 512) * 128 * 8 * nt * 4 + packed


@pytest.fixture(scope="module")
def tiny():
    case = synth.qmatmul_case(1001, 512, 512, 8)
    return case, (dev(case.wq), dev(case.ws)), dev(case.x)


def test_parity_tiny_all_widths(tiny):
    case, w, x = tiny
    ref = oracle.qmatmul(case.wq, case.ws, case.x, 512, 512)
    for n in WIDTHS:
        y = run(w, x, n, 512, 512)
        assert rel_err_rows(host(y)[:n], ref[:n]) <= TOL


def test_width_n_equals_n_width1_calls_bitwise(tiny):
    case, w, x = tiny
    singles = torch.cat([run(w, x[j:j + 1], 1, 512, 512) for j in range(8)])
    for n in range(1, 9):
        y = run(w, x, n, 512, 512)
        assert bits_equal(y[:n], singles[:n]), f"width {n}"


@pytest.mark.parametrize("N,K", [(200, 768), (1000, 2048), (96, 5120), (130, 17408)])
def test_ragged_rows_and_ksplits_parity_and_invariance(N, K):
    case = synth.qmatmul_case(7000 + N, N, K, 5)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    y = run(w, x, 5, N, K)
    ref = oracle.qmatmul(case.wq, case.ws, case.x, N, K)
    assert rel_err_rows(host(y), ref) <= TOL
    for j in range(5):
        assert bits_equal(run(w, x[j:j + 1], 1, N, K)[0], y[j])


def test_column_placement_and_tile_width_do_not_change_bits(tiny):
    case, w, x = tiny
    L = _lib()
    probe = x[3:4]
    ref = run(w, probe, 1, 512, 512)[0]
    g = np.random.default_rng(5)
    for n_cols in (8, 16, 37, 80):
        xs = dev(synth.activations_bf16(int(g.integers(1 << 30)), n_cols, 512))
        for pos in sorted({0, n_cols // 2, n_cols - 1, min(7, n_cols - 1)}):
            xs[pos] = probe[0]
            y = run(w, xs, n_cols, 512, 512)
            assert bits_equal(y[pos], ref), (n_cols, pos)
            # 10: 80-column pass on mma.sync, 11: on tcgen05; 12 / 13: 16- / 8-column
            # passes, several column groups per launch
            for nt in (1, 2, 10, 11, 12, 13):
                yy = torch.zeros((n_cols, 512), dtype=torch.float32, device="cuda")
                wsp = workspace(debug_nt_ws(512, 512, nt))
                L.spec_qmatmul_debug_nt(w[0], w[1], 512, 512, xs, n_cols, 512, yy, 512, nt, wsp, wsp.numel() * 4)
                torch.cuda.synchronize()
                assert bits_equal(yy, y), (n_cols, nt)


def test_padding_columns_and_ldx_do_not_leak(tiny):
    case, w, x = tiny
    ldx = 640
    xp = torch.full((3, ldx), 0x7FC0, dtype=torch.int16, device="cuda")  # NaN in the padding
    xp[:, :512] = x[:3]
    y = run(w, xp, 3, 512, 512, ldx=ldx)
    assert torch.isfinite(y).all()
    assert bits_equal(y, run(w, x[:3], 3, 512, 512))


def test_bf16_output_and_accumulate(tiny):
    case, w, x = tiny
    y32 = run(w, x, 4, 512, 512)
    ybf = run(w, x, 4, 512, 512, out_dt=2)
    assert torch.equal(ybf, y32.to(torch.bfloat16))
    base = torch.randn(4, 512, device="cuda")
    acc = base.clone()
    run(w, x, 4, 512, 512, y=acc, accumulate=1)
    assert bits_equal(acc, base + y32)


def test_zero_columns_is_a_noop(tiny):
    case, w, x = tiny
    y = torch.full((1, 512), 7.0, device="cuda")
    run(w, x, 0, 512, 512, y=y)
    assert bool((y == 7.0).all())


@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408), (5120, 5120)])
def test_dense_sweep_shapes_sampled_parity_and_invariance(N, K):
    """Full-size shapes of a 27B-class decoder: parity on sampled output rows,
    bitwise width-n == n width-1 calls on every output."""
    case = synth.qmatmul_case(1002 + K % 97, N, K, 8)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    singles = torch.cat([run(w, x[j:j + 1], 1, N, K) for j in range(8)])
    for n in WIDTHS:
        y = run(w, x, n, N, K)
        assert bits_equal(y[:n], singles[:n]), f"width {n}"
    rows = np.random.default_rng(3).choice(N, 48, replace=False)
    ref = oracle.qmatmul_rows(case.wq, case.ws, case.x, K, rows)      # [8][48]
    got = host(singles)[:, rows]
    full_scale = np.abs(host(singles)).max(axis=1, keepdims=True)     # row max over all N outputs
    assert float((np.abs(got - ref) / full_scale).max()) <= TOL


def test_noninvariant_variant_matches_oracle(tiny):
    case, w, x = tiny
    L = _lib()
    ref = oracle.qmatmul(case.wq, case.ws, case.x, 512, 512)
    for seg in (0, 1, 2):
        y = torch.zeros((8, 512), dtype=torch.float32, device="cuda")
        wsp = workspace(L.spec_qmatmul_workspace(512, 512, 8))
        L.spec_qmatmul_noninvariant(w[0], w[1], 512, 512, x, 8, 512, y, 512, seg, wsp, wsp.numel() * 4)
        torch.cuda.synchronize()
        assert rel_err_rows(host(y), ref) <= TOL


def test_workspace_is_left_zeroed_and_calls_repeat_bitwise():
    L = _lib()
    case = synth.qmatmul_case(55, 1000, 2048, 80)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    need = L.spec_qmatmul_workspace(1000, 2048, 80)
    wsp = torch.zeros(need // 4 + 16, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        y = torch.zeros((80, 1000), dtype=torch.float32, device="cuda")
        L.spec_qmatmul(w[0], w[1], 1000, 2048, x, 80, 2048, y, 0, 1000, 0, wsp, wsp.numel() * 4)
        torch.cuda.synchronize()
        outs.append(y)
        # the first 64 KB, where any call's arrival counters lie, is zero again
        assert int(wsp[:16384].abs().sum().item()) == 0
    assert bits_equal(outs[0], outs[1]) and bits_equal(outs[1], outs[2])
    ref = oracle.qmatmul(case.wq, case.ws, case.x, 1000, 2048)
    assert rel_err_rows(host(outs[0]), ref) <= TOL
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul(w[0], w[1], 1000, 2048, x, 80, 2048, outs[0], 0, 1000, 0, wsp, 64)
    assert e.value.status == 3


@pytest.mark.parametrize("N,K,n", [(1, 256, 3), (129, 256, 17), (300, 1280, 81), (140, 512, 161)])
def test_edge_shapes_and_pass_boundaries(N, K, n):
    """One output row, a single 256-k segment, 17 columns (first wide pass), and
    81 / 161 columns (two and three 80-column passes): parity and width-1 bits."""
    case = synth.qmatmul_case(8800 + N + n, N, K, n)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    y = run(w, x, n, N, K)
    assert rel_err_rows(host(y), oracle.qmatmul(case.wq, case.ws, case.x, N, K)) <= TOL
    for j in sorted({0, n // 2, n - 1}):
        assert bits_equal(run(w, x[j:j + 1], 1, N, K)[0], y[j]), j


@pytest.mark.parametrize("N,K,n", [(2048, 5632, 80), (2048, 2048, 80), (3072, 2048, 48), (32000, 2048, 32),
                                   (1000, 2304, 23)])
def test_grouped_plans_parity_invariance_and_workspace(N, K, n):
    """Shapes where spec_qmatmul runs its columns as one launch of 16- or
    8-column groups: parity with the oracle on sampled columns, every sampled
    column equal to its width-1 call and to the 80-column pass bit for bit, and
    the workspace's counter area left zero."""
    L = _lib()
    plan = L.spec_qmatmul_plan(N, K, n)
    assert plan in (8, 16, 80) and plan == L.spec_qmatmul_plan(N, K, n)
    case = synth.qmatmul_case(9100 + n, N, K, n)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    need = L.spec_qmatmul_workspace(N, K, n)
    wsp = torch.zeros(need // 4 + 16, dtype=torch.int32, device="cuda")
    y = torch.zeros((n, N), dtype=torch.float32, device="cuda")
    L.spec_qmatmul(w[0], w[1], N, K, x, n, K, y, 0, N, 0, wsp, wsp.numel() * 4)
    torch.cuda.synchronize()
    assert int(wsp[:16384].abs().sum().item()) == 0
    cols = sorted({0, 7, 8, 15, 16, n // 2, n - 1} & set(range(n)))
    ref = oracle.qmatmul(case.wq, case.ws, case.x[cols], N, K)
    assert rel_err_rows(host(y)[cols], ref) <= TOL
    for j in cols[::2]:
        assert bits_equal(run(w, x[j:j + 1], 1, N, K)[0], y[j]), j
    y10 = torch.zeros((n, N), dtype=torch.float32, device="cuda")
    w10 = workspace(debug_nt_ws(N, K, 10))
    L.spec_qmatmul_debug_nt(w[0], w[1], N, K, x, n, K, y10, N, 10, w10, w10.numel() * 4)
    torch.cuda.synchronize()
    assert bits_equal(y10, y)


def test_calls_of_different_tile_counts_share_one_workspace():
    """A call with few tiles stores its partial sums where a later call with
    many tiles keeps its arrival counters; every call leaves the workspace zero,
    so the later call is unaffected (results equal those on a fresh workspace)."""
    L = _lib()
    small = synth.qmatmul_case(61, 3072, 2048, 80)
    big = synth.qmatmul_case(62, 32000, 2048, 80)
    need = max(L.spec_qmatmul_workspace(3072, 2048, 80), L.spec_qmatmul_workspace(32000, 2048, 80))
    shared = torch.zeros(need // 4 + 16, dtype=torch.int32, device="cuda")
    fresh = torch.zeros(need // 4 + 16, dtype=torch.int32, device="cuda")
    ws_, wb_, xb_ = dev(small.wq), dev(small.ws), dev(small.x)
    wq, wsc, xb = dev(big.wq), dev(big.ws), dev(big.x)
    ys = torch.zeros((80, 3072), dtype=torch.float32, device="cuda")
    yb = torch.zeros((80, 32000), dtype=torch.float32, device="cuda")
    ref = torch.zeros((80, 32000), dtype=torch.float32, device="cuda")
    L.spec_qmatmul(wq, wsc, 32000, 2048, xb, 80, 2048, ref, 0, 32000, 0, fresh, fresh.numel() * 4)
    for _ in range(4):
        L.spec_qmatmul(ws_, wb_, 3072, 2048, xb_, 80, 2048, ys, 0, 3072, 0, shared, shared.numel() * 4)
        L.spec_qmatmul(wq, wsc, 32000, 2048, xb, 80, 2048, yb, 0, 32000, 0, shared, shared.numel() * 4)
        torch.cuda.synchronize()
        assert bits_equal(yb, ref)
