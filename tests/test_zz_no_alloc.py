"""spec_qmatmul_static_scratch: the int4 matmul with library-owned scratch.

The call must give the same results as spec_qmatmul (which takes a
caller-supplied workspace) on two calls in a row, and must refuse shapes whose
scratch would not fit its fixed size.  Kept in its own module, collected last,
so it runs both in a fresh process and after every other GPU test.
"""
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, bits_equal, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu


def _reference(L, w, x, N, K, n, y_dt):
    need = L.spec_qmatmul_workspace(N, K, n)
    wsp = torch.zeros(need // 4 + 16, dtype=torch.int32, device="cuda")
    y = torch.zeros((n, N), dtype=torch.float32 if y_dt == L.SPEC_F32 else torch.bfloat16, device="cuda")
    L.spec_qmatmul(w[0], w[1], N, K, x, n, K, y, y_dt, N, 0, wsp, wsp.numel() * 4)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("N,K,n", [(512, 512, 5), (1000, 2048, 8), (17408, 5120, 8), (200, 768, 40)])
def test_static_scratch_matches_workspace_call_twice(N, K, n):
    import invariant_speculative_verification_gb300 as L
    case = synth.qmatmul_case(4100 + N, N, K, n)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    ref = _reference(L, w, x, N, K, n, L.SPEC_F32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        y = torch.full((n, N), float("nan"), dtype=torch.float32, device="cuda")
        L.spec_qmatmul_static_scratch(w[0], w[1], N, K, x, n, K, y, L.SPEC_F32, N, 0, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert bits_equal(y, ref)
        if N * K <= 2048 * 2048:
            assert rel_err_rows(host(y), oracle.qmatmul(case.wq, case.ws, case.x, N, K)) <= TOL
        else:
            assert rel_err_rows(host(y), host(ref)) <= TOL


def test_static_scratch_bf16_output_and_width1_invariance():
    import invariant_speculative_verification_gb300 as L
    N, K = 1000, 2048
    case = synth.qmatmul_case(4200, N, K, 4)
    w, x = (dev(case.wq), dev(case.ws)), dev(case.x)
    ref = _reference(L, w, x, N, K, 4, L.SPEC_BF16)
    y = torch.zeros((4, N), dtype=torch.bfloat16, device="cuda")
    L.spec_qmatmul_static_scratch(w[0], w[1], N, K, x, 4, K, y, L.SPEC_BF16, N, 0)
    y1 = torch.zeros((1, N), dtype=torch.bfloat16, device="cuda")
    L.spec_qmatmul_static_scratch(w[0], w[1], N, K, x[2:3], 1, K, y1, L.SPEC_BF16, N, 0)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert torch.equal(y1[0], y[2])


def test_static_scratch_rejects_shapes_beyond_its_size():
    import invariant_speculative_verification_gb300 as L
    N, K = 17408, 5120   # fits at 8 columns, not at 80
    wq = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((N, K // 32), dtype=torch.int16, device="cuda")
    x = torch.zeros((80, K), dtype=torch.int16, device="cuda")
    y = torch.full((80, N), 3.0, dtype=torch.float32, device="cuda")
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul_static_scratch(wq, ws, N, K, x, 80, K, y, L.SPEC_F32, N, 0)
    assert e.value.status == 3
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
