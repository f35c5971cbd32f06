"""The bounded-wait error path, run on the GPU in the allowed form: a wait on an
mbarrier phase that can never complete (16 transaction bytes expected, no copy
issued, nothing in flight) runs out after a short poll limit; the kernel
reports SPEC_DEVERR_TIMEOUT through the device error word and returns, and
the next call on the same stream computes correctly."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import TOL, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_the_stream_stays_usable():
    import invariant_speculative_verification_gb300 as L
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_debug_wait_timeout(1000, err)
    torch.cuda.synchronize()
    assert int(err.item()) & L.DEVERR["TIMEOUT"]
    # a normal call right after it, on the same stream, is correct and reports nothing
    N, K, n = 512, 512, 5
    qc = synth.qmatmul_case(91, N, K, n)
    y = torch.zeros((n, N), dtype=torch.float32, device="cuda")
    wsb = L.spec_qmatmul_workspace(N, K, n)
    ws = torch.zeros(wsb // 4 + 16, dtype=torch.int32, device="cuda")
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_debug_wait_timeout(10, err)
    L.spec_qmatmul(dev(qc.wq), dev(qc.ws), N, K, dev(qc.x), n, K, y, L.SPEC_F32, N, 0, ws, wsb, err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    assert rel_err_rows(host(y), oracle.qmatmul(qc.wq, qc.ws, qc.x, N, K)) <= TOL


def test_wait_timeout_hook_checks_its_arguments():
    import invariant_speculative_verification_gb300 as L
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(L.SpecError):
        L.spec_debug_wait_timeout(0, err)
    with pytest.raises(L.SpecError):
        L.spec_debug_wait_timeout(1000, None)
    assert np.all(host(err) == 0)
