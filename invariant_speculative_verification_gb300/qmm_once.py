"""Run spec_qmatmul on one synthetic shape a few times (for profiler captures).

    python -m invariant_speculative_verification_gb300.qmm_once N K n_cols [calls] [nt]

Weights are seeded int4 block-32 (N(0, 0.02) quantised), activations seeded
bf16 N(0, 1); the output is checked for finiteness only.  A profiler can then
select the kernel by name (qmm_kernel for passes of up to 16 columns,
qmm_tc_kernel for the 80-column pass) and capture one or a few launches.
With `nt`, every call forces that pass width (spec_qmatmul_debug_nt: 1, 2 or
10 column tiles per pass on the mma.sync kernel, 11 for the tcgen05 kernel).
"""
from __future__ import annotations

import sys

import numpy as np
import torch

from . import _lib as L


def main(argv):
    N, K, n = int(argv[1]), int(argv[2]), int(argv[3])
    calls = int(argv[4]) if len(argv) > 4 else 3
    nt = int(argv[5]) if len(argv) > 5 else 0
    g = np.random.default_rng(11)
    codes = g.integers(0, 16, size=(N, K), dtype=np.uint8)
    wq = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)).cuda()
    ws = torch.from_numpy((np.abs(g.normal(0, 0.003, (N, K // 32))) + 1e-4).astype(np.float16).view(np.int16)).cuda()
    x = torch.from_numpy((g.normal(0, 1, (n, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.int16)).cuda()
    y = torch.zeros((n, N), dtype=torch.float32, device="cuda")
    wsb = L.spec_qmatmul_workspace(N, K, n)
    wsp = torch.zeros(wsb // 4 + 64, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(calls):
        if nt:
            L.spec_qmatmul_debug_nt(wq, ws, N, K, x, n, K, y, N, nt, wsp, wsb)
        else:
            L.spec_qmatmul(wq, ws, N, K, x, n, K, y, L.SPEC_F32, N, 0, wsp, wsb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and bool(torch.isfinite(y).all())
    print(f"qmm_once: {N}x{K}, {n} columns, {calls} calls: ok")


if __name__ == "__main__":
    L.load()
    main(sys.argv)
