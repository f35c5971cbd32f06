"""Run spec_flash_decode on one synthetic case a few times (for profiler captures).

    python -m invariant_speculative_verification_gb300.attn_once L n [calls]

One sequence, 40 query heads and 8 KV heads of 128 (bf16), a paged cache of
L keys (seeded N(0, 1) K and V, random page order), n query rows at positions
L - n .. L - 1 (Q ~ N(0, 1) / sqrt(128), scale folded into Q).  The output is
checked for finiteness only.  A profiler can select attn_partial_kernel or
attn_combine_kernel by name and capture one or a few launches.
"""
from __future__ import annotations

import math
import sys

import numpy as np
import torch

import synth

from . import _lib as L


def main(argv):
    Lk, n = int(argv[1]), int(argv[2])
    calls = int(argv[3]) if len(argv) > 3 else 3
    Hq, Hkv, D = 40, 8, 128
    c = synth.attention_case(1003 + Lk + 10 * n, rows=[n], ctx=[Lk - n], Hq=Hq, Hkv=Hkv, D=D, dt=synth.DT_BF16,
                             q_std=1 / math.sqrt(D), scale=1.0, poison=False)

    def up(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    q, kc, vc, bt = up(c.q), up(c.k_cache), up(c.v_cache), up(c.block_table)
    wsb = L.spec_flash_decode_workspace(n, Hq, D, Lk)
    ws = torch.empty(wsb // 4 + 64, dtype=torch.float32, device="cuda")
    out = torch.zeros((n, Hq, D), dtype=torch.float32, device="cuda")
    ctx = torch.tensor([Lk - n], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(calls):
        L.spec_flash_decode(q, L.SPEC_BF16, Hq, Hkv, D, 1.0, kc, vc, c.k_cache.shape[0], bt, c.block_table.shape[1],
                            ctx, cu, 1, n, Lk, out, L.SPEC_F32, ws, wsb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and bool(torch.isfinite(out).all())
    print(f"attn_once: L={Lk}, {n} rows, {calls} calls: ok")


if __name__ == "__main__":
    L.load()
    main(sys.argv)
