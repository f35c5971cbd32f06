"""K4 (spec_verify_greedy) and K5 (spec_kv_compact): integer outputs must equal
the oracle exactly.

proofoftech.org, "'Lossless' speculative decoding isn't free", opening section
(accept the agreed prefix, correct the first disagreement) and section
"Batching breaks the implementation" (ragged acceptance, realignment).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import DT_BF16, DT_F32
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def gpu_verify(case, logits=None, drafts=None):
    import invariant_speculative_verification_gb300 as L
    S, R, V = case.S, case.R, case.V
    lg = dev(case.logits if logits is None else logits)
    dr = dev(case.drafts if drafts is None else drafts) if R > S else None
    ws_bytes = L.spec_verify_greedy_workspace(R, V)
    ws = torch.empty(ws_bytes // 8 + 2, dtype=torch.int64, device="cuda")
    am = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    acc, cor, cn = (torch.full((S,), -1, dtype=torch.int32, device="cuda") for _ in range(3))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_verify_greedy(lg, 0 if case.dt == DT_F32 else 2, V, dev(case.cu_rows), S, R, dr, dev(case.ctx_start), am,
                         acc, cor, cn, ws, ws_bytes, err)
    torch.cuda.synchronize()
    return dict(argmax=host(am), accepted=host(acc), correction=host(cor), ctx_new=host(cn), err=int(err.item()))


def check_exact(case, **kw):
    got = gpu_verify(case, **kw)
    ref = oracle.verify_greedy(kw.get("logits", case.logits), case.dt, case.V, case.cu_rows,
                               kw.get("drafts", case.drafts), case.ctx_start)
    for k in ("argmax", "accepted", "correction", "ctx_new"):
        assert np.array_equal(got[k], ref[k]), k
    return got, ref


def test_tiny_fp32_with_near_ties():
    case = synth.verify_case(1001, [4, 4], 1000, DT_F32, sigma=1.0, tie_frac=0.1)
    got, _ = check_exact(case)
    assert got["err"] == 0
    assert np.array_equal(got["argmax"], case.planted_top)


def test_ragged_bf16_large_vocab():
    g = np.random.default_rng(1004)
    L = g.integers(1, 8, size=64)
    case = synth.verify_case(1004, L, 152064, DT_BF16, sigma=2.0, tie_frac=0.01)
    got, _ = check_exact(case)
    assert got["err"] == 0
    assert np.array_equal(got["argmax"], case.planted_top)


@pytest.mark.parametrize("R_seqs", [64, 8])
def test_ragged_bf16_natural_rows_and_lower_index_ties(R_seqs):
    """Rows whose maximum comes from the raw N(0, 2) bf16 draws, 5 % of them with a
    planted competitor: exact ties at a lower index (within a scan split and across
    every candidate split boundary), one-ulp-lower values at a lower index, and ties
    at a higher index.  The drafts copy the oracle's argmax with probability 0.7.
    tokenstrom.com, "'Lossless,' but not quite", section "Why the math checks out and
    the text still flips": near ties decide the token, so the tie rule must hold."""
    V = 152064
    g = np.random.default_rng(1044 + R_seqs)
    L = g.integers(1, 8, size=R_seqs)
    nvec = V // 8
    edges = sorted({8 * (nvec * k // sp) for sp in range(2, 9) for k in range(1, sp)})
    case = synth.verify_case_natural(1044 + R_seqs, L, V, sigma=2.0, tie_frac=0.05, edges=edges)
    # drafts from the oracle's own argmax (probability 0.7), else uniform
    am = oracle.verify_greedy(case.logits, case.dt, V, case.cu_rows, case.drafts, case.ctx_start)["argmax"]
    drafts = case.drafts.copy()
    for s in range(case.S):
        for i in range(int(L[s])):
            if g.random() < 0.7:
                drafts[case.cu_rows[s] - s + i] = am[case.cu_rows[s] + i]
    got, ref = check_exact(case, drafts=drafts)
    assert got["err"] == 0
    assert ref["accepted"].sum() > 0
    # the planted lower-index ties really decide some rows
    tie_rows = np.nonzero(case.tie_rows)[0]
    assert len(tie_rows) > 0
    lower = 0
    for r in tie_rows:
        row = synth.bf16_bits_to_f32(case.logits[r])
        lower += int(np.sum(row == row[am[r]]) > 1 and am[r] == np.flatnonzero(row == row.max())[0])
    assert lower > 0


def test_width1_rows_and_all_or_nothing_acceptance():
    case = synth.verify_case(33, [0, 3, 0, 7, 1], 4096, DT_BF16, sigma=2.0, tie_frac=0.3)
    check_exact(case)
    good = np.concatenate([case.planted_top[case.cu_rows[s]:case.cu_rows[s + 1] - 1] for s in range(case.S)])
    got, _ = check_exact(case, drafts=good)
    assert np.array_equal(got["accepted"], np.diff(case.cu_rows) - 1)


def test_nan_and_out_of_range_drafts_are_flagged():
    import invariant_speculative_verification_gb300 as Lb
    case = synth.verify_case(8, [2, 2], 1024, DT_F32)
    lg = case.logits.copy()
    lg[1, 5] = np.nan
    dr = case.drafts.copy()
    dr[0] = 5000
    got = gpu_verify(case, logits=lg, drafts=dr)
    ref = oracle.verify_greedy(lg, DT_F32, case.V, case.cu_rows, dr, case.ctx_start)
    assert np.array_equal(got["argmax"], ref["argmax"]) and np.array_equal(got["accepted"], ref["accepted"])
    assert got["err"] & Lb.DEVERR["NAN"] and got["err"] & Lb.DEVERR["TOKEN_RANGE"]


def gpu_compact(case, staged=True, accepted=None):
    import invariant_speculative_verification_gb300 as L
    acc = case.accepted if accepted is None else accepted
    kc, vc = dev(case.k_cache), dev(case.v_cache)
    cuk = torch.full((case.S + 1,), -1, dtype=torch.int32, device="cuda")
    src = torch.full((case.R,), -1, dtype=torch.int32, device="cuda")
    dst = torch.full((case.R,), -1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_kv_compact(dev(case.k_stage) if staged else None, dev(case.v_stage) if staged else None, kc, vc,
                      case.Hkv, case.D, case.k_cache.shape[0], dev(case.block_table), case.block_table.shape[1],
                      dev(case.ctx_start), dev(acc), dev(case.cu_rows), case.S, case.R, cuk, src, dst, err)
    torch.cuda.synchronize()
    return host(kc, np.uint16), host(vc, np.uint16), host(cuk), host(src), host(dst), int(err.item())


@pytest.mark.parametrize("staged", [True, False])
def test_kv_compaction_matches_oracle_exactly(staged):
    g = np.random.default_rng(1004)
    L = g.integers(1, 8, size=64)
    case = synth.compact_case(1004, L, Hkv=32, D=128, ctx_range=(256, 8192))
    kc, vc, cuk, src, dst, err = gpu_compact(case, staged)
    rk, rv, rcuk, rsrc, rdst = oracle.kv_compact(case.k_stage if staged else None, case.v_stage if staged else None,
                                                 case.k_cache, case.v_cache, 32, 128, case.block_table,
                                                 case.ctx_start, case.accepted, case.cu_rows)
    n = int(rcuk[-1])
    assert err == 0
    assert np.array_equal(cuk, rcuk)
    assert np.array_equal(src[:n], rsrc) and np.array_equal(dst[:n], rdst)
    assert np.array_equal(kc, rk) and np.array_equal(vc, rv)


def test_verify_then_compact_pipeline_on_device():
    """The realign pair: accepted counts produced by verify drive compaction."""
    import invariant_speculative_verification_gb300 as L
    g = np.random.default_rng(5)
    lens = g.integers(1, 8, size=16)
    vc_case = synth.verify_case(5, lens, 2048, DT_BF16, sigma=2.0)
    got = gpu_verify(vc_case)
    cc = synth.compact_case(6, lens, Hkv=4, D=64, ctx_range=(16, 300), accepted=got["accepted"])
    kc, vcache, cuk, src, dst, err = gpu_compact(cc)
    rk, rv, rcuk, rsrc, rdst = oracle.kv_compact(cc.k_stage, cc.v_stage, cc.k_cache, cc.v_cache, 4, 64,
                                                 cc.block_table, cc.ctx_start, got["accepted"], cc.cu_rows)
    assert err == 0 and np.array_equal(kc, rk) and np.array_equal(cuk, rcuk)
