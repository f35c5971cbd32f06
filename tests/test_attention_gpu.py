"""K2 + K3 (spec_flash_decode): parity with the oracle and bit-exact invariance
across verify widths, row positions and ragged batch compositions.

Test shape from ramgpt.org, "When Lossless Speculation Stops Being Lossless on
Blackwell", section "Flash Attention Changes Geometry With Batch Width" (widths
1-4 at three KV lengths, each batched row against its serial evaluation) and
"A Better Backend Test Matrix" (long-context KV lengths, widths up to 8).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import DT_BF16, DT_F16
from tests.gpu_util import TOL, bits_equal, dev, host, rel_err_rows

pytestmark = pytest.mark.gpu


class Dev:
    """An attention case uploaded once (the paged cache is shared by every call)."""

    def __init__(self, case: synth.AttentionCase):
        self.case = case
        self.q = dev(case.q)
        self.k = dev(case.k_cache)
        self.v = dev(case.v_cache)
        self.bt = dev(case.block_table)
        self.pages = case.k_cache.shape[0]

    def call(self, rows_idx=None, ctx=None, cu=None, out_dt=0, max_kv_len=None):
        """Run spec_flash_decode on the selected global rows of q (default: the case's own batch)."""
        import invariant_speculative_verification_gb300 as L
        c = self.case
        if rows_idx is None:
            q = self.q
            ctx = c.ctx_start
            cu = c.cu_rows
            seq_of = None
        else:
            q = self.q[torch.as_tensor(rows_idx, device="cuda", dtype=torch.long)].contiguous()
        S, R = len(ctx), int(cu[-1])
        max_kv_len = max_kv_len or int(max(np.asarray(ctx) + np.diff(cu)))
        ws_bytes = L.spec_flash_decode_workspace(R, c.Hq, c.D, max_kv_len)
        ws = torch.empty(ws_bytes // 4 + 64, dtype=torch.float32, device="cuda")
        out = torch.zeros((R, c.Hq, c.D), dtype=torch.float32 if out_dt == 0 else torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.spec_flash_decode(q, c.dt, c.Hq, c.Hkv, c.D, c.scale, self.k, self.v, self.pages, self._bt(rows_idx, ctx, cu),
                            self.case.block_table.shape[1], dev(np.asarray(ctx, np.int32)),
                            dev(np.asarray(cu, np.int32)), S, R, max_kv_len, out, out_dt, ws, ws_bytes, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, hex(int(err.item()))
        return out

    def _bt(self, rows_idx, ctx, cu):
        return self.bt if rows_idx is None else self._sub_bt

    def single_row(self, s, i):
        """Evaluate row i of sequence s alone at width 1 (position ctx[s] + i)."""
        c = self.case
        self._sub_bt = self.bt[s:s + 1].contiguous()
        r = int(c.cu_rows[s]) + i
        return self.call([r], [int(c.ctx_start[s]) + i], [0, 1])[0]

    def sequence_alone(self, s):
        c = self.case
        self._sub_bt = self.bt[s:s + 1].contiguous()
        r0, r1 = int(c.cu_rows[s]), int(c.cu_rows[s + 1])
        return self.call(list(range(r0, r1)), [int(c.ctx_start[s])], [0, r1 - r0])


def test_tiny_config_parity_and_invariance():
    # 4 query heads, 2 KV heads, head_dim 64, KV length 256, fp16; widths 1..8
    for n in range(1, 9):
        case = synth.attention_case(1001 + n, rows=[n, n], ctx=[256 - n, 256 - n], Hq=4, Hkv=2, D=64, dt=DT_F16,
                                    scale=1 / math.sqrt(64))
        d = Dev(case)
        out = d.call()
        ref = oracle.attention(case)
        assert rel_err_rows(host(out), ref) <= TOL, n
        for s in range(2):
            for i in range(n):
                assert bits_equal(d.single_row(s, i), out[int(case.cu_rows[s]) + i]), (n, s, i)


@pytest.mark.parametrize("L", [1024, 4096, 16384])
def test_long_context_gqa_parity_and_width_invariance(L):
    # 40 query heads, 8 KV heads, head_dim 128, bf16, Q ~ N(0,1)/sqrt(128) (scale folded in: 1.0)
    for n in (1, 2, 3, 4, 5, 8):
        case = synth.attention_case(1003 + L + n, rows=[n], ctx=[L - n], Hq=40, Hkv=8, D=128, dt=DT_BF16,
                                    q_std=1 / math.sqrt(128), scale=1.0)
        d = Dev(case)
        out = d.call()
        for i in range(n):
            assert bits_equal(d.single_row(0, i), out[i]), (L, n, i)
        # oracle on every (row, head) pair at the shortest length; at the longer ones on
        # the block's first and last rows with all 40 heads, plus sampled pairs
        want = np.zeros((n, 40), np.uint8)
        if L == 1024:
            want[:] = 1
        else:
            want[0, :] = want[n - 1, :] = 1
            g = np.random.default_rng(L + n)
            want[g.integers(0, n, 6), g.integers(0, 40, 6)] = 1
        ref = oracle.attention(case, want=want)
        got = host(out)
        rr, hh = np.nonzero(want)
        assert rel_err_rows(got[rr, hh], ref[rr, hh]) <= TOL


def test_ragged_batch_composition_is_bit_invariant():
    g = np.random.default_rng(17)
    rows = [1, 5, 8, 2, 3, 7, 1, 4]
    ctx = list(g.integers(0, 900, len(rows)))
    ctx[0] = 0            # a sequence whose first row is position 0
    ctx[3] = 255          # block straddles a chunk boundary
    case = synth.attention_case(4242, rows=rows, ctx=ctx, Hq=16, Hkv=4, D=128, dt=DT_BF16,
                                scale=1 / math.sqrt(128))
    d = Dev(case)
    out = d.call()
    ref = oracle.attention(case)
    assert rel_err_rows(host(out), ref) <= TOL
    for s in range(len(rows)):
        alone = d.sequence_alone(s)
        r0 = int(case.cu_rows[s])
        assert bits_equal(alone, out[r0:r0 + rows[s]]), s
        for i in range(rows[s]):
            assert bits_equal(d.single_row(s, i), out[r0 + i]), (s, i)
    # a shuffled order of the same sequences gives the same rows
    perm = g.permutation(len(rows))
    rows_idx = np.concatenate([np.arange(case.cu_rows[s], case.cu_rows[s + 1]) for s in perm])
    d._sub_bt = d.bt[torch.as_tensor(perm, device="cuda", dtype=torch.long)].contiguous()
    cu = np.concatenate([[0], np.cumsum(np.asarray(rows)[perm])]).astype(np.int32)
    shuf = d.call(list(rows_idx), list(np.asarray(ctx)[perm]), cu)
    assert bits_equal(shuf, out[torch.as_tensor(rows_idx, device="cuda", dtype=torch.long)])


def test_bf16_output_and_larger_bound_do_not_change_values():
    case = synth.attention_case(77, rows=[4, 2], ctx=[300, 17], Hq=8, Hkv=2, D=128, dt=DT_BF16)
    d = Dev(case)
    out = d.call()
    assert torch.equal(d.call(out_dt=2), out.to(torch.bfloat16))
    assert bits_equal(d.call(max_kv_len=5000), out)


def test_split_chunks_of_short_and_whole_chunks_of_long_sequences():
    # Five rows per sequence (more than one M-tile on average): the chunks of
    # sequences of at most 8 chunks are halved over two items, the 10-chunk
    # one keeps whole chunks; a decoder-sized key bound (21 chunks, an odd
    # grid of mostly empty items) gives the same bits as the tight one.
    rows = [5] * 15 + [8]
    ctx = [127, 300, 511, 1023, 0, 2040, 60, 700, 1500, 200, 900, 1200, 30, 400, 800, 2300]
    case = synth.attention_case(5150, rows=rows, ctx=ctx, Hq=16, Hkv=4, D=128, dt=DT_BF16,
                                scale=1 / math.sqrt(128))
    d = Dev(case)
    out = d.call()
    assert rel_err_rows(host(out), oracle.attention(case)) <= TOL
    assert bits_equal(d.call(max_kv_len=5277), out)
    for s in (0, 4, 5, 15):
        r0 = int(case.cu_rows[s])
        assert bits_equal(d.sequence_alone(s), out[r0:r0 + rows[s]]), s
        assert bits_equal(d.single_row(s, rows[s] - 1), out[r0 + rows[s] - 1]), s


def test_prefill_block_many_rows():
    # 128-row block at position 0 (several M-tile rounds per CTA)
    case = synth.attention_case(91, rows=[128], ctx=[0], Hq=4, Hkv=1, D=64, dt=DT_BF16)
    d = Dev(case)
    out = d.call()
    assert rel_err_rows(host(out), oracle.attention(case)) <= TOL
    for i in (0, 1, 63, 64, 127):
        assert bits_equal(d.single_row(0, i), out[i])


def test_bad_block_table_is_reported_not_faulted():
    import invariant_speculative_verification_gb300 as L
    case = synth.attention_case(5, rows=[2], ctx=[40], Hq=4, Hkv=2, D=64, dt=DT_F16)
    bt = case.block_table.copy()
    bt[0, 1] = 10 ** 6
    case.block_table = bt
    d = Dev(case)
    ws_bytes = L.spec_flash_decode_workspace(2, 4, 64, 42)
    ws = torch.empty(ws_bytes // 4 + 64, dtype=torch.float32, device="cuda")
    out = torch.zeros((2, 4, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_flash_decode(d.q, case.dt, 4, 2, 64, case.scale, d.k, d.v, d.pages, d.bt, bt.shape[1],
                        dev(case.ctx_start), dev(case.cu_rows), 1, 2, 42, out, 0, ws, ws_bytes, err)
    torch.cuda.synchronize()
    assert int(err.item()) & L.DEVERR["BLOCK_TABLE"]
    with pytest.raises(L.SpecError):
        L.spec_flash_decode(d.q, case.dt, 4, 2, 64, case.scale, d.k, d.v, d.pages, d.bt, bt.shape[1],
                            dev(case.ctx_start), dev(case.cu_rows), 1, 2, 42, out, 0, ws, 16, err)


def test_rows_of_a_sequence_longer_than_the_bound_are_zeros():
    # Sequence 1 ends past max_kv_len (positions 198..201 against a bound of
    # 200) although its first rows lie inside it: the partial kernel rejects
    # the whole sequence and reports it, and the combine writes zeros for all
    # of its rows instead of reading partials that were never written (the
    # workspace starts as NaN).  Sequence 0 is unaffected.
    import invariant_speculative_verification_gb300 as L
    case = synth.attention_case(6, rows=[3, 4], ctx=[100, 198], Hq=8, Hkv=2, D=128, dt=DT_BF16)
    d = Dev(case)
    R, bound = 7, 200
    ws_bytes = L.spec_flash_decode_workspace(R, 8, 128, bound)
    ws = torch.full((ws_bytes // 4 + 64,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full((R, 8, 128), 7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.spec_flash_decode(d.q, case.dt, 8, 2, 128, case.scale, d.k, d.v, d.pages, d.bt, case.block_table.shape[1],
                        dev(case.ctx_start), dev(case.cu_rows), 2, R, bound, out, 0, ws, ws_bytes, err)
    torch.cuda.synchronize()
    assert int(err.item()) & L.DEVERR["LENGTH"]
    assert torch.count_nonzero(out[3:]).item() == 0
    assert bits_equal(out[:3], d.sequence_alone(0))


@pytest.mark.parametrize("D", [64, 128])
def test_rows_across_subtile_and_chunk_edges(D):
    """Verify blocks whose rows cross the 64-key sub-tile and 256-key chunk edges:
    every row equals its width-1 evaluation and the oracle."""
    for ctx, n in ((60, 8), (125, 6), (190, 5), (250, 8), (511, 3), (0, 1), (63, 1), (64, 1)):
        case = synth.attention_case(5100 + ctx + D, rows=[n], ctx=[ctx], Hq=8, Hkv=2, D=D, dt=DT_BF16,
                                    scale=1 / math.sqrt(D))
        d = Dev(case)
        out = d.call()
        assert rel_err_rows(host(out), oracle.attention(case)) <= TOL, (ctx, n)
        for i in range(n):
            assert bits_equal(d.single_row(0, i), out[i]), (ctx, n, i)


def test_empty_sequences_in_a_batch():
    """Sequences with no rows contribute nothing and change no other row."""
    rows = [3, 0, 2, 0]
    ctx = [100, 40, 300, 7]
    case = synth.attention_case(6100, rows=rows, ctx=ctx, Hq=8, Hkv=2, D=128, dt=DT_BF16, scale=1 / math.sqrt(128))
    d = Dev(case)
    out = d.call()
    assert rel_err_rows(host(out), oracle.attention(case)) <= TOL
    for s, n in enumerate(rows):
        for i in range(n):
            assert bits_equal(d.single_row(s, i), out[int(case.cu_rows[s]) + i]), (s, i)
