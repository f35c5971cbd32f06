"""ctypes binding of libspec.so: argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors (device memory) and plain ints, passes their data pointers and the
current CUDA stream, and raises ``SpecError`` on any status other than SPEC_OK.
There is no fallback: if the library is missing or fails to load, the import
of this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SPEC_F32, SPEC_F16, SPEC_BF16 = 0, 1, 2
DEVERR = {"TOKEN_RANGE": 0x1, "NAN": 0x2, "BLOCK_TABLE": 0x4, "LENGTH": 0x8, "TIMEOUT": 0x10, "LAYOUT": 0x20}


class SpecError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {_status_name(status)}: {msg}")
        self.status = status


_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes)
_SIGS = {
    "spec_status_string": (ctypes.c_char_p, [_i32]),
    "spec_last_error": (ctypes.c_char_p, []),
    "spec_qmatmul_workspace": (_sz, [_i32, _i32, _i32]),
    "spec_qmatmul": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "spec_qmatmul_sb": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "spec_qmatmul_noninvariant": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _sz, _vp]),
    "spec_qmatmul_debug_nt": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _sz, _vp]),
    "spec_qmatmul_static_scratch": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _i32, _vp, _vp]),
    "spec_flash_decode_workspace": (_sz, [_i32, _i32, _i32, _i32]),
    "spec_flash_decode": (_i32, [_vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32,
                                 _i32, _vp, _i32, _vp, _sz, _vp, _vp]),
    "spec_verify_greedy_workspace": (_sz, [_i32, _i32]),
    "spec_verify_greedy": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "spec_verify_sample": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _f32, ctypes.c_uint64, _vp, _vp,
                                  _vp, _vp, _vp, _sz, _vp, _vp]),
    "spec_kv_compact": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp,
                               _vp, _vp, _vp]),
    "spec_embed": (_i32, [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp]),
    "spec_add_rmsnorm": (_i32, [_vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp]),
    "spec_rope_table": (_i32, [_vp, _i32, _i32, _f32, _vp]),
    "spec_rope_append": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp,
                                _i32, _vp, _vp, _vp, _vp]),
    "spec_swiglu": (_i32, [_vp, _i32, _i32, _vp, _vp]),
    "spec_add_rmsnorm_packed": (_i32, [_vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp]),
    "spec_swiglu_packed": (_i32, [_vp, _i32, _i32, _vp, _vp, _vp]),
    "spec_packed_activation_bytes": (_sz, [_i32]),
    "spec_qmatmul_plan": (_i32, [_i32, _i32, _i32, _i32]),
    "spec_qmatmul_swiglu": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _sz, _vp, _vp]),
    "spec_flash_decode_packed": (_i32, [_vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _i32, _vp, _i32, _vp, _vp, _i32,
                                        _i32, _i32, _vp, _vp, _sz, _vp, _vp, _vp]),
    "spec_qmatmul_packed": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "spec_cast_bf16": (_i32, [_vp, _sz, _vp, _vp]),
    "spec_ngram_draft": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "spec_commit_accepted": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp]),
    "spec_debug_wait_timeout": (_i32, [ctypes.c_uint32, _vp, _vp]),
    "spec_qmatmul_devcols": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _i32, _i32, _i32, _vp, _i32, _vp, _sz,
                                    _vp, _vp]),
    "spec_margin_gate_workspace": (_sz, [_i32, _i32]),
    "spec_margin_gate": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _sz, _vp,
                                _vp]),
    "spec_gate_scatter": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _vp]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libspec.so (building it first when it is absent or older than its sources)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if _build.is_stale():
        if not build_if_missing:
            raise ImportError(f"libspec.so is not built or is out of date ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _status_name(st: int) -> str:
    try:
        return load().spec_status_string(st).decode()
    except Exception:
        return str(st)


def _check(fn: str, st: int):
    if st != 0:
        raise SpecError(fn, st, load().spec_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if torch.cuda.is_available():
        return torch.cuda.current_stream().cuda_stream
    return None


def _dt(t: torch.Tensor) -> int:
    return {torch.float32: SPEC_F32, torch.float16: SPEC_F16, torch.bfloat16: SPEC_BF16,
            torch.int16: SPEC_BF16, torch.uint16: SPEC_BF16}[t.dtype]


# ---------------------------------------------------------------------------
# wrappers (names follow the C ABI)
# ---------------------------------------------------------------------------
def spec_qmatmul_workspace(N, K, n_cols) -> int:
    return int(load().spec_qmatmul_workspace(N, K, n_cols))


def spec_qmatmul(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, workspace, ws_bytes, dev_err=None,
                 stream=None):
    _check("spec_qmatmul", load().spec_qmatmul(_ptr(wq), _ptr(ws), N, K, _ptr(x), n_cols, ldx, _ptr(y), y_dt, ldy,
                                               int(accumulate), _ptr(workspace), int(ws_bytes), _ptr(dev_err),
                                               _stream(stream)))


def spec_qmatmul_devcols(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, dev_cols, min_cols, workspace,
                         ws_bytes, dev_err=None, stream=None):
    _check("spec_qmatmul_devcols", load().spec_qmatmul_devcols(
        _ptr(wq), _ptr(ws), N, K, _ptr(x), n_cols, ldx, _ptr(y), y_dt, ldy, int(accumulate), _ptr(dev_cols),
        int(min_cols), _ptr(workspace), int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_margin_gate_workspace(R, V) -> int:
    return int(load().spec_margin_gate_workspace(R, V))


def spec_margin_gate(logits, V, R, x, H, ldx, err_coef, top, rows, count, overflow, capacity, x_gathered, workspace,
                     ws_bytes, dev_err=None, stream=None):
    _check("spec_margin_gate", load().spec_margin_gate(
        _ptr(logits), V, R, _ptr(x), H, ldx, float(err_coef), _ptr(top), _ptr(rows), _ptr(count), _ptr(overflow),
        int(capacity), _ptr(x_gathered), _ptr(workspace), int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_gate_scatter(y_gathered, V, rows, count, capacity, logits, stream=None):
    _check("spec_gate_scatter", load().spec_gate_scatter(_ptr(y_gathered), V, _ptr(rows), _ptr(count), int(capacity),
                                                         _ptr(logits), _stream(stream)))


def spec_qmatmul_sb(wq, sbr, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, workspace, ws_bytes, dev_err=None,
                    stream=None):
    _check("spec_qmatmul_sb", load().spec_qmatmul_sb(_ptr(wq), _ptr(sbr), N, K, _ptr(x), n_cols, ldx, _ptr(y), y_dt,
                                                     ldy, int(accumulate), _ptr(workspace), int(ws_bytes),
                                                     _ptr(dev_err), _stream(stream)))


def spec_qmatmul_noninvariant(wq, ws, N, K, x, n_cols, ldx, y, ldy, seg_stages, workspace, ws_bytes, stream=None):
    _check("spec_qmatmul_noninvariant", load().spec_qmatmul_noninvariant(
        _ptr(wq), _ptr(ws), N, K, _ptr(x), n_cols, ldx, _ptr(y), ldy, int(seg_stages), _ptr(workspace),
        int(ws_bytes), _stream(stream)))


def spec_qmatmul_static_scratch(wq, ws, N, K, x, n_cols, ldx, y, y_dt, ldy, accumulate, dev_err=None, stream=None):
    _check("spec_qmatmul_static_scratch",
           load().spec_qmatmul_static_scratch(_ptr(wq), _ptr(ws), N, K, _ptr(x), n_cols, ldx, _ptr(y), y_dt, ldy,
                                              int(accumulate), _ptr(dev_err), _stream(stream)))


def spec_qmatmul_debug_nt(wq, ws, N, K, x, n_cols, ldx, y, ldy, nt, workspace, ws_bytes, stream=None):
    _check("spec_qmatmul_debug_nt", load().spec_qmatmul_debug_nt(_ptr(wq), _ptr(ws), N, K, _ptr(x), n_cols, ldx,
                                                                 _ptr(y), ldy, nt, _ptr(workspace), int(ws_bytes),
                                                                 _stream(stream)))


def spec_debug_wait_timeout(polls, dev_err, stream=None):
    _check("spec_debug_wait_timeout", load().spec_debug_wait_timeout(int(polls), _ptr(dev_err), _stream(stream)))


def spec_flash_decode_workspace(R, Hq, D, max_kv_len) -> int:
    return int(load().spec_flash_decode_workspace(R, Hq, D, max_kv_len))


def spec_flash_decode(q, qkv_dt, Hq, Hkv, D, scale, k_cache, v_cache, num_pages, block_table, max_blocks, ctx_start,
                      cu_rows, S, R, max_kv_len, out, out_dt, workspace, ws_bytes, dev_err=None, stream=None):
    _check("spec_flash_decode", load().spec_flash_decode(
        _ptr(q), qkv_dt, Hq, Hkv, D, float(scale), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(block_table),
        max_blocks, _ptr(ctx_start), _ptr(cu_rows), S, R, max_kv_len, _ptr(out), out_dt, _ptr(workspace),
        int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_verify_greedy_workspace(R, V) -> int:
    return int(load().spec_verify_greedy_workspace(R, V))


def spec_verify_greedy(logits, dt, V, cu_rows, S, R, drafts, ctx_start, argmax_out, accepted, correction, ctx_new,
                       workspace, ws_bytes, dev_err=None, stream=None):
    _check("spec_verify_greedy", load().spec_verify_greedy(
        _ptr(logits), dt, V, _ptr(cu_rows), S, R, _ptr(drafts), _ptr(ctx_start), _ptr(argmax_out), _ptr(accepted),
        _ptr(correction), _ptr(ctx_new), _ptr(workspace), int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_verify_sample(logits, dt, V, cu_rows, S, R, drafts, ctx_start, seq_id, inv_temperature, seed, token_out,
                       accepted, correction, ctx_new, workspace, ws_bytes, dev_err=None, stream=None):
    _check("spec_verify_sample", load().spec_verify_sample(
        _ptr(logits), dt, V, _ptr(cu_rows), S, R, _ptr(drafts), _ptr(ctx_start), _ptr(seq_id), float(inv_temperature),
        int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(token_out), _ptr(accepted), _ptr(correction), _ptr(ctx_new),
        _ptr(workspace), int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_kv_compact(k_stage, v_stage, k_cache, v_cache, Hkv, D, num_pages, block_table, max_blocks, ctx_start,
                    accepted, cu_rows, S, R, cu_kept, kept_src, dst_slot, dev_err=None, stream=None):
    _check("spec_kv_compact", load().spec_kv_compact(
        _ptr(k_stage), _ptr(v_stage), _ptr(k_cache), _ptr(v_cache), Hkv, D, num_pages, _ptr(block_table), max_blocks,
        _ptr(ctx_start), _ptr(accepted), _ptr(cu_rows), S, R, _ptr(cu_kept), _ptr(kept_src), _ptr(dst_slot),
        _ptr(dev_err), _stream(stream)))


def spec_embed(emb, V, H, tokens, R, h, dev_err=None, stream=None):
    _check("spec_embed", load().spec_embed(_ptr(emb), V, H, _ptr(tokens), R, _ptr(h), _ptr(dev_err), _stream(stream)))


def spec_add_rmsnorm(h, delta, w, R, H, eps, out, stream=None):
    _check("spec_add_rmsnorm", load().spec_add_rmsnorm(_ptr(h), _ptr(delta), _ptr(w), R, H, float(eps), _ptr(out),
                                                       _stream(stream)))


def spec_rope_table(tab, max_pos, D, theta, stream=None):
    _check("spec_rope_table", load().spec_rope_table(_ptr(tab), max_pos, D, float(theta), _stream(stream)))


def spec_rope_append(qkv, R, Hq, Hkv, D, rope_tab, max_pos, cu_rows, ctx_start, S, q_out, k_cache, v_cache,
                     num_pages, block_table, max_blocks, k_stage=None, v_stage=None, dev_err=None, stream=None):
    _check("spec_rope_append", load().spec_rope_append(
        _ptr(qkv), R, Hq, Hkv, D, _ptr(rope_tab), max_pos, _ptr(cu_rows), _ptr(ctx_start), S, _ptr(q_out),
        _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(block_table), max_blocks, _ptr(k_stage), _ptr(v_stage),
        _ptr(dev_err), _stream(stream)))


def spec_swiglu(gu, R, F, out, stream=None):
    _check("spec_swiglu", load().spec_swiglu(_ptr(gu), R, F, _ptr(out), _stream(stream)))


def spec_add_rmsnorm_packed(h, delta, w, R, H, eps, out, xpk, stream=None):
    _check("spec_add_rmsnorm_packed", load().spec_add_rmsnorm_packed(_ptr(h), _ptr(delta), _ptr(w), R, H, float(eps),
                                                                     _ptr(out), _ptr(xpk), _stream(stream)))


def spec_swiglu_packed(gu, R, F, out, xpk, stream=None):
    _check("spec_swiglu_packed", load().spec_swiglu_packed(_ptr(gu), R, F, _ptr(out), _ptr(xpk), _stream(stream)))


def spec_flash_decode_packed(q, qkv_dt, Hq, Hkv, D, scale, k_cache, v_cache, num_pages, block_table, max_blocks,
                             ctx_start, cu_rows, S, R, max_kv_len, out, workspace, ws_bytes, xpk, dev_err=None,
                             stream=None):
    _check("spec_flash_decode_packed", load().spec_flash_decode_packed(
        _ptr(q), qkv_dt, Hq, Hkv, D, float(scale), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(block_table),
        max_blocks, _ptr(ctx_start), _ptr(cu_rows), S, R, max_kv_len, _ptr(out), _ptr(workspace), int(ws_bytes),
        _ptr(xpk), _ptr(dev_err), _stream(stream)))


def spec_packed_activation_bytes(K):
    return int(load().spec_packed_activation_bytes(int(K)))


def spec_qmatmul_swiglu(wq, ws, F, K, x, xpk, n_cols, ldx, act, ld_act, workspace, ws_bytes, dev_err=None,
                        stream=None):
    _check("spec_qmatmul_swiglu", load().spec_qmatmul_swiglu(_ptr(wq), _ptr(ws), F, K, _ptr(x), _ptr(xpk), n_cols,
                                                             ldx, _ptr(act), ld_act, _ptr(workspace), ws_bytes,
                                                             _ptr(dev_err), _stream(stream)))


def spec_qmatmul_plan(N, K, n_cols, packed_input=False) -> int:
    return int(load().spec_qmatmul_plan(int(N), int(K), int(n_cols), 1 if packed_input else 0))


def spec_qmatmul_packed(wq, ws, N, K, xpk, n_cols, y, y_dt, ldy, accumulate, workspace, ws_bytes, dev_err=None,
                        stream=None):
    _check("spec_qmatmul_packed", load().spec_qmatmul_packed(_ptr(wq), _ptr(ws), N, K, _ptr(xpk), n_cols, _ptr(y),
                                                             int(y_dt), ldy, int(accumulate), _ptr(workspace),
                                                             int(ws_bytes), _ptr(dev_err), _stream(stream)))


def spec_cast_bf16(inp, n, out, stream=None):
    _check("spec_cast_bf16", load().spec_cast_bf16(_ptr(inp), int(n), _ptr(out), _stream(stream)))


def spec_ngram_draft(hist, hist_cap, hist_len, S, W, pad, drafts, matched_n=None, block_tokens=None, stream=None):
    _check("spec_ngram_draft", load().spec_ngram_draft(_ptr(hist), hist_cap, _ptr(hist_len), S, W, _ptr(pad),
                                                       _ptr(drafts), _ptr(matched_n), _ptr(block_tokens),
                                                       _stream(stream)))


def spec_commit_accepted(hist, hist_cap, hist_len, drafts, W, accepted, correction, ctx_new, ctx, S, dev_err=None,
                         stream=None):
    _check("spec_commit_accepted", load().spec_commit_accepted(
        _ptr(hist), hist_cap, _ptr(hist_len), _ptr(drafts), W, _ptr(accepted), _ptr(correction), _ptr(ctx_new),
        _ptr(ctx), S, _ptr(dev_err), _stream(stream)))
