"""Batch-invariant greedy speculative verification on GB300 (sm_103a).

The compute path lives in libspec.so (CUDA kernels behind a C ABI, see
include/spec.h); this package is its ctypes binding plus the end-to-end
decoder harness that drives it.  Importing the package loads the library and
raises if it cannot: there is no CPU path.
"""
from ._lib import (DEVERR, SPEC_BF16, SPEC_F16, SPEC_F32, SpecError, library_path, load,  # noqa: F401
                   spec_add_rmsnorm, spec_add_rmsnorm_packed, spec_cast_bf16, spec_commit_accepted, spec_debug_wait_timeout, spec_embed,
                   spec_flash_decode, spec_flash_decode_packed, spec_flash_decode_workspace, spec_gate_scatter, spec_kv_compact, spec_margin_gate,
                   spec_margin_gate_workspace, spec_ngram_draft, spec_packed_activation_bytes, spec_qmatmul,
                   spec_qmatmul_devcols, spec_qmatmul_packed, spec_qmatmul_plan, spec_qmatmul_swiglu,
                   spec_qmatmul_debug_nt, spec_qmatmul_noninvariant, spec_qmatmul_sb, spec_qmatmul_static_scratch,
                   spec_qmatmul_workspace,
                   spec_rope_append, spec_rope_table,
                   spec_swiglu, spec_swiglu_packed, spec_verify_greedy, spec_verify_greedy_workspace, spec_verify_sample)

load()
