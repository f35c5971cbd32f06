"""The C ABI library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching the
device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "spec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import invariant_speculative_verification_gb300 as L
    lib = L.load()
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    import invariant_speculative_verification_gb300 as L
    lib = L.load()
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(3) == b"SPEC_ERR_WORKSPACE"


FAKE = 1 << 20  # a 16-byte aligned non-NULL pointer value; never dereferenced by the host checks


@pytest.mark.parametrize("kw,msg", [
    (dict(K=100), "K >= 256"),
    (dict(K=512 + 32), "multiple of 256"),
    (dict(ldx=500), "ldx"),
    (dict(x=FAKE + 4), "16-byte aligned"),
    (dict(y_dt=1), "y_dt"),
    (dict(N=2097152 + 1, ldy=2097152 + 1), "N must be <= 2097152"),
])
def test_qmatmul_host_validation(kw, msg):
    import invariant_speculative_verification_gb300 as L
    a = dict(wq=FAKE, ws=FAKE, N=64, K=512, x=FAKE, n_cols=1, ldx=512, y=FAKE, y_dt=0, ldy=64)
    a.update(kw)
    if "ldx" not in kw:
        a["ldx"] = max(a["K"], 8) if a["K"] % 8 == 0 else 512
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul(a["wq"], a["ws"], a["N"], a["K"], a["x"], a["n_cols"], a["ldx"], a["y"], a["y_dt"], a["ldy"],
                       0, FAKE, 1 << 30, stream=0)
    assert msg in str(e.value) and e.value.status == 1


@pytest.mark.parametrize("kw,msg,status", [
    (dict(K=768 + 32), "multiple of 256", 1),
    (dict(sbr=FAKE + 8), "16-byte aligned", 1),
    (dict(N=0), "N >= 1", 1),
    (dict(y_dt=1), "y_dt", 1),
    (dict(ws_bytes=16), "workspace", 3),
])
def test_qmatmul_sb_host_validation(kw, msg, status):
    import invariant_speculative_verification_gb300 as L
    a = dict(wq=FAKE, sbr=FAKE, N=64, K=768, x=FAKE, n_cols=2, ldx=1024, y=FAKE, y_dt=0, ldy=64, ws_bytes=1 << 30)
    a.update(kw)
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul_sb(a["wq"], a["sbr"], a["N"], a["K"], a["x"], a["n_cols"], a["ldx"], a["y"], a["y_dt"], a["ldy"],
                          0, FAKE, a["ws_bytes"], stream=0)
    assert msg in str(e.value) and e.value.status == status


def test_flash_decode_host_validation_and_workspace():
    import invariant_speculative_verification_gb300 as L
    ws = L.spec_flash_decode_workspace(10, 8, 128, 1000)
    assert ws >= 10 * 8 * 4 * (128 + 2) * 4
    args = [FAKE, 2, 8, 2, 128, 1.0, FAKE, FAKE, 16, FAKE, 8, FAKE, FAKE, 2, 10, 1000, FAKE, 0, FAKE, ws]
    bad_d = list(args)
    bad_d[4] = 96
    with pytest.raises(L.SpecError, match="D must be"):
        L.spec_flash_decode(*bad_d, stream=0)
    bad_g = list(args)
    bad_g[3] = 3
    with pytest.raises(L.SpecError, match="Hq"):
        L.spec_flash_decode(*bad_g, stream=0)
    short = list(args)
    short[19] = ws - 1
    with pytest.raises(L.SpecError) as e:
        L.spec_flash_decode(*short, stream=0)
    assert e.value.status == 3


def test_qmatmul_workspace_is_checked_on_the_host():
    import invariant_speculative_verification_gb300 as L
    need = L.spec_qmatmul_workspace(64, 512, 8)
    assert need > 0
    with pytest.raises(L.SpecError) as e:
        L.spec_qmatmul(FAKE, FAKE, 64, 512, FAKE, 8, 512, FAKE, 0, 64, 0, FAKE, 16, stream=0)
    assert e.value.status == 3


def test_qmatmul_plan_is_a_host_query_with_fixed_narrow_and_wide_widths():
    """spec_qmatmul_plan: 8 columns -> one 8-column pass, 9-16 -> one 16-column
    pass, more than 80 -> 80-column passes, 17-80 -> one of the three widths;
    packed activations (no packing launch) never make the 80-column pass a
    worse choice; invalid shapes answer 0."""
    import invariant_speculative_verification_gb300 as L
    shapes = [(2048, 2048), (3072, 2048), (2048, 5632), (11264, 2048), (32000, 2048), (17408, 5120), (5120, 17408)]
    for N, K in shapes:
        for n in (1, 8):
            assert L.spec_qmatmul_plan(N, K, n) == 8
        for n in (9, 16):
            assert L.spec_qmatmul_plan(N, K, n) == 16
        for n in (81, 161):
            assert L.spec_qmatmul_plan(N, K, n) == 80
        for n in (17, 33, 48, 64, 80):
            plain, packed = L.spec_qmatmul_plan(N, K, n), L.spec_qmatmul_plan(N, K, n, True)
            assert plain in (8, 16, 80) and packed in (8, 16, 80)
            assert plain != 80 or packed == 80
            assert L.spec_qmatmul_workspace(N, K, n) >= L.spec_qmatmul_workspace(N, K, 8)
    assert L.spec_qmatmul_plan(0, 512, 8) == 0 and L.spec_qmatmul_plan(64, 512, 0) == 0


def test_verify_and_compact_host_validation():
    import invariant_speculative_verification_gb300 as L
    with pytest.raises(L.SpecError, match="multiple of 8"):
        L.spec_verify_greedy(FAKE, 0, 1001, FAKE, 2, 10, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, stream=0)
    with pytest.raises(L.SpecError, match="both or neither"):
        L.spec_kv_compact(FAKE, None, FAKE, FAKE, 8, 128, 16, FAKE, 8, FAKE, FAKE, FAKE, 2, 10, FAKE, FAKE, FAKE,
                          stream=0)


@pytest.mark.parametrize("inv_temp", [0.0, -1.0, float("inf"), float("nan")])
def test_verify_sample_rejects_temperatures_that_are_not_positive_and_finite(inv_temp):
    import invariant_speculative_verification_gb300 as L
    with pytest.raises(L.SpecError, match="inv_temperature") as e:
        L.spec_verify_sample(FAKE, 0, 1000, FAKE, 2, 10, FAKE, FAKE, None, inv_temp, 7, FAKE, FAKE, FAKE, FAKE, FAKE,
                             1 << 20, stream=0)
    assert e.value.status == 1


def test_verify_sample_host_validation():
    import invariant_speculative_verification_gb300 as L
    with pytest.raises(L.SpecError, match="multiple of 8"):
        L.spec_verify_sample(FAKE, 0, 1001, FAKE, 2, 10, FAKE, FAKE, None, 1.25, 7, FAKE, FAKE, FAKE, FAKE, FAKE,
                             1 << 20, stream=0)
    with pytest.raises(L.SpecError, match="S <= R"):
        L.spec_verify_sample(FAKE, 0, 1000, FAKE, 4, 3, FAKE, FAKE, None, 1.25, 7, FAKE, FAKE, FAKE, FAKE, FAKE,
                             1 << 20, stream=0)
    with pytest.raises(L.SpecError, match="16-byte aligned"):
        L.spec_verify_sample(FAKE + 4, 0, 1000, FAKE, 2, 10, FAKE, FAKE, None, 1.25, 7, FAKE, FAKE, FAKE, FAKE, FAKE,
                             1 << 20, stream=0)


def test_zero_sized_calls_launch_nothing():
    import invariant_speculative_verification_gb300 as L
    L.spec_qmatmul(FAKE, FAKE, 64, 512, FAKE, 0, 512, FAKE, 0, 64, 0, None, 0, stream=0)
    L.spec_verify_greedy(FAKE, 0, 1000, FAKE, 0, 0, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, stream=0)


def test_header_compiles_as_c_and_a_c_program_links_and_runs(tmp_path):
    """include/spec.h is plain C: a C11 program that takes the address of every
    declared entry point compiles, links against libspec.so and runs (the calls it
    makes need no GPU)."""
    import shutil
    import subprocess
    import invariant_speculative_verification_gb300 as L
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    names = declared_functions()
    src = tmp_path / "abi.c"
    src.write_text(
        '#include <stdio.h>\n#include "spec.h"\n'
        "typedef void (*fp)(void);\n"
        "static const fp table[] = {\n" + ",\n".join(f"    (fp){n}" for n in names) + "\n};\n"
        "int main(void) {\n"
        "    int n = 0;\n"
        "    for (unsigned i = 0; i < sizeof(table) / sizeof(table[0]); ++i) n += table[i] != 0;\n"
        '    printf("%d %s %s\\n", n, spec_status_string(SPEC_OK), spec_status_string(SPEC_ERR_WORKSPACE));\n'
        "    return 0;\n}\n")
    lib = L.library_path()
    exe = tmp_path / "abi"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out == [str(len(names)), "SPEC_OK", "SPEC_ERR_WORKSPACE"]


def test_glue_host_validation():
    """Each glue entry point rejects bad sizes, NULLs or misalignment on the host
    (status 1, nothing launched)."""
    import invariant_speculative_verification_gb300 as L
    bad = [
        ("embed: bad sizes", lambda: L.spec_embed(FAKE, 0, 64, FAKE, 4, FAKE, stream=0)),
        ("embed: NULL", lambda: L.spec_embed(FAKE, 100, 64, None, 4, FAKE, stream=0)),
        ("H % 4", lambda: L.spec_add_rmsnorm(FAKE, None, FAKE, 4, 66, 1e-6, FAKE, stream=0)),
        ("add_rmsnorm", lambda: L.spec_add_rmsnorm(FAKE + 4, None, FAKE, 4, 64, 1e-6, FAKE, stream=0)),
        ("rope_table", lambda: L.spec_rope_table(FAKE, 128, 63, 10000.0, stream=0)),
        ("rope_table", lambda: L.spec_rope_table(FAKE, 128, 64, -1.0, stream=0)),
        ("swiglu: bad sizes", lambda: L.spec_swiglu(FAKE, 4, 0, FAKE, stream=0)),
        ("65535", lambda: L.spec_swiglu(FAKE, 65536, 64, FAKE, stream=0)),
        ("cast_bf16", lambda: L.spec_cast_bf16(None, 8, FAKE, stream=0)),
        ("ngram_draft: bad sizes", lambda: L.spec_ngram_draft(FAKE, 0, FAKE, 2, 4, FAKE, FAKE, stream=0)),
        ("ngram_draft: NULL", lambda: L.spec_ngram_draft(FAKE, 64, FAKE, 2, 4, None, FAKE, stream=0)),
        ("commit_accepted: bad sizes",
         lambda: L.spec_commit_accepted(FAKE, 0, FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, 2, stream=0)),
    ]
    for msg, call in bad:
        with pytest.raises(L.SpecError) as e:
            call()
        assert e.value.status == 1 and msg.split(":")[0] in str(e.value), (msg, str(e.value))
