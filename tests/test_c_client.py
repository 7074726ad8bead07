"""The C ABI from plain C: a C99 program that includes only include/pa.h,
links libpagedattn.so and calls the host-only entry points and host-side
checks (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_calls_the_abi(tmp_path):
    from paged_kv_cache_context_gb300 import build
    lib = build.build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "pa_client")
    libdir = os.path.dirname(lib)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_client", "pa_client.c"), "-o", exe,
                        "-L", libdir, "-l:libpagedattn.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    got = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert int(got["version"]) >= 1 << 16
    assert got["status_shape"] == "inconsistent or unsupported sizes"
    assert got["plan_rc"] == "0" and got["plan_covers"] == "1"
    assert int(got["ws_g4_d128"]) > 3840
    assert got["budget_mb"] == "1024" and got["budget_ctx"] == "32"
    assert got["decode_empty"] == "0"
    assert got["decode_head_dim"] == "-4" and got["decode_group"] == "-3"
    assert got["write_null"] == "-1" and got["int8_f32_query"] == "-2"
    assert got["prefill_fp8_scale"] == "-11"
    assert got["cascade_fp8_head_dim"] == "-4" and got["cascade_int8_null_scales"] == "-1"
