"""The C ABI from plain C99 (CPU): tests/c/abi_host.c includes include/llm.h and llm_ops.h,
links libllm.so and calls the host-only entry points."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_program_uses_the_abi(tmp_path):
    import quantized_decode_gb300 as qd
    lib = qd.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_host"
    libdir = os.path.dirname(lib)
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", str(exe),
                           "-L", libdir, "-lllm", f"-Wl,-rpath,{libdir}"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"
