"""The C ABI from plain C: tests/c/abi_consumer.c, a C99 program that sees
only include/moelora.h, is compiled with gcc against the built library and
run.  Its calls are host-only (sizing, status strings, argument checks), so
it needs no GPU."""
import os
import shutil
import subprocess

import pytest

from lora_mixture_experts_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_program_uses_the_abi(tmp_path, lib):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    so = binding.library_path()
    exe = str(tmp_path / "abi_consumer")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_consumer.c"),
           "-o", exe, so, "-Wl,-rpath," + os.path.dirname(so)]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK"), r.stdout
    # the C program sizes the workspace exactly as the Python binding does
    d = binding.moelora_dims(16, 4, 32, 2880, 2880, 8, 32)
    assert int(r.stdout.split()[1]) == binding.moelora_workspace_bytes(d)
