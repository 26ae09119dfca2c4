"""The boundary as a plain C ABI: tests/c_client.c includes only
include/mla_decode.h, links libmla_decode.so with gcc and runs without Python
or torch in the process (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from mla_decode_attention_uk_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_library_through_the_header(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    binding.lib()  # builds the library if it is missing or stale
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path / "c_client")
    subprocess.run([gcc, "-std=c11", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_client.c"),
                    "-L", libdir, "-l:" + os.path.basename(binding.LIB_PATH),
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client: ok" in r.stdout
