"""The C ABI from plain C: include/qgemm.h compiles as strict C99, a C
program links against libqgemm.so and gets the host-side answers (a workspace
query, a refused width and its status string) without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built_lib():
    from gemm_blockwise_dequant_gb300 import build

    return build.build()


def test_c99_program_links_and_runs(built_lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(built_lib)
    exe = str(tmp_path / "c_abi_host")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_host.c"), "-L", libdir, "-lqgemm", "-Wl,-rpath," + libdir,
                    "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.split() == ["0", "2", "QG_ERR_UNSUPPORTED"]
