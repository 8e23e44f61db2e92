"""The C ABI from plain C: include/nbody.h compiles as C99 and C++, and a C
program linked against libnbody.so computes forces and steps on the GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
CUDA = "/usr/local/cuda"


def _cuda_include():
    return os.path.join(CUDA, "include")


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles_standalone(tmp_path, lang):
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "nbody.h"\nint main(void) { return (int)NBODY_OK; }\n')
    std = "-std=c99" if lang == "c" else "-std=c++17"
    cc = "gcc" if lang == "c" else "g++"
    subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I" + INCLUDE,
                    "-I" + _cuda_include(), str(src)], check=True)


@pytest.mark.gpu
def test_c_program_on_the_gpu(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    lib_dir = os.path.join(ROOT, "all_pairs_gravitational_gb300")
    exe = tmp_path / "abi_check"
    cudart = os.path.join(CUDA, "lib64")
    if not os.path.isdir(cudart):
        cudart = os.path.join(CUDA, "lib")
    subprocess.run(["gcc", "-std=c99", "-O2", "-I" + INCLUDE, "-I" + _cuda_include(),
                    os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", str(exe),
                    "-L" + lib_dir, "-lnbody", "-L" + cudart, "-lcudart", "-lm",
                    "-Wl,-rpath," + lib_dir + ":" + cudart], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "bit for bit" in r.stdout
