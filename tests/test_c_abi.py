"""The C ABI from plain C: swz.h compiles as strict C99 on its own, and a C99
program (tests/c/swz_abi_example.c) links libswz.so and calls it.  The host
entry points run without a GPU; the --gpu run allocates device memory through
the CUDA runtime and checks a forward and inverse relayout."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _lib_dir():
    import xor_swizzle_movement_gb300 as m
    if not os.path.exists(m.library_path()):
        from xor_swizzle_movement_gb300 import build
        build.build()
    return os.path.dirname(m.library_path())


@pytest.fixture(scope="module")
def example(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib_dir = _lib_dir()
    out = str(tmp_path_factory.mktemp("c_abi") / "swz_abi_example")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", f"-I{ROOT}/include", f"-I{CUDA}/include",
           os.path.join(ROOT, "tests", "c", "swz_abi_example.c"), "-o", out, f"-L{lib_dir}", "-lswz",
           f"-L{CUDA}/lib64", "-lcudart", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{CUDA}/lib64"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def test_header_is_strict_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "hdr.c"
    src.write_text('#include "swz.h"\nint main(void) { return swz_version() > 0 ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{ROOT}/include",
                    "-fsyntax-only", str(src)], check=True, capture_output=True, text=True)


def test_c_caller_host_functions(example):
    r = subprocess.run([example], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "ok" in r.stdout


@pytest.mark.gpu
def test_c_caller_relayout_on_gpu(example):
    r = subprocess.run([example, "--gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
