"""The C ABI from plain C: tests/c_client/tpmlp_c_client.c includes only include/tpmlp.h and the
CUDA runtime API. On the CPU it must compile as strict C11 (the header is valid C) and link
against libtpmlp.so; on a GPU it runs the block and checks it against the fp64 oracle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "tpmlp_c_client.c")
PKG = os.path.join(ROOT, "tensor_transformer_mlp_tmem_gb300")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build(tmp_path):
    from tensor_transformer_mlp_tmem_gb300 import _build as b
    b.build()
    cuda = _cuda_home()
    exe = str(tmp_path / "tpmlp_c_client")
    obj = str(tmp_path / "tpmlp_c_client.o")
    inc = ["-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include")]
    # the client alone under strict C11 warnings: the header must be valid C
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Wpedantic", "-Werror", "-O2", *inc,
                    "-c", SRC, "-o", obj], check=True, capture_output=True, text=True)
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", obj,
           os.path.join(ROOT, "synth", "synth.c"), os.path.join(ROOT, "oracle", "tpmlp_oracle.c"),
           "-L", PKG, "-ltpmlp", "-Wl,-rpath," + PKG,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-lm", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_compiles_as_c11_and_links(tmp_path):
    exe = _build(tmp_path)
    assert os.path.exists(exe)


@pytest.mark.gpu
@pytest.mark.parametrize("args", [(), ("768", "3072", "4", "1000", "1")])
def test_c_client_runs_the_block(lib, tmp_path, args):
    exe = _build(tmp_path)
    out = subprocess.run([exe, *args], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "c client:" in out.stdout
    print(out.stdout.strip())
