"""The C ABI used from plain C: tests/c_abi/moe_c_client.c includes only
include/moe_layout.h and the CUDA runtime header, links libmoe_layout.so, and
checks the library's outputs bit for bit against the oracle's C functions.

The host part (status strings, plan and workspace queries, synchronous
argument rejection) runs without a GPU; the GPU part runs layout+dispatch
(bf16 and FP8) and combine on a decode-sized and a prefill-sized batch.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CLIENT_SRC = os.path.join(ROOT, "tests", "c_abi", "moe_c_client.c")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cuda_lib_dir():
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        d = os.path.join(CUDA_HOME, sub)
        if os.path.exists(os.path.join(d, "libcudart_static.a")):
            return d
    return None


@pytest.fixture(scope="module")
def c_client(tmp_path_factory, oracle):
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_lib = _cuda_lib_dir()
    if cc is None or cuda_lib is None:
        pytest.skip("needs a C compiler and the CUDA runtime's static library")
    from combine_moe_layout_05_gb300 import build as lib_build
    lib = lib_build.build()
    oracle_lib = oracle.build()
    out = str(tmp_path_factory.mktemp("c_abi") / "moe_c_client")
    lib_dir, oracle_dir = os.path.dirname(lib), os.path.dirname(oracle_lib)
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror",
           f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(CUDA_HOME, 'include')}",
           CLIENT_SRC, "-o", out,
           f"-L{lib_dir}", f"-L{oracle_dir}", f"-L{cuda_lib}",
           "-lmoe_layout", "-loracle", "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-lm",
           f"-Wl,-rpath,{lib_dir}:{oracle_dir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return out


def _run(client, mode, timeout):
    res = subprocess.run([client, mode], capture_output=True, text=True, timeout=timeout)
    assert res.returncode == 0, f"stdout:\n{res.stdout}\nstderr:\n{res.stderr}"
    return res.stdout


def test_c_client_host_checks(c_client):
    assert "all checks passed" in _run(c_client, "host", 60)


@pytest.mark.gpu
def test_c_client_gpu_parity(c_client):
    out = _run(c_client, "gpu", 300)
    assert "all checks passed" in out
    # the decode-sized batch took the single-kernel path, the prefill-sized
    # one the two-launch path
    assert "T=128 H=1024 K=8 E=64 R=8 bf16: 1 launches" in out
    assert "T=4096 H=1024 K=8 E=128 R=16 fp8: 2 launches" in out
