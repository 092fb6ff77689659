"""The C ABI used from plain C: tests/c_abi/abi_client.c is compiled with gcc
as C99 against include/sga.h and linked to libsga.so (no torch, no Python in
the loop).  On CPU it checks host-side validation; on a GPU it runs a two-shard
argmax + reduce on cudaMalloc'd buffers and checks the ids."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_client.c")


def build_client(tmp_path, sga_lib):
    lib_dir = os.path.dirname(sga_lib.LIB_PATH)
    exe = tmp_path / "abi_client"
    cuda_lib = "/usr/local/cuda/lib64"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"), SRC,
                    "-o", str(exe), "-L" + lib_dir, "-l:libsga.so", "-L" + cuda_lib, "-lcudart",
                    "-Wl,-rpath," + lib_dir + ":" + cuda_lib, "-lm"],
                   check=True, capture_output=True, text=True)
    return exe


def test_c_client_host_checks(tmp_path, sga_lib):
    exe = build_client(tmp_path, sga_lib)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_client_gpu_argmax(tmp_path, sga_lib):
    exe = build_client(tmp_path, sga_lib)
    r = subprocess.run([str(exe), "gpu"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
