"""Builds and runs tests/c_abi/spconv_c_test.c: the C ABI driven from plain C
(gcc, no Python or PyTorch in the process), checked against the C oracle."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build(tmp_path):
    from sparse_weight_direct_gb300 import build as b
    b.build()
    lib_dir = os.path.dirname(b.LIB)
    subprocess.run(["make", "-s", "-C", os.path.join(ROOT, "oracle")], check=True)
    cuda = b.cuda_home()
    exe = str(tmp_path / "spconv_c_test")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi", "spconv_c_test.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", lib_dir, "-lspconv", "-L", os.path.join(ROOT, "oracle"), "-loracle",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(ROOT, "oracle"),
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_abi_host_only(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "--host-only"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host-only ok" in r.stdout


@pytest.mark.gpu
def test_c_abi_forward_parity(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 out of tolerance" in r.stdout
