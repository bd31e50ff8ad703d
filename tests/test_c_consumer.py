"""The C ABI from plain C: tests/c_consumer.c (C11, no Python, no C++) quantizes on the GPU
through include/mxfp8.h and compares every byte with the oracle.  The CPU suite compiles it
(the header is valid C); the GPU suite runs it."""
import os
import subprocess

import pytest

import mxfp8_block_scaled_04_gb300 as mx
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_consumer(out):
    lib = mx.binding.lib()._name
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_consumer.c"), lib,
                    oracle.build(), "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", out], check=True)


def test_c_consumer_compiles(tmp_path):
    build_consumer(str(tmp_path / "c_consumer"))


@pytest.mark.gpu
def test_c_consumer_runs(tmp_path):
    exe = str(tmp_path / "c_consumer")
    build_consumer(exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c consumer ok" in r.stdout
