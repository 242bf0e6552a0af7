"""The C ABI used from plain C: tests/c/abi_consumer.c is compiled as C99
against include/ddp_reducer.h, linked to the in-tree libddpreducer.so and run
(bucket assignment, locators and the readiness state machine in dry run; no
GPU needed)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "reduction_reducer_gb300")


@pytest.fixture(scope="module")
def lib_path():
    from reduction_reducer_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.LIB_PATH


def test_c_consumer(lib_path, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-L", PKG, "-lddpreducer",
                    f"-Wl,-rpath,{PKG}", "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "c abi ok"


def _cuda_home():
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    return os.environ.get("CUDA_HOME") or (os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if nvcc else None)


def _build_gpu_consumer(lib_path, out):
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = _cuda_home()
    if cc is None or cuda is None:
        pytest.skip("no C compiler or CUDA toolkit")
    cudalib = os.path.join(cuda, "lib64")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "abi_gpu.c"),
                    "-L", PKG, "-lddpreducer", "-L", cudalib, "-lcudart", f"-Wl,-rpath,{PKG}",
                    f"-Wl,-rpath,{cudalib}", "-o", str(out)], check=True, capture_output=True, text=True)


def test_c_gpu_consumer_builds(lib_path, tmp_path):
    """The GPU consumer compiles and links against the header, the library and
    the CUDA runtime (running it needs a GPU: test_c_gpu_consumer)."""
    _build_gpu_consumer(lib_path, tmp_path / "abi_gpu")


@pytest.mark.gpu
def test_c_gpu_consumer(lib_path, tmp_path):
    """One iteration through the C ABI from plain C on the GPU: cudaMalloc'd
    replicas, bind, mark_ready_many, every copied-back element and the bucket
    arena checked against the exact means."""
    exe = tmp_path / "abi_gpu"
    _build_gpu_consumer(lib_path, exe)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "c abi gpu ok"
