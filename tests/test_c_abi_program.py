"""The C ABI from plain C: tests/c/abi_roundtrip.c and tests/c/pdl_graph.c
compile as C11 against include/ep.h and link against the library (CPU); on
the GPU the first runs the hand-worked two-rank example (also as a
partitioned group), the second captures it into CUDA graphs and checks the
edge EP_LAUNCH_PDL records."""
import os
import shutil
import subprocess

import pytest

from combine_topk_ids_dest_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_roundtrip.c")
PDL_SRC = os.path.join(ROOT, "tests", "c", "pdl_graph.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path, src=SRC):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = _lib.load()._name
    exe = os.path.join(str(tmp_path), os.path.splitext(os.path.basename(src))[0])
    libdir = os.path.dirname(lib)
    cuda_lib = next((d for d in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"))
                     if os.path.exists(os.path.join(d, "libcudart.so"))), os.path.join(CUDA, "lib64"))
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), src, "-o", exe, f"-L{libdir}", "-l:libep_gb300.so",
           f"-Wl,-rpath,{libdir}", f"-L{cuda_lib}", "-lcudart", f"-Wl,-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))
    assert os.path.exists(_build(tmp_path, PDL_SRC))


@pytest.mark.gpu
def test_c_program_runs_worked_example(tmp_path, cuda_device):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_roundtrip: ok" in r.stdout


@pytest.mark.gpu
def test_c_program_pdl_graph_edges(tmp_path, cuda_device):
    exe = _build(tmp_path, PDL_SRC)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "pdl_graph: ok" in r.stdout
