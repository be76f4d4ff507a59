"""The library as a plain C program sees it: tests/c_caller/usm_c_caller.c
includes include/usm.h, links libusm.so and the CUDA runtime, and runs
row_swizzle_build, csr_spmm and csr_sddmm on device memory it allocates
itself.  The CPU test only compiles and links it; the GPU test runs it and
checks its outputs against the oracle."""
import os
import subprocess

import numpy as np
import pytest

import workloads as W
from parity_util import TOL, assert_within, oracle_sddmm, oracle_spmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "usm_c_caller.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_caller(out_dir):
    from unstructured_sparse_matmul_gb300 import build as usm_build
    lib = usm_build.build_library()
    lib_dir = os.path.dirname(lib)
    exe = os.path.join(out_dir, "usm_c_caller")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", lib_dir, "-lusm",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    exe = compile_caller(str(tmp_path))
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_caller_runs_spmm_and_sddmm(tmp_path):
    M, K, N, D = 300, 700, 200, 152  # ragged strips and tiles; pitches of 16-byte multiples
    csr = W.random_csr(160, M, K, 0.1)
    rng = np.random.default_rng(161)
    B, X, Y = W.dense(rng, K, N), W.dense(rng, M, D), W.dense(rng, K, D)
    header = np.array([M, K, N, D, csr.nnz], dtype=np.int32)
    with open(tmp_path / "problem.bin", "wb") as f:
        for a in (header, csr.row_offsets.astype(np.int32), csr.col_indices.astype(np.int32),
                  csr.values.astype(np.float32), B, X, Y):
            f.write(np.ascontiguousarray(a).tobytes())
    exe = compile_caller(str(tmp_path))
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    C = np.fromfile(tmp_path / "C.bin", dtype=np.float32).reshape(M, N)
    out = np.fromfile(tmp_path / "out.bin", dtype=np.float32)
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(C, ref, S, TOL["f32"], "spmm from C")
    ref, S, _ = oracle_sddmm(csr, X, Y, "f32")
    assert_within(out, ref, S, TOL["f32"], "sddmm from C")
