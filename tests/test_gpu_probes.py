"""Hardware facts the kernels rely on, measured on the GPU by the probes in
tests/probes/ (compiled here with nvcc for sm_103a):

* shared memory delivers 128 bytes per clock per SM to LDS.32/64/128 at
  random staged rows, and the FP32 pipe does 128 FMAs per clock per SM
  (fma.rn.f32x2), so one dense element per useful FMA from shared memory
  caps fp32 at a quarter of the FP32 peak (the operand-delivery bound);
* tcgen05.ld from tensor memory delivers more than shared memory does, and
  the two paths work side by side;
* tcgen05.cp.32x128b.warpx4 puts row i of a 512-byte shared-memory block
  into lane i of every subpartition (the layout the SpMM kernel's
  tensor-memory rows use), bit for bit, and issuing it from every warp
  fills tensor memory several times faster than from one thread.

The rates are taken with clock64() inside each CTA, so they do not depend on
the SM clock."""
import json
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
PROBES = os.path.join(HERE, "probes")


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    pytest.skip("nvcc not found")


def run_probe(tmp_path, name, *args):
    exe = str(tmp_path / name)
    subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "--expt-extended-lambda", "-o", exe, os.path.join(PROBES, name + ".cu")], check=True)
    r = subprocess.run([exe, *args], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    out = {}
    for line in r.stdout.splitlines():
        d = json.loads(line)
        out[d.get("probe", "summary")] = d
    return out


def test_operand_delivery_rates(tmp_path):
    p = run_probe(tmp_path, "operand_probe", "t")
    for k in ("lds32_random_rows", "lds64_random_rows", "lds128_random_rows"):
        assert 120 <= p[k]["bytes_per_clk_sm"] <= 129, p[k]
    assert 250 <= p["fma_f32x2"]["flop_per_clk_sm"] <= 257
    assert p["fma_f32_bf16"]["flop_per_clk_sm"] >= 230
    assert p["tmem_ld_32x32b_x4"]["bytes_per_clk_sm"] > 1.5 * p["lds128_same_loop"]["bytes_per_clk_sm"]
    # side by side: the mixed loop moves about twice what LDS alone does
    assert p["tmem_ld_plus_lds128_mixed"]["bytes_per_clk_sm"] > 1.8 * p["lds128_same_loop"]["bytes_per_clk_sm"]


def test_tensor_memory_copy_layout(tmp_path):
    p = run_probe(tmp_path, "tmem_cp_probe")
    cp = p["tcgen05_cp_32x128b_warpx4"]
    assert cp["mismatches"] == 0 and cp["timeouts"] == 0 and cp["checked_words"] == 128 * 512
    assert p["tcgen05_ld_32x32b_x8_4perwait"]["bytes_per_clk_sm_16warps"] > 200


def test_tensor_memory_fill_rates(tmp_path):
    p = run_probe(tmp_path, "tmem_fill_probe")
    assert p["summary"]["timeouts"] == 0
    one = p["cp32x128b_warpx4_1thr"]["source_bytes_per_clk"]
    all16 = p["cp32x128b_warpx4_16thr"]["source_bytes_per_clk"]
    assert all16 > 4 * one
