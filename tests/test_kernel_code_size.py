"""The decode kernel's code stays small (CPU: nvcc only, no GPU).

On short units the tail warps' once-per-unit code ran at the speed of
instruction fetch: a block of a few dozen instructions took about a
microsecond.  Routing the producer's and the MMA warp's walks through one
issue loop each and not unrolling the loops over cluster ranks took the
group-4 kernel from ~262 KB to ~162 KB (whole-unit launches) and from ~249 KB
to ~195 KB (planned launches), and ragged serving from 226 to 203 us per
launch.  This test compiles one instantiation of each to a cubin and fails if
either grows back past a bound with some headroom.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_kv_cache_gb300", "csrc")

# bytes of cubin for one instantiation (whole units, planned launches)
LIMITS = {"false": 185_000, "true": 220_000}


@pytest.mark.parametrize("split", ["false", "true"])
def test_decode_kernel_cubin_size(tmp_path, split):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "one.cu"
    src.write_text('#include "lf_decode_tc.cuh"\nnamespace lf {\n'
                   'const void* take() { return reinterpret_cast<const void*>('
                   f'&decode_step_tc_kernel<4, {split}>); }}\n}}\n')
    out = tmp_path / "one.cubin"
    cmd = [nvcc, "-O3", "-std=c++17", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           "-gencode", "arch=compute_103a,code=sm_103a", "-cubin", "-o", str(out), str(src)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    size = out.stat().st_size
    assert size < LIMITS[split], f"decode_step_tc_kernel<4, {split}>: {size} bytes of cubin"
