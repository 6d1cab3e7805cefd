"""Host-side logic of the chunked prefill, checked on the CPU: the split
schedule's pieces cover every chunk of every unit exactly once, the K order
of S' in TMEM (kperm) is the permutation S -> S' writes, and every kernel
shape's shared memory and stage counts fit one CTA.  The checks are C++
(tests/host_schedule.cu) compiled against the kernel header by nvcc; no GPU
is used."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.mark.skipif(not (os.path.exists(NVCC) or shutil.which("nvcc")), reason="nvcc not installed")
def test_host_schedule_and_layout(tmp_path):
    exe = str(tmp_path / "host_schedule")
    subprocess.check_call([NVCC if os.path.exists(NVCC) else "nvcc", "-std=c++17", "--expt-relaxed-constexpr",
                           "-gencode", "arch=compute_103a,code=sm_103a", "-I", os.path.join(HERE, "..", "include"),
                           "-o", exe, os.path.join(HERE, "host_schedule.cu")])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok: 0 failures" in r.stdout
