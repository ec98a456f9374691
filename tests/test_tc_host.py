"""The decode kernel's shared-memory stage layout and stream-K bookkeeping,
checked on the host.

``tests/tc_host_check.cu`` includes the kernel header and checks, for every
template configuration, that the consumers' row addresses are where the
producer's 4-D TMA boxes land, that each row keeps its swizzle phase, and that
the bytes a stage expects equal the bytes delivered; then, by brute force,
that the chunk-to-CTA and chunk-to-sequence maps match their definitions and
that no sequence spans more CTAs than the partial slots the plan reserves;
and, over plain and shared-prefix units, that the partial slots of all
partitions are distinct, match each sequence's listed ranges, stay within
the workspace bound and cover its whole context (planted slot mistakes must
fail).
Built with nvcc for the host; no GPU is needed.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_115_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_stage_layout_and_stream_k_bookkeeping(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "tc_host_check")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-DPKV_BUILD", "-o", exe,
           os.path.join(ROOT, "tests", "tc_host_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "layout ok" in r.stdout and "stream-K ok" in r.stdout
    assert "partial slots ok" in r.stdout
