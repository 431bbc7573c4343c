"""The decode kernels' shared-memory layouts, checked on the host: tests/native/layout_check.cu
includes the kernels' own layout functions and sweeps layer shapes (formats, expert counts,
widths, token counts, top-k); for every shape a kernel accepts, its regions must be ordered,
16-byte aligned, large enough for their contents and within one CTA's opt-in shared memory."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_shared_memory_layouts(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "layout_check")
    src = os.path.join(ROOT, "tests", "native", "layout_check.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17",
                        "-I", os.path.join(ROOT, "include"), "-o", exe, src], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-3000:]
    assert " 0 failures" in out.stdout
    n = int(out.stdout.split("checked ")[1].split()[0])
    assert n > 10000
