"""The GEMM kernel compiles with no stack frame and no register spills.

A `tcgen05.ld` writes its destination registers asynchronously; they are
valid only after `tcgen05.wait::ld`.  When the epilogue held more
accumulator words than the 128-register cap of a 512-thread CTA allows,
ptxas spilled some of them, and repeated full-size launches on the same
operands differed in a few thousand output elements.  The epilogue now
keeps at most 64 accumulator words live and issues each load with its wait
in one statement; this test keeps it that way.  It needs nvcc only (the
compile targets sm_103a without a GPU), and reads the figures ptxas prints
with -v.
"""
import os
import re
import shutil
import subprocess

import pytest

from quantize_block_scaled_amax_gb300 import build as nvbuild


def _nvcc():
    try:
        return nvbuild.nvcc()
    except RuntimeError:
        return None


@pytest.mark.skipif(_nvcc() is None, reason="nvcc not available")
def test_gemm_kernel_has_no_spills(tmp_path):
    src = os.path.join(nvbuild.CSRC, "gemm.cu")
    cmd = [_nvcc(), *nvbuild.ARCH, *nvbuild.NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o", str(tmp_path / "gemm.o")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    out = r.stdout + r.stderr
    # ptxas prints, per entry function: "Compiling entry function '<name>'",
    # then "<s> bytes stack frame, <st> bytes spill stores, <ld> bytes spill loads"
    found = {}
    current = None
    for line in out.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and current is not None and current not in found:
            found[current] = tuple(int(v) for v in m.groups())
    gemm = {name: v for name, v in found.items() if "nvf4_gemm_kernel" in name}
    assert gemm, f"no ptxas report for nvf4_gemm_kernel in:\n{out}"
    for name, (stack, spill_st, spill_ld) in gemm.items():
        assert (stack, spill_st, spill_ld) == (0, 0, 0), (
            f"{name}: {stack} bytes stack frame, {spill_st} bytes spill stores, {spill_ld} bytes spill loads")
