"""The checked build (NVFP4_CHECKED=1): every kernel tests the indices of
the global-memory accesses it computes against its tensor's extent and
reports a stray one as NVFP4_ERR_BOUNDS.  Compute sanitizers are not
available everywhere this library runs; this build answers the same
question for the library's own index arithmetic.

The parity suites of the quantizers, the GEMM and the linear layer run again
in a child process that loads the checked library: every one of their calls
is followed by a status check, so an index outside its tensor fails them
(and their results are compared with the oracle as usual).  The self-test
shows that the check itself works: one guarded store one past its buffer is
skipped and reported, and the word behind the buffer stays untouched.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = ["tests/test_gpu_10_quantize.py", "tests/test_gpu_15_mxfp4.py", "tests/test_gpu_17_rht_fprop_dgrad.py",
          "tests/test_gpu_19_quantize_with_rht.py", "tests/test_gpu_20_gemm.py", "tests/test_gpu_30_linear.py"]


def _child(code_or_args, is_pytest=False):
    env = dict(os.environ, NVFP4_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *code_or_args] if is_pytest \
        else [sys.executable, "-c", code_or_args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)


def test_checked_library_reports_a_stray_index():
    r = _child("import sys; sys.path.insert(0, '.')\n"
               "from quantize_block_scaled_amax_gb300 import build; build.build()\n"
               "import quantize_block_scaled_amax_gb300 as nv\n"
               "assert build.CHECKED and nv.nvfp4_checked_build(), 'not the checked library'\n"
               "st = nv.nvfp4_checked_selftest()\n"
               "assert st == nv.ERR_BOUNDS, st\n"
               "assert nv.nvfp4_sync_status() == nv.OK\n"
               "print('selftest ok')\n")
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "selftest ok" in r.stdout


def test_parity_suites_pass_on_the_checked_library():
    r = _child(SUITES, is_pytest=True)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_normal_build_is_not_checked():
    from quantize_block_scaled_amax_gb300 import build
    if build.CHECKED:
        pytest.skip("this process runs the checked build")
    build.build()
    import quantize_block_scaled_amax_gb300 as nv
    assert not nv.nvfp4_checked_build()
    assert nv.nvfp4_checked_selftest() == nv.ERR_UNSUPPORTED
