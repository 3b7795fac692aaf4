"""The range-checked build of the library (libnomas_checked.so).

Compute-sanitizer is not available to this project's GPU runs, so out-of-range
work is caught by a second build of the same kernels in which every computed
global-memory index is checked before its access (a bad index records
NOMAS_ERR_INVALID_ARG in the device error word and the access is skipped;
nothing traps).  These tests check that the check mechanism reports, and run
the GPU parity suites against that build in a child process: every test there
asserts afterwards that the device error word is still 0, so a green run means
no kernel computed an index outside its buffers on any of those inputs.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_sparse.py", "tests/test_gpu_fp8.py",
          "tests/test_gpu_append_rope.py", "tests/test_gpu_archive.py", "tests/test_gpu_camera.py",
          "tests/test_gpu_session.py", "tests/test_gpu_resume.py", "tests/test_gpu_expand.py"]


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_checked_library_reports_a_failed_range_check():
    _need_gpu()
    code = (
        "import torch, segment_causal_kv_int8_b300 as n\n"
        "assert n.nomas_bounds_checked() == 1, n.LIB_PATH\n"
        "assert n.device_error(clear=True) == 0\n"
        "assert n.nomas_selftest_bounds_check(n._stream_ptr()) == n.NOMAS_OK\n"
        "torch.cuda.synchronize()\n"
        "assert n.device_error(clear=True) == n.NOMAS_ERR_INVALID_ARG\n"
        "assert n.device_error(clear=False) == 0\n"
        "x = torch.arange(8, device='cuda', dtype=torch.float32)\n"
        "assert float(x.sum()) == 28.0\n"
    )
    env = dict(os.environ, NOMAS_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr


def test_regular_library_has_no_range_checks():
    _need_gpu()
    import segment_causal_kv_int8_b300 as n
    if n.nomas_bounds_checked():
        pytest.skip("this process loaded the checked build")
    assert n.nomas_selftest_bounds_check(n._stream_ptr()) == n.NOMAS_ERR_UNSUPPORTED


def test_gpu_parity_suites_under_the_checked_build():
    _need_gpu()
    env = dict(os.environ, NOMAS_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
