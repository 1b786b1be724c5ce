"""The debug build (compiled with MOE_DEBUG_BOUNDS): every index the kernels
read from data (permutation and inverse entries, list entries, expert ids
taken from a list) is checked against the extent of the array it indexes; a
bad one is recorded and the access skipped, and moe_sync_status reports
MOE_ERR_BOUNDS.  The parent test runs a representative part of the GPU suite
through the debug library in a child process (MOE_FFN_DEBUG_BOUNDS=1): the
correct runs keep their parity and raise no bounds flag.  The self-test,
which only that child runs, shows that a bad index is reported and skipped.
The release library checks nothing and refuses the self-test."""
import os
import re
import subprocess
import sys

import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
from _gpu import DEV

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEBUG = os.environ.get("MOE_FFN_DEBUG_BOUNDS") == "1"

# the suite's cases run through the debug library: routing (fused and split
# clusters, hash, near ties), dispatch, the bf16 forward on the small layers
# and edge shapes, the top-1 fused combine, bad ids and tokens, the A8W8 and
# MX forwards and the backward
CHILD_SELECTION = ("selftest or route_matches or route_split or one_lane or large_scores or near_ties or "
                   "dispatch or forward_matches or edge_shapes or m64 or ragged or dense or top1 or bad_ or "
                   "poisoned or quantisation or (backward_matches and not 1040)")
CHILD_FILES = ["tests/test_gpu_debug_bounds.py", "tests/test_gpu_parity.py", "tests/test_gpu_a8w8.py",
               "tests/test_gpu_mx.py", "tests/test_gpu_backward.py"]


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


@pytest.mark.skipif(DEBUG, reason="the child process runs the debug library")
def test_release_library_refuses_the_bounds_selftest():
    ws = moe.alloc_workspace(moe.make_params(1, 64, 8, 1, 64), DEV)
    assert moe.moe_selftest_bounds(ws, 40) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_OK


@pytest.mark.skipif(not DEBUG, reason="runs in the child process of test_debug_build_runs_the_suite")
def test_bounds_selftest_reports_and_skips():
    ws = moe.alloc_workspace(moe.make_params(1, 64, 8, 1, 64), DEV)
    for i in (0, 31):
        assert moe.moe_selftest_bounds(ws, i) == moe.MOE_OK
        assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_OK
    for i in (32, -1, 1 << 40):
        assert moe.moe_selftest_bounds(ws, i) == moe.MOE_OK
        assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_ERR_BOUNDS
        # the word is cleared by the report
        assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_OK
    # the skipped writes left the array (bytes 128.. of the status header) alone
    arr = ws[128:256].view(torch.int32).cpu()
    assert int(arr[0]) == 1 and int(arr[31]) == 1 and int(arr[1:31].sum()) == 0


@pytest.mark.skipif(DEBUG, reason="the parent")
def test_debug_build_runs_the_suite():
    env = dict(os.environ, MOE_FFN_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-rs", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", CHILD_SELECTION, *CHILD_FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    out = r.stdout + r.stderr
    tail = "\n".join(out.splitlines()[-30:])
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", tail)
    assert m and int(m.group(1)) >= 40, tail  # the selection above is ~60 cases
    assert "runs in the child process" not in out, tail  # the self-test ran there
