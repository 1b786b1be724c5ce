import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


DEBUG_BOUNDS = os.environ.get("MOE_FFN_DEBUG_BOUNDS") == "1"


def _lib_is_stale():
    from mixture_experts_ffn_route_gb300 import build as b
    lib = b.LIB_DEBUG if DEBUG_BOUNDS else b.LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = b.sources() + [os.path.join(b.CSRC, f) for f in os.listdir(b.CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "moe_ffn.h"))
    return any(os.path.getmtime(d) > t for d in deps)


@pytest.fixture(scope="session")
def built_lib():
    """The in-tree CUDA library, (re)built with nvcc when missing or stale
    (the bounds-checked debug build under MOE_FFN_DEBUG_BOUNDS=1)."""
    from mixture_experts_ffn_route_gb300 import build as b
    if _lib_is_stale():
        b.build(debug=DEBUG_BOUNDS)
    return b.LIB_DEBUG if DEBUG_BOUNDS else b.LIB


def pytest_terminal_summary(terminalreporter):
    """Print the Y parity of every checked case: max|err|/RMS against the
    oracle rounded at the path's rounding points (the bar is 2e-2), and
    against the exact oracle with the count of elements beyond 2e-2 RMS."""
    mod = sys.modules.get("_gpu")
    if mod is None or not mod.Y_STATS:
        return
    Y_STATS = mod.Y_STATS
    tr = terminalreporter
    tr.write_sep("-", "Y parity (max|err|/RMS against bf16(Y_ref); bar 2e-2)")
    for what, r, nf, n, xr, xb in Y_STATS:
        extra = "" if xr is None else f"  exact oracle: {xr:.3e}, {xb} beyond the bar"
        tr.write_line(f"{what[:60]:60s} {r:.3e}  {nf} one-ulp flips of {n}{extra}")
