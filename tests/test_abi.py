"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, sizes its workspace, and rejects bad arguments before
touching the GPU.  Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

import mixture_experts_ffn_route_gb300 as moe
from mixture_experts_ffn_route_gb300 import accounting

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


@pytest.fixture(scope="module")
def lib(built_lib):
    return moe.lib()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("moe_workspace_size", "moe_route", "moe_dispatch", "moe_forward",
              "moe_sync_status", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    names = header_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} is declared but not exported"
        assert n in moe.SIGNATURES, f"{n} has no binding"
    assert moe.moe_abi_version() == 1


def test_params_struct_layout():
    # nine 4-byte fields, no padding: the C struct of the header
    assert ctypes.sizeof(moe.MoeParams) == 36


def test_status_strings(lib):
    for code in range(8):
        assert moe.status_string(code) not in ("", "unknown status")
    assert moe.status_string(99) == "unknown status"


def _p(**kw):
    base = dict(T=256, H=512, E=16, k=4, I=256, has_shared=0, score_fn=0, alpha=1.0, renorm=1)
    base.update(kw)
    return moe.make_params(**base)


def test_workspace_size_and_invalid_params(lib):
    n = moe.moe_workspace_size(_p())
    A, H, I = 256 * 4, 512, 256
    assert n >= A * H * 2 + A * I * 2 + A * H * 2  # Xp, Act, Yp
    assert moe.moe_workspace_size(_p(has_shared=1)) > n
    for bad in (dict(k=17, E=32), dict(k=5, E=4), dict(H=500), dict(I=100), dict(T=-1),
                dict(E=0), dict(score_fn=3), dict(has_shared=2), dict(E=5000)):
        assert moe.moe_workspace_size(_p(**bad)) == 0, bad


def _call_forward(p, ws_ptr, ws_bytes, X=16, E_ids=16, G=16, W1=16, W2=16, Y=16):
    return moe.lib().moe_forward(ctypes.byref(p), X, E_ids, G, W1, W2, None, None, Y,
                                 ws_ptr, ws_bytes, None)


def test_argument_errors_return_before_any_launch(lib):
    p = _p()
    need = moe.moe_workspace_size(p)
    fake_ws = 1 << 20  # an aligned address that is never dereferenced
    assert _call_forward(p, None, need) == moe.MOE_ERR_WORKSPACE
    assert _call_forward(p, fake_ws, need - 1) == moe.MOE_ERR_WORKSPACE
    assert _call_forward(p, fake_ws + 8, need) == moe.MOE_ERR_WORKSPACE
    assert _call_forward(p, fake_ws, need, X=None) == moe.MOE_ERR_INVALID_ARG
    assert _call_forward(p, fake_ws, need, X=24) == moe.MOE_ERR_INVALID_ARG  # misaligned
    assert _call_forward(_p(H=96), fake_ws, need) == moe.MOE_ERR_UNSUPPORTED
    ps = _p(has_shared=1)
    assert _call_forward(ps, fake_ws, moe.moe_workspace_size(ps)) == moe.MOE_ERR_INVALID_ARG
    # T = 0 is a valid empty call and launches nothing
    p0 = _p(T=0)
    assert _call_forward(p0, fake_ws, moe.moe_workspace_size(p0)) == moe.MOE_OK

    def route(p, bias=None, tok=None, tab=None, V=0):
        return lib.moe_route(ctypes.byref(p), 16, 16, bias, tok, tab, V, 16, 16, fake_ws,
                             moe.moe_workspace_size(p), None)
    assert route(_p(score_fn=2), bias=16) == moe.MOE_ERR_INVALID_ARG     # softmax + bias
    assert route(_p(), bias=16, tok=16, tab=16, V=10) == moe.MOE_ERR_INVALID_ARG
    assert route(_p(), tok=16, tab=None, V=10) == moe.MOE_ERR_INVALID_ARG
    assert route(_p(E=12, k=2)) == moe.MOE_ERR_UNSUPPORTED               # E % 8 != 0
    assert route(_p(T=0)) == moe.MOE_OK

    def fwd_q(p, ws_bytes=None):
        n = moe.moe_workspace_size_a8w8(p) if ws_bytes is None else ws_bytes
        return lib.moe_forward_a8w8(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, fake_ws, n,
                                    None, None)
    assert fwd_q(_p(has_shared=1)) == moe.MOE_ERR_UNSUPPORTED  # the A8W8 form has no shared expert
    assert fwd_q(_p(), ws_bytes=1024) == moe.MOE_ERR_WORKSPACE
    assert fwd_q(_p(T=0)) == moe.MOE_OK

    def fwd_mx(p, fmt=0, ws_bytes=None, s1=16, wfmt=None):
        n = moe.moe_workspace_size_mx(p) if ws_bytes is None else ws_bytes
        return lib.moe_forward_mx(ctypes.byref(p), fmt, fmt if wfmt is None else wfmt, 16, 16, 16, 16, s1,
                                  16, 16, 16, fake_ws, n, None, None)
    assert fwd_mx(_p(has_shared=1)) == moe.MOE_ERR_UNSUPPORTED  # the MX form has no shared expert
    assert fwd_mx(_p(H=192)) == moe.MOE_ERR_UNSUPPORTED        # H, I multiples of 128
    assert fwd_mx(_p(I=320)) == moe.MOE_ERR_UNSUPPORTED
    assert fwd_mx(_p(), fmt=2) == moe.MOE_ERR_INVALID_ARG
    assert fwd_mx(_p(), fmt=5, wfmt=0) == moe.MOE_ERR_UNSUPPORTED   # E2M1 activations need E2M1 weights
    assert fwd_mx(_p(T=0), fmt=0, wfmt=5) == moe.MOE_OK
    assert fwd_mx(_p(T=0), fmt=5) == moe.MOE_OK
    assert fwd_mx(_p(), ws_bytes=1024) == moe.MOE_ERR_WORKSPACE
    assert fwd_mx(_p(), s1=18) == moe.MOE_ERR_INVALID_ARG      # scales 4-byte aligned
    assert fwd_mx(_p(T=0)) == moe.MOE_OK
    assert lib.moe_quantize_mx(0, 16, 4, 48, 16, 16, None) == moe.MOE_ERR_INVALID_ARG  # cols % 32
    assert lib.moe_quantize_mx(3, 16, 4, 64, 16, 16, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_mx(5, 16, 0, 64, 16, 16, None) == moe.MOE_OK
    assert lib.moe_quantize_mx(0, 16, 0, 64, 16, 16, None) == moe.MOE_OK


def test_mx_workspace_holds_codes_scales_and_fp32_rows():
    p = _p()
    T, H, I, k, E = p.T, p.H, p.I, p.k, p.E
    A = T * k
    need = T * H + T * H // 32 + A * I + A * I // 32 + A * H * 4 + 2 * A * 4
    assert moe.moe_workspace_size_mx(p) >= need


def test_accounting_pins_from_the_pages():
    MiB = 1 << 20
    # Megatron/DeepSeek-V4 page, section "一轮 V4 的数据量": 4096 token rows per
    # rank, top-6, h = 7168 -> 336 MiB of permuted rows, 63/64 of it remote
    # under EP64 = 330.75 MiB.
    v4 = accounting.dispatch_payload_bytes(4096, 7168, 6)
    assert v4 == 336 * MiB and v4 * 63 / 64 == 330.75 * MiB
    # Parallelism page, section 4.6 (通信数据量计算): B=2, S=8192, H=8192, k=2 -> 512 MiB,
    # 7/8 of it leaves the card under EP8: ~448 MiB per all-to-all.
    ep = accounting.dispatch_payload_bytes(2 * 8192, 8192, 2)
    assert ep == 512 * MiB and ep * 7 / 8 == 448 * MiB
    # Megatron/DeepSeek-V4 page, expert parameter count P_e = 3hf.
    assert accounting.expert_params(7168, 3072) == 66_060_288
    # routed weights of 6 experts x 8 layers at f = 3072, bf16: ~5.906 GiB
    gib = 6 * 8 * accounting.expert_params(7168, 3072) * 2 / (1 << 30)
    assert abs(gib - 5.906) < 1e-3


def test_accounting_counts_active_experts_once():
    counts = [0, 3, 130, 0]
    H, I = 256, 128
    assert accounting.gemm1_flops(counts, H, I) == 2 * 133 * H * 2 * I
    assert accounting.gemm1_bytes(counts, H, I) == 2 * H * 2 * I * 2 + 133 * H * 2 + 133 * I * 2
    with_shared = accounting.gemm2_bytes(counts, H, I, has_shared=1, T=10)
    assert with_shared == 3 * I * H * 2 + 143 * I * 2 + 143 * H * 4
