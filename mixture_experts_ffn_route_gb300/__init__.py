"""Python binding of ``libmoe_ffn.so``, the sm_103a routed MoE FFN forward pass.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The functions carry the C names of ``include/moe_ffn.h`` and take
torch tensors (device memory) where the C calls take device pointers.  A
missing library is an error; there is no fallback implementation.

    p  = make_params(T, H, E, k, I, has_shared=0, score_fn=SCORE_SIGMOID, alpha=1.0, renorm=1)
    ws = alloc_workspace(p, device)
    moe_route(p, X, Wg, bias, None, None, 0, E_ids, G, ws)
    moe_forward(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws)
    moe_sync_status(ws)   # raises MoEError on a device-side error
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_FFN_DEBUG_BOUNDS=1 loads the bounds-checked debug build instead (built
# by build.build(debug=True)): every index the kernels read from data is
# checked against its array and a bad one reported as MOE_ERR_BOUNDS.
LIB_PATH = os.path.join(_PKG, "libmoe_ffn_debug.so" if os.environ.get("MOE_FFN_DEBUG_BOUNDS") == "1"
                        else "libmoe_ffn.so")

SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1
SCORE_SOFTMAX = 2

MOE_MX_E4M3 = 0
MOE_MX_E5M2 = 1
MOE_MX_E2M1 = 5
MX_FORMATS = {"e4m3": MOE_MX_E4M3, "e5m2": MOE_MX_E5M2, "e2m1": MOE_MX_E2M1}

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_BAD_EXPERT_ID = 4
MOE_ERR_BAD_TOKEN_ID = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_CUDA = 7
MOE_ERR_BOUNDS = 8

# every function the C header declares, with (restype, argtypes)
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I32 = ctypes.c_int32


class MoeParams(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("has_shared", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("alpha", ctypes.c_float), ("renorm", ctypes.c_int32)]

    def __repr__(self):
        return "MoeParams(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_PP = ctypes.POINTER(MoeParams)
SIGNATURES = {
    "moe_workspace_size": (_SZ, [_PP]),
    "moe_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "moe_route": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "moe_route_logits": (ctypes.c_int, [_PP, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_timed": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                         ctypes.POINTER(ctypes.c_void_p)]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P]),
    "moe_workspace_size_a8w8": (_SZ, [_PP]),
    "moe_forward_a8w8": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    "moe_workspace_size_train": (_SZ, [_PP]),
    "moe_forward_train": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_backward": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _SZ, _P, ctypes.POINTER(ctypes.c_void_p)]),
    "moe_quantize_mx": (ctypes.c_int, [_I32, _P, _I32, _I32, _P, _P, _P]),
    "moe_workspace_size_mx": (_SZ, [_PP]),
    "moe_forward_mx": (ctypes.c_int, [_PP, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                      ctypes.POINTER(ctypes.c_void_p)]),
    "moe_sync_status": (ctypes.c_int, [_P, _SZ, _P]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [_P, _SZ, ctypes.c_uint32, _P]),
    "moe_selftest_bounds": (ctypes.c_int, [_P, _SZ, ctypes.c_int64, _P]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_abi_version": (ctypes.c_int32, []),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def lib() -> ctypes.CDLL:
    """Load the library once.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def make_params(T, H, E, k, I, has_shared=0, score_fn=SCORE_SIGMOID, alpha=1.0, renorm=1) -> MoeParams:
    return MoeParams(int(T), int(H), int(E), int(k), int(I), int(has_shared), int(score_fn),
                     float(alpha), int(renorm))


def params_from_config(cfg: dict, T: int | None = None) -> MoeParams:
    """MoeParams for a workload dict (keys T, H, E, k, I, shared, score_fn, alpha, renorm)."""
    return make_params(cfg["T"] if T is None else T, cfg["H"], cfg["E"], cfg["k"], cfg["I"],
                       cfg.get("shared", 0), cfg.get("score_fn", SCORE_SIGMOID),
                       cfg.get("alpha", 1.0), cfg.get("renorm", 1))


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(code: int, where: str) -> int:
    if code != MOE_OK:
        raise MoEError(code, where)
    return code


def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_workspace_size(p: MoeParams) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(p)))


def moe_workspace_init(ws, stream=None):
    return _check(lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def alloc_workspace(p: MoeParams, device="cuda", stream=None):
    """A zero-headed uint8 device tensor of moe_workspace_size(p) bytes."""
    import torch
    n = moe_workspace_size(p)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_route(p, X, Wg, bias, token_ids, tid2eid, V, E_ids, G, ws, stream=None):
    return _check(lib().moe_route(ctypes.byref(p), _ptr(X), _ptr(Wg), _ptr(bias), _ptr(token_ids),
                                  _ptr(tid2eid), int(V), _ptr(E_ids), _ptr(G), _ptr(ws), ws.numel(),
                                  _stream(stream)), "moe_route")


def moe_route_logits(p, X, Wg, logits, ws, stream=None):
    return _check(lib().moe_route_logits(ctypes.byref(p), _ptr(X), _ptr(Wg), _ptr(logits), _ptr(ws),
                                         ws.numel(), _stream(stream)), "moe_route_logits")


def moe_dispatch(p, E_ids, counts, offsets, perm, ws, stream=None):
    return _check(lib().moe_dispatch(ctypes.byref(p), _ptr(E_ids), _ptr(counts), _ptr(offsets),
                                     _ptr(perm), _ptr(ws), ws.numel(), _stream(stream)), "moe_dispatch")


def moe_dispatch_noalloc(p, E_ids, counts, offsets, perm, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate device
    memory where they route tokens; scratch is a fixed array in the library
    (limits T*k <= 262144, E <= 512).  Calls that overlap on the GPU race."""
    return _check(lib().moe_dispatch_noalloc(ctypes.byref(p), _ptr(E_ids), _ptr(counts), _ptr(offsets),
                                             _ptr(perm), _stream(stream)), "moe_dispatch_noalloc")


def moe_forward(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, stream=None):
    return _check(lib().moe_forward(ctypes.byref(p), _ptr(X), _ptr(E_ids), _ptr(G), _ptr(W1), _ptr(W2),
                                    _ptr(Ws1), _ptr(Ws2), _ptr(Y), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moe_forward")


def moe_forward_timed(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, stage_events, stream=None):
    """moe_forward recording five torch.cuda.Event objects (or None) at the
    stage boundaries: start, after dispatch, after Linear1, after Linear2, end.
    Each event must have been recorded once before (so that it exists)."""
    arr = (ctypes.c_void_p * 5)(*[(ev.cuda_event if ev is not None else None) for ev in stage_events])
    return _check(lib().moe_forward_timed(ctypes.byref(p), _ptr(X), _ptr(E_ids), _ptr(G), _ptr(W1),
                                          _ptr(W2), _ptr(Ws1), _ptr(Ws2), _ptr(Y), _ptr(ws), ws.numel(),
                                          _stream(stream), arr), "moe_forward_timed")


def moe_workspace_size_a8w8(p: MoeParams) -> int:
    return int(lib().moe_workspace_size_a8w8(ctypes.byref(p)))


def alloc_workspace_a8w8(p: MoeParams, device="cuda", stream=None):
    """A zero-headed uint8 device tensor of moe_workspace_size_a8w8(p) bytes."""
    import torch
    n = moe_workspace_size_a8w8(p)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size_a8w8")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_forward_a8w8(p, X, E_ids, G, W1q, S1, W2q, S2, Y, ws, stage_events=None, stream=None):
    """A8W8-INT layer forward (int8 weights with per-channel scales)."""
    arr = None
    if stage_events is not None:
        arr = (ctypes.c_void_p * 5)(*[(ev.cuda_event if ev is not None else None) for ev in stage_events])
    return _check(lib().moe_forward_a8w8(ctypes.byref(p), _ptr(X), _ptr(E_ids), _ptr(G), _ptr(W1q), _ptr(S1),
                                         _ptr(W2q), _ptr(S2), _ptr(Y), _ptr(ws), ws.numel(), _stream(stream),
                                         arr), "moe_forward_a8w8")


def moe_workspace_size_train(p: MoeParams) -> int:
    return int(lib().moe_workspace_size_train(ctypes.byref(p)))


def alloc_workspace_train(p: MoeParams, device="cuda", stream=None):
    """A zero-headed uint8 device tensor of moe_workspace_size_train(p) bytes."""
    import torch
    n = moe_workspace_size_train(p)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size_train")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_forward_train(p, X, E_ids, G, W1, W2, Ws1, Ws2, Y, ws, stream=None):
    return _check(lib().moe_forward_train(ctypes.byref(p), _ptr(X), _ptr(E_ids), _ptr(G), _ptr(W1), _ptr(W2),
                                          _ptr(Ws1), _ptr(Ws2), _ptr(Y), _ptr(ws), ws.numel(),
                                          _stream(stream)), "moe_forward_train")


def moe_backward(p, X, Wg, E_ids, G, W1, W2, Ws1, Ws2, dY, dX, dWg, dW1, dW2, dWs1, dWs2, dG, ws,
                 stage_events=None, stream=None):
    """Layer backward after moe_forward_train on the same workspace."""
    arr = None
    if stage_events is not None:
        arr = (ctypes.c_void_p * 5)(*[(ev.cuda_event if ev is not None else None) for ev in stage_events])
    return _check(lib().moe_backward(ctypes.byref(p), _ptr(X), _ptr(Wg), _ptr(E_ids), _ptr(G), _ptr(W1),
                                     _ptr(W2), _ptr(Ws1), _ptr(Ws2), _ptr(dY), _ptr(dX), _ptr(dWg), _ptr(dW1),
                                     _ptr(dW2), _ptr(dWs1), _ptr(dWs2), _ptr(dG), _ptr(ws), ws.numel(),
                                     _stream(stream), arr), "moe_backward")


def moe_quantize_mx(fmt: int, X, Q, S, stream=None):
    """Q_MX of the bf16 rows of X [rows, cols] into codes Q (E2M1: packed,
    [rows, cols / 2]) and E8M0 scales S."""
    rows, cols = X.shape
    return _check(lib().moe_quantize_mx(int(fmt), _ptr(X), int(rows), int(cols), _ptr(Q), _ptr(S),
                                        _stream(stream)), "moe_quantize_mx")


def moe_workspace_size_mx(p: MoeParams) -> int:
    return int(lib().moe_workspace_size_mx(ctypes.byref(p)))


def alloc_workspace_mx(p: MoeParams, device="cuda", stream=None):
    """A zero-headed uint8 device tensor of moe_workspace_size_mx(p) bytes."""
    import torch
    n = moe_workspace_size_mx(p)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size_mx")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_forward_mx(p, fmt: int, X, E_ids, G, W1, S1, W2, S2, Y, ws, stage_events=None, stream=None,
                   wfmt: int | None = None):
    """MX (FP8 / FP4 codes + E8M0 group scales) layer forward; fmt is the
    activations' element format, wfmt the weights' (default: fmt)."""
    arr = None
    if stage_events is not None:
        arr = (ctypes.c_void_p * 5)(*[(ev.cuda_event if ev is not None else None) for ev in stage_events])
    wf = int(fmt) if wfmt is None else int(wfmt)
    return _check(lib().moe_forward_mx(ctypes.byref(p), int(fmt), wf, _ptr(X), _ptr(E_ids), _ptr(G), _ptr(W1),
                                       _ptr(S1), _ptr(W2), _ptr(S2), _ptr(Y), _ptr(ws), ws.numel(),
                                       _stream(stream), arr), "moe_forward_mx")


def moe_selftest_wait_timeout(ws, limit_us: int, stream=None):
    return _check(lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)),
                  "moe_selftest_wait_timeout")


def moe_selftest_bounds(ws, index: int, stream=None) -> int:
    """Status of the bounds self-test launch (MOE_ERR_UNSUPPORTED from the
    release library); the check's outcome comes from moe_sync_status."""
    return int(lib().moe_selftest_bounds(_ptr(ws), ws.numel(), int(index), _stream(stream)))


def moe_sync_status(ws, stream=None, raise_on_error=True) -> int:
    code = lib().moe_sync_status(_ptr(ws), ws.numel(), _stream(stream))
    if raise_on_error:
        _check(code, "moe_sync_status")
    return code
