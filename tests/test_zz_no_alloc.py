"""moe_dispatch_noalloc, the dispatch for callers that cannot allocate device
memory where they route tokens (their memory belongs to another allocator, or
a cudaMalloc that may synchronise the device is not allowed on their path).
Its scratch is a fixed array inside the library, so the test checks that
calls in a row, on different inputs, each match moe_dispatch and the CPU
oracle's dispatch exactly (the dispatch is integer work: bit-exact), one of
them with ids outside [0, E), which are dropped and show as offsets[E] < T k."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle

DEV = torch.device("cuda:0")


def _ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1)[:, :k].astype(np.int32)


def _with_workspace(p, E_ids):
    ws = moe.alloc_workspace(p, DEV)
    c = torch.empty(p.E, dtype=torch.int32, device=DEV)
    o = torch.empty(p.E + 1, dtype=torch.int32, device=DEV)
    m = torch.empty(p.T * p.k, dtype=torch.int32, device=DEV)
    moe.moe_dispatch(p, E_ids, c, o, m, ws)
    moe.moe_sync_status(ws)
    return c.cpu().numpy(), o.cpu().numpy(), m.cpu().numpy()


def _without_workspace(p, E_ids):
    c = torch.full((p.E,), -9, dtype=torch.int32, device=DEV)
    o = torch.full((p.E + 1,), -9, dtype=torch.int32, device=DEV)
    m = torch.full((p.T * p.k,), -9, dtype=torch.int32, device=DEV)
    moe.moe_dispatch_noalloc(p, E_ids, c, o, m)
    torch.cuda.synchronize()
    return c.cpu().numpy(), o.cpu().numpy(), m.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_dispatch_matches_the_workspace_dispatch_and_the_oracle(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)
    # first call: V4-Pro-like routing (E 384, top-6, 4096 tokens: several chunks);
    # second call: a different, smaller problem whose results must not carry
    # anything over from the first; third: ids outside [0, E) in two chunks
    cases = [(4096, 384, 6, 1, False), (1000, 40, 3, 2, False), (5000, 24, 3, 3, True)]
    for T, E, k, seed, bad in cases:
        p = moe.make_params(T, 64, E, k, 64)
        ids = _ids(T, E, k, seed)
        if bad:
            ids[7, 1] = -1
            ids[4100, 0] = E
            ids[4999, 2] = 10 ** 6
        E_ids = torch.from_numpy(ids).to(DEV)
        got = _without_workspace(p, E_ids)
        rc, ro, rp, _ = oracle.dispatch(ids, E)
        n = int(ro[-1])
        np.testing.assert_array_equal(got[0], rc)
        np.testing.assert_array_equal(got[1], ro)
        np.testing.assert_array_equal(got[2][:n], rp)
        assert (got[2][n:] == -9).all()  # entries past offsets[E] are left untouched
        assert n == T * k - (3 if bad else 0)
        if not bad:
            want = _with_workspace(p, E_ids)
            for w, g in zip(want, got):
                np.testing.assert_array_equal(g, w)


def test_noalloc_dispatch_rejects_sizes_past_its_limits(built_lib):
    f = moe.lib().moe_dispatch_noalloc
    too_many_tokens = moe.make_params(262144 // 6 + 1, 64, 384, 6, 64)
    too_many_experts = moe.make_params(16, 64, 513, 2, 64)
    for p in (too_many_tokens, too_many_experts):
        assert f(ctypes.byref(p), 16, 16, 16, 16, None) == moe.MOE_ERR_UNSUPPORTED
