"""Parity of the CUDA library (through its C ABI) with the CPU oracle.

Expert ids, counts, offsets and the permutation must match bit for bit; gates
within 2e-4 relative; Y within max|err| <= 2e-2 * RMS(Y_ref), Y_ref the oracle
rounded once to bf16 (tests/_gpu.py).  Small workloads are compared element by
element; the full-size workloads compare routing and dispatch on every token
and Y element by element on a seeded token set that reaches every routed
expert, plus random tokens."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle
import synth
from _gpu import (DEV, bf, check_gates, check_y, check_y_layer, host_bits, mixed_load_ids, params, run_forward,
                  run_route, to_device, to_host)

pytestmark = pytest.mark.gpu

SMALL_ROUTED = ["c1", "c3s", "c3s_sp", "c4s", "c5s"]
SMALL_ALL = ["c1", "c2s", "c3s", "c3s_sp", "c4s", "c5s"]


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


def oracle_route(h):
    c = h["cfg"]
    if c["routing"] == "hash":
        return oracle.route_hash(h["X"], h["Wg"], h["token_ids"], h["tid2eid"], c["score_fn"],
                                 c["alpha"], c["renorm"])
    return oracle.route(h["X"], h["Wg"], h["bias"], c["score_fn"], c["k"], c["alpha"], c["renorm"])


def host_inputs(name, **kw):
    h = synth.make_inputs(name, **kw)
    return h, to_device(h)


# ---------------------------------------------------------------------- router
@pytest.mark.parametrize("name", ["c1", "c3s", "c3s_sp", "c5s"])
def test_router_scores_within_decision_band(name):
    h, dd = host_inputs(name)
    c = h["cfg"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    L = torch.empty((c["T"], c["E"]), dtype=torch.float32, device=DEV)
    moe.moe_route_logits(p, dd["X"], dd["Wg"], L, ws)
    moe.moe_sync_status(ws)
    l32 = L.cpu().numpy().astype(np.float64)
    l64 = oracle.router_logits(h["X"], h["Wg"])
    if c["score_fn"] == oracle.SCORE_SOFTMAX:
        # selection on the logit, band 1e-3 * max(1, |l|): keep the error below a quarter
        assert (np.abs(l32 - l64) / np.maximum(1.0, np.abs(l64))).max() < 2.5e-4
    else:
        s32 = oracle.affinity(l32, c["score_fn"])
        s64 = oracle.affinity(l64, c["score_fn"])
        assert np.abs(s32 - s64).max() < 5e-5  # a quarter of the 2e-4 score band


@pytest.mark.parametrize("name", ["c3", "c3_sp", "c5"])
def test_router_scores_within_decision_band_full_size(name):
    dd = synth.make_inputs_torch(name, device=DEV, weights=False)
    c = dd["cfg"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    L = torch.empty((c["T"], c["E"]), dtype=torch.float32, device=DEV)
    moe.moe_route_logits(p, dd["X"], dd["Wg"], L, ws)
    moe.moe_sync_status(ws)
    l32 = L.cpu().numpy().astype(np.float64)
    l64 = oracle.router_logits(host_bits(dd["X"]), host_bits(dd["Wg"]))
    if c["score_fn"] == oracle.SCORE_SOFTMAX:
        assert (np.abs(l32 - l64) / np.maximum(1.0, np.abs(l64))).max() < 2.5e-4
    else:
        s32 = oracle.affinity(l32, c["score_fn"])
        s64 = oracle.affinity(l64, c["score_fn"])
        assert np.abs(s32 - s64).max() < 5e-5


@pytest.mark.parametrize("name", SMALL_ROUTED)
def test_route_matches_oracle(name):
    h, dd = host_inputs(name)
    p = params(h["cfg"])
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref, _ = oracle_route(h)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_gates(G, G_ref, name)


# shapes that take the fused router's split of H over clusters of 1, 2, 4 and
# 8 CTAs, one or two MMAs per k-step (E <= 256 or up to 384) and padded
# expert columns (E not a multiple of 64)
ROUTER_SHAPES = [
    dict(T=300, H=4096, E=64, k=4, I=64, bias=True),                          # 8 CTAs per tile
    dict(T=256, H=1024, E=384, k=6, I=64, bias=True, alpha=2.5),              # 2, two MMAs
    dict(T=200, H=2048, E=128, k=8, I=64, score="softmax", renorm=0),         # 4
    dict(T=130, H=512, E=320, k=3, I=64, score="sqrt_softplus", bias=True),   # 1, N = 256 + 64
    dict(T=77, H=1024, E=40, k=5, I=64, bias=True),                           # 2, padded columns
    # more than 384 experts: the general path (fp32 logits, selection kernel)
    dict(T=300, H=512, E=512, k=8, I=64, bias=True),
    dict(T=200, H=256, E=448, k=4, I=64, score="softmax", renorm=0),
]


@pytest.mark.parametrize("shape", ROUTER_SHAPES, ids=lambda s: "T{T}_H{H}_E{E}_k{k}".format(**s))
def test_route_split_over_clusters(shape):
    h, dd = host_inputs(dict(shape), seed=31)
    c = h["cfg"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref, l64 = oracle_route(h)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_gates(G, G_ref, str(shape))
    L = torch.empty((c["T"], c["E"]), dtype=torch.float32, device=DEV)
    moe.moe_route_logits(p, dd["X"], dd["Wg"], L, ws)
    moe.moe_sync_status(ws)
    l32 = L.cpu().numpy().astype(np.float64)
    if c["score_fn"] == oracle.SCORE_SOFTMAX:
        assert (np.abs(l32 - l64) / np.maximum(1.0, np.abs(l64))).max() < 2.5e-4
    else:
        assert np.abs(oracle.affinity(l32, c["score_fn"]) - oracle.affinity(l64, c["score_fn"])).max() < 5e-5


def test_route_equal_scores_go_to_the_lower_id():
    rng = np.random.default_rng(11)
    T, H, E, k = 64, 128, 16, 4
    X = synth.bf16_bits_from_f32(rng.standard_normal((T, H)))
    Wg = rng.standard_normal((H, E)).astype(np.float32) / 11
    Wg[:, 9] = Wg[:, 2]
    Wg[:, 13] = Wg[:, 2]
    bias = np.zeros(E, np.float32)
    bias[[2, 9, 13]] = 0.75  # always selected, always tied
    Wg = synth.bf16_bits_from_f32(Wg)
    p = moe.make_params(T, H, E, k, 64)
    ws = moe.alloc_workspace(p, DEV)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    moe.moe_route(p, bf(X), bf(Wg), torch.from_numpy(bias).to(DEV), None, None, 0, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids = E_ids.cpu().numpy()
    assert (ids[:, :3] == [2, 9, 13]).all()
    ids_ref, G_ref, _ = oracle.route(X, Wg, bias, 0, k, 1.0, 1)
    assert np.array_equal(ids, ids_ref)
    check_gates(G, G_ref)


@pytest.mark.parametrize("E,k", [(384, 8), (8, 8), (64, 16)])
def test_route_one_lane_holds_the_top_entries(E, k):
    # The fused router's lane l scores the columns 4c .. 4c + 3 of chunks
    # c = l, l + 32, l + 64 and keeps its best three.  A large bias on lane
    # 0's columns puts the whole top-(k+1) there, so that lane gives up all
    # three and rescans its columns (twice at E = 384), with two of its
    # columns exactly tied (the lower id first).  E = k = 8: every column is
    # taken, four from each of two lanes.
    rng = np.random.default_rng(17)
    T, H = 160, 256
    X = synth.bf16_bits_from_f32(rng.standard_normal((T, H)))
    Wg = (rng.standard_normal((H, E)) / 16).astype(np.float32)
    lane0 = [4 * c + q for c in range(0, (E + 3) // 4, 32) for q in range(4) if 4 * c + q < E]
    bias = np.zeros(E, np.float32)
    bias[lane0] = 2.0
    if len(lane0) > 5:
        Wg[:, lane0[5]] = Wg[:, lane0[1]]  # an exact tie inside the lane
    Wg = synth.bf16_bits_from_f32(Wg)
    p = moe.make_params(T, H, E, k, 64)
    ws = moe.alloc_workspace(p, DEV)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    moe.moe_route(p, bf(X), bf(Wg), torch.from_numpy(bias).to(DEV), None, None, 0, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids = E_ids.cpu().numpy()
    ids_ref, G_ref, _ = oracle.route(X, Wg, bias, 0, k, 1.0, 1)
    assert np.array_equal(ids, ids_ref)
    assert np.isin(ids[:, :min(k, len(lane0))], lane0).all()
    check_gates(G, G_ref)


def test_hash_route_general_path():
    # 512 experts take the general router (fp32 logits, then the selection
    # kernel's table lookup): ids exactly the table's, gates from the logits
    h, dd = host_inputs(dict(T=150, H=256, E=512, k=6, I=64, routing="hash", V=1000), seed=37)
    p = params(h["cfg"])
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref, _ = oracle_route(h)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_gates(G, G_ref, "hash, 512 experts")


@pytest.mark.parametrize("T,E", [(2048, 16), (5000, 16), (2048, 512)])
def test_route_many_close_tokens(T, E):
    # Every token ties (three identical, always-selected columns), so every
    # token is listed for the float64 re-decision: more tokens than its
    # blocks, each block taking several in turn (and, at T = 5000, the fused
    # router's list spread over 40 row tiles' segments; at E = 512 the general
    # path's single list, whose counters the re-decision zeroes for the next
    # call).
    rng = np.random.default_rng(29)
    H, k = 128, 4
    X = synth.bf16_bits_from_f32(rng.standard_normal((T, H)))
    Wg = rng.standard_normal((H, E)).astype(np.float32) / 11
    Wg[:, 9] = Wg[:, 2]
    Wg[:, 13] = Wg[:, 2]
    bias = np.zeros(E, np.float32)
    bias[[2, 9, 13]] = 2.0  # above every other score (sigmoid < 1)
    Wg = synth.bf16_bits_from_f32(Wg)
    p = moe.make_params(T, H, E, k, 64)
    ws = moe.alloc_workspace(p, DEV)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    for _ in range(2):  # the lists are rebuilt on every call
        moe.moe_route(p, bf(X), bf(Wg), torch.from_numpy(bias).to(DEV), None, None, 0, E_ids, G, ws)
        moe.moe_sync_status(ws)
        ids = E_ids.cpu().numpy()
        assert (ids[:, :3] == [2, 9, 13]).all()
        ids_ref, G_ref, _ = oracle.route(X, Wg, bias, 0, k, 1.0, 1)
        assert np.array_equal(ids, ids_ref)
        check_gates(G, G_ref)


def test_route_large_scores_a_few_1e4_apart():
    # The fused router's keys keep 23 bits of the biased score (the low 9
    # hold the id): at scores near 9 they resolve ~5e-4, coarser than the
    # decision band of 2e-4.  Experts 3 and 5 carry a bias of 8.5 and differ
    # by 2.4e-4 in score (one bf16 step of Wg[0] times X[:, 0] = +-1, through
    # the sigmoid's slope 1/4), in an order that alternates by token: the
    # pair must still be decided exactly.
    rng = np.random.default_rng(19)
    T, H, E, k = 96, 256, 32, 4
    X = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    X[:, 0] = np.where(np.arange(T) % 2 == 0, 1.0, -1.0)
    Wg = (rng.standard_normal((H, E)) / 16).astype(np.float32)
    Wg[:, 5] = Wg[:, 3]
    Wg[0, 3] = 2.0 ** -4
    Wg[0, 5] = 2.0 ** -4 + 2.0 ** -10
    Xb, Wgb = synth.bf16_bits_from_f32(X), synth.bf16_bits_from_f32(Wg)
    bias = np.zeros(E, np.float32)
    bias[[3, 5]] = 8.5
    p = moe.make_params(T, H, E, k, 64)
    ws = moe.alloc_workspace(p, DEV)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    moe.moe_route(p, bf(Xb), bf(Wgb), torch.from_numpy(bias).to(DEV), None, None, 0, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids = E_ids.cpu().numpy()
    ids_ref, G_ref, _ = oracle.route(Xb, Wgb, bias, 0, k, 1.0, 1)
    assert np.array_equal(ids, ids_ref)
    assert (ids[0::2, :2] == [5, 3]).all() and (ids[1::2, :2] == [3, 5]).all()
    check_gates(G, G_ref)


@pytest.mark.parametrize("score", [0, 1, 2])
def test_route_near_ties_are_decided_exactly(score):
    # experts 3 and 5 differ only in Wg[0, :], by one bf16 step of 2^-11, and
    # X[:, 0] = +-2^-20: their logits differ by exactly 2^-31, far below what an
    # fp32 accumulation resolves, so the order comes from the re-decision.
    rng = np.random.default_rng(13)
    T, H, E, k = 64, 256, 16, 4
    X = rng.standard_normal((T, H)).astype(np.float32)
    X[:, 0] = np.where(np.arange(T) % 2 == 0, 2.0 ** -20, -(2.0 ** -20))
    Wg = (rng.standard_normal((H, E)) / 16).astype(np.float32)
    Wg[:, 5] = Wg[:, 3]
    Wg[0, 3] = 2.0 ** -4
    Wg[0, 5] = 2.0 ** -4 + 2.0 ** -11
    Xb, Wgb = synth.bf16_bits_from_f32(X), synth.bf16_bits_from_f32(Wg)
    bias = None
    if score != oracle.SCORE_SOFTMAX:
        bias = np.zeros(E, np.float32)
        bias[[3, 5]] = 5.0  # always the first two
    else:
        # softmax selects on the logit: make columns 3 and 5 large (and equal
        # apart from row 0) against positive token rows
        Xb = synth.bf16_bits_from_f32(np.concatenate([X[:, :1], np.abs(X[:, 1:])], 1))
        Wgb[1:, 3] = synth.bf16_bits_from_f32(np.full(H - 1, 0.25, np.float32))
        Wgb[1:, 5] = Wgb[1:, 3]
    p = moe.make_params(T, H, E, k, 64, score_fn=score, renorm=0 if score == 2 else 1)
    ws = moe.alloc_workspace(p, DEV)
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    b = torch.from_numpy(bias).to(DEV) if bias is not None else None
    moe.moe_route(p, bf(Xb), bf(Wgb), b, None, None, 0, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref, l64 = oracle.route(Xb, Wgb, bias, score, k, 1.0, p.renorm)
    assert (np.abs(l64[:, 5] - l64[:, 3]) == 2.0 ** -31).all()
    ids = E_ids.cpu().numpy()
    want = np.where((np.arange(T) % 2 == 0)[:, None], [5, 3], [3, 5])
    assert (ids[:, :2] == want).all()
    assert np.array_equal(ids, ids_ref)


# ---------------------------------------------------------------------- dispatch
def _dispatch_gpu(p, E_ids):
    ws = moe.alloc_workspace(p, DEV)
    counts = torch.full((p.E,), -5, dtype=torch.int32, device=DEV)
    offsets = torch.full((p.E + 1,), -5, dtype=torch.int32, device=DEV)
    perm = torch.full((p.T * p.k,), -5, dtype=torch.int32, device=DEV)
    moe.moe_dispatch(p, E_ids, counts, offsets, perm, ws)
    code = moe.moe_sync_status(ws, raise_on_error=False)
    return code, counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()


@pytest.mark.parametrize("name", ["c2s", "c3s", "c4s", "c5s"])
def test_dispatch_matches_oracle(name):
    h, dd = host_inputs(name)
    c = h["cfg"]
    ids = h["E_ids"] if c["routing"] == "given" else oracle_route(h)[0]
    code, counts, offsets, perm = _dispatch_gpu(params(c), torch.from_numpy(ids).to(DEV))
    assert code == moe.MOE_OK
    rc, ro, rp, _ = oracle.dispatch(ids, c["E"])
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro)
    assert np.array_equal(perm, rp)


def test_dispatch_drops_bad_ids_and_reports_them():
    rng = np.random.default_rng(12)
    T, E, k = 5000, 24, 3  # two chunks of assignments
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[7, 1] = -1
    ids[4100, 0] = E
    ids[4999, 2] = 10 ** 6
    p = moe.make_params(T, 64, E, k, 64)
    code, counts, offsets, perm = _dispatch_gpu(p, torch.from_numpy(ids).to(DEV))
    assert code == moe.MOE_ERR_BAD_EXPERT_ID
    rc, ro, rp, _ = oracle.dispatch(ids, E)
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro)
    assert np.array_equal(perm[:len(rp)], rp)


# ---------------------------------------------------------------------- forward
def _reference_ids(h):
    c = h["cfg"]
    if c["routing"] == "given":
        return h["E_ids"], h["G"].astype(np.float64)
    ids, G, _ = oracle_route(h)
    return ids, G


@pytest.mark.parametrize("name", SMALL_ALL)
def test_forward_matches_oracle(name):
    h, dd = host_inputs(name)
    c = h["cfg"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    ids_ref, G_ref = _reference_ids(h)
    if c["routing"] == "given":
        E_ids, G = dd["E_ids"], dd["G"]
    else:
        E_ids, G = run_route(p, dd, ws)
    Y = run_forward(p, dd, E_ids, G, ws)
    moe.moe_sync_status(ws)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_y_layer(Y, name, h["X"], ids_ref, G_ref, h["W1"], h["W2"], h["Ws1"], h["Ws2"])


EDGE = [
    dict(T=1, H=64, E=1, k=1, I=64),
    dict(T=3, H=128, E=2, k=2, I=64),
    dict(T=17, H=64, E=5, k=5, I=128, shared=1),
    dict(T=129, H=192, E=3, k=1, I=64),
    dict(T=40, H=256, E=40, k=2, I=64),
    dict(T=600, H=128, E=6, k=1, I=192, hot=True),
    dict(T=260, H=320, E=9, k=3, I=448, shared=1),
    dict(T=700, H=192, E=12, k=2, I=320, shared=1, mixed=True),
    # experts of several hundred rows (every group dense in the tile order),
    # partial last row tiles and partial column tiles
    dict(T=700, H=192, E=2, k=2, I=320, shared=1),
    dict(T=520, H=256, E=4, k=2, I=128),
    dict(T=300, H=128, E=1, k=1, I=64),
]


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "T{T}_H{H}_E{E}_k{k}_I{I}".format(**s))
def test_forward_edge_shapes(shape):
    shape = dict(shape)
    hot = shape.pop("hot", False)
    mixed = shape.pop("mixed", False)
    h = synth.make_inputs(dict(shape, routing="given", score="softmax", renorm=0), seed=99)
    if hot:
        h["E_ids"][:] = 0  # every token to expert 0: several 128-row tiles, other experts empty
    if mixed:
        h["E_ids"][:] = mixed_load_ids(shape["T"], shape["E"])
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    Y = run_forward(p, dd, dd["E_ids"], dd["G"], ws)
    moe.moe_sync_status(ws)
    check_y_layer(Y, str(shape), h["X"], h["E_ids"], h["G"].astype(np.float64), h["W1"], h["W2"],
                              h["Ws1"], h["Ws2"])


@pytest.mark.parametrize("k", [1, 2])
def test_forward_groups_at_the_m64_boundary(k):
    """Expert groups of 63, 64, 65, 128 and 129 rows: the grouped GEMMs run a
    tile of at most 64 rows as an M = 64 MMA (its rows in the first 16 lanes
    of each TMEM lane quarter) and a longer one as M = 128, so the groups
    straddle that switch and the 128-row tile edge.  k = 1 takes the top-1
    combine in Linear2's epilogue, k = 2 the combine kernel."""
    sizes = [63, 64, 65, 128, 129]
    T = sum(sizes)
    h = synth.make_inputs(dict(T=T, H=192, E=len(sizes), k=k, I=128, routing="given", score="softmax",
                               renorm=0), seed=23)
    first = np.repeat(np.arange(len(sizes)), sizes)
    ids = first[:, None] if k == 1 else np.stack([first, (first + 2) % len(sizes)], axis=1)
    h["E_ids"] = np.ascontiguousarray(ids, dtype=np.int32)
    h["G"] = np.random.default_rng(24).uniform(0.25, 1.0, size=(T, k)).astype(np.float32)
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    Y = run_forward(p, dd, dd["E_ids"], dd["G"], ws)
    moe.moe_sync_status(ws)
    check_y_layer(Y, f"M=64 boundary groups, k={k}", h["X"], h["E_ids"], h["G"].astype(np.float64),
                  h["W1"], h["W2"])


@pytest.mark.parametrize("T", [1, 64, 65, 129, 192, 193])
def test_route_ragged_row_tiles(T):
    """The router on T % 128 in {1, 64, 65} (tiles of one row, exactly 64 rows
    and 65 rows) and T below one tile."""
    h, dd = host_inputs("c1", T=T)
    p = params(h["cfg"])
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref, _ = oracle_route(h)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_gates(G, G_ref, f"c1 T={T}")


def test_routed_forward_dense_experts():
    """The c5s layer with T = 1040 (260 routed rows per expert on average: every
    expert spans several 128-row tiles): routing and Y."""
    h = synth.make_inputs("c5s", T=1040)
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    Y = run_forward(p, dd, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref = _reference_ids(h)
    assert np.array_equal(E_ids.cpu().numpy(), ids_ref)
    check_y_layer(Y, "c5s T=1040", h["X"], ids_ref, G_ref, h["W1"], h["W2"], h["Ws1"], h["Ws2"])


def test_forward_with_no_tokens_writes_nothing():
    h, dd = host_inputs("c3s")
    p = params(h["cfg"], T=0)
    ws = moe.alloc_workspace(p, DEV)
    Y = torch.full((4, h["cfg"]["H"]), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(p, dd["X"], dd["X"], dd["X"], dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], Y, ws)
    moe.moe_sync_status(ws)
    assert (Y == 3.0).all()


def test_bad_expert_ids_are_skipped_and_reported():
    h, dd = host_inputs("c2s")
    c = h["cfg"]
    ids = h["E_ids"].copy()
    ids[3, 0] = -1
    ids[100, 2] = c["E"] + 5
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    Y = run_forward(p, dd, torch.from_numpy(ids).to(DEV), dd["G"], ws)
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_ERR_BAD_EXPERT_ID
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_OK  # cleared
    check_y_layer(Y, "dropped assignments", h["X"], ids, h["G"].astype(np.float64), h["W1"], h["W2"])


def test_top1_combine_in_the_linear2_epilogue():
    """k = 1 without a shared expert: Linear2's epilogue writes each gate-scaled
    row straight into its token's row of Y (no combine pass); a token whose one
    id is bad gets a zero row, as the combine would give it."""
    h = synth.make_inputs(dict(T=300, H=192, E=5, k=1, I=128, routing="given", score="softmax", renorm=0),
                          seed=7)
    c = h["cfg"]
    # a softmax over one logit is 1: draw gates that make the scaling visible
    h["G"] = np.random.default_rng(11).uniform(0.25, 2.0, size=h["G"].shape).astype(np.float32)
    ids = h["E_ids"].copy()
    bad = [0, 17, 299]
    ids[bad, 0] = [-1, c["E"], 2 * c["E"]]
    dd = to_device(h)
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    Y = torch.full((c["T"], c["H"]), float("nan"), dtype=torch.bfloat16, device=DEV)
    run_forward(p, dd, torch.from_numpy(ids).to(DEV), dd["G"], ws, Y=Y)
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_ERR_BAD_EXPERT_ID
    assert torch.equal(Y[bad].float(), torch.zeros((len(bad), c["H"]), device=DEV))
    check_y_layer(Y, "top-1, fused combine", h["X"], ids, h["G"].astype(np.float64), h["W1"], h["W2"])


def test_bad_hash_token_ids_are_reported():
    h, dd = host_inputs("c4s")
    c = h["cfg"]
    tok = h["token_ids"].copy()
    tok[5] = c["V"]
    tok[6] = -3
    dd["token_ids"] = torch.from_numpy(tok).to(DEV)
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_ERR_BAD_TOKEN_ID
    ids = E_ids.cpu().numpy()
    assert (ids[5] == -1).all() and (ids[6] == -1).all() and (G.cpu().numpy()[5:7] == 0).all()
    good = np.ones(c["T"], bool)
    good[5:7] = False
    ids_ref = h["tid2eid"][h["token_ids"]]
    assert np.array_equal(ids[good], ids_ref[good])


def test_poisoned_workspace_does_not_leak_into_the_output():
    h, dd = host_inputs("c3s")
    c = h["cfg"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    ws.fill_(0xFF)  # NaN patterns in every bf16 and fp32 scratch buffer
    moe.moe_workspace_init(ws)
    E_ids, G = run_route(p, dd, ws)
    Y = run_forward(p, dd, E_ids, G, ws)
    moe.moe_sync_status(ws)
    ids_ref, G_ref = _reference_ids(h)
    check_y_layer(Y, "poisoned workspace", h["X"], ids_ref, G_ref, h["W1"], h["W2"], h["Ws1"], h["Ws2"])


def test_forward_is_deterministic():
    h, dd = host_inputs("c5s")
    p = params(h["cfg"])
    ws = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws)
    Y1 = run_forward(p, dd, E_ids, G, ws).clone()
    Y2 = run_forward(p, dd, E_ids, G, ws)
    moe.moe_sync_status(ws)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


def test_device_wait_limit_reports_timeout():
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    moe.moe_workspace_init(ws)
    moe.moe_selftest_wait_timeout(ws, 20000)  # 20 ms
    assert moe.moe_sync_status(ws, raise_on_error=False) == moe.MOE_ERR_TIMEOUT
    # the context is still usable
    h, dd = host_inputs("c1")
    p = params(h["cfg"])
    ws2 = moe.alloc_workspace(p, DEV)
    E_ids, _ = run_route(p, dd, ws2)
    moe.moe_sync_status(ws2)
    assert np.array_equal(E_ids.cpu().numpy(), oracle_route(h)[0])


# ---------------------------------------------------------------------- full size
# tokens whose Y is compared: (tokens chosen to reach every routed expert, at
# least this many in all, then this many more random tokens)
FULL = {"c2": (512, 0), "c3": (512, 256), "c4": (512, 256), "c5": (256, 0), "c3_sp": (512, 256),
        "c3_f3072": (256, 0), "c5x": (128, 64), "c5x_sh": (128, 64)}


def host_expert_weights(w):
    """Expert e's weights as float64 on the host (an exact widening of the
    bf16 values), fetched one expert at a time."""
    return lambda e: w[e].cpu().to(torch.float64).numpy()


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workload(name):
    dd = synth.make_inputs_torch(name, device=DEV)
    c = dd["cfg"]
    T, k, E = c["T"], c["k"], c["E"]
    p = params(c)
    ws = moe.alloc_workspace(p, DEV)
    hX = host_bits(dd["X"])
    # routing on every token
    if c["routing"] == "given":
        E_ids, G = dd["E_ids"], dd["G"]
        ids_ref, G_ref = E_ids.cpu().numpy(), G.cpu().numpy().astype(np.float64)
    else:
        E_ids, G = run_route(p, dd, ws)
        moe.moe_sync_status(ws)
        hWg = host_bits(dd["Wg"])
        if c["routing"] == "hash":
            ids_ref, G_ref, l64 = oracle.route_hash(hX, hWg, dd["token_ids"].cpu().numpy(),
                                                    dd["tid2eid"].cpu().numpy(), c["score_fn"],
                                                    c["alpha"], c["renorm"])
        else:
            bias = dd["bias"].cpu().numpy() if dd["bias"] is not None else None
            ids_ref, G_ref, l64 = oracle.route(hX, hWg, bias, c["score_fn"], k, c["alpha"], c["renorm"])
        assert np.array_equal(E_ids.cpu().numpy(), ids_ref), "expert ids differ"
        check_gates(G, G_ref, name)
    # dispatch on every assignment
    code, counts, offsets, perm = _dispatch_gpu(p, E_ids)
    assert code == moe.MOE_OK
    rc, ro, rp, _ = oracle.dispatch(ids_ref, E)
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro) and np.array_equal(perm, rp)
    # Y element by element on tokens that reach every routed expert
    Y = run_forward(p, dd, E_ids, G, ws)
    Y2 = run_forward(p, dd, E_ids, G, ws, Y=torch.empty_like(Y))
    moe.moe_sync_status(ws)
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16)), "not deterministic"
    n_min, n_extra = FULL[name]
    rows = synth.covering_tokens(ids_ref, E, n_min, n_extra)
    assert np.unique(ids_ref[rows]).size == np.unique(ids_ref).size, "an expert is not reached"
    Ws1 = host_bits(dd["Ws1"]) if dd["Ws1"] is not None else None
    Ws2 = host_bits(dd["Ws2"]) if dd["Ws2"] is not None else None
    Y_ref = oracle.forward_tokens(rows, hX[rows], ids_ref[rows], G_ref[rows], host_expert_weights(dd["W1"]),
                                  host_expert_weights(dd["W2"]), Ws1, Ws2, act_round_bf16=True, E=E)
    check_y(Y[torch.from_numpy(rows).to(DEV)], Y_ref, f"{name} full size, {rows.size} tokens")
