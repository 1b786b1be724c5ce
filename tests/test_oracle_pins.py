"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, the pages' worked split example, brute-force loops on tiny
inputs, reductions to a dense SwiGLU FFN and to library routines, and the
invariants the pages state (k ids per token, sum of counts = T*k, the shared
expert alone when every gate is zero)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth


def _bits(x):
    return synth.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------------ bf16 numbers
def test_round_to_bf16_ties_even():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 keeps 7 fraction bits
    cases = {one + ulp / 2: one,                    # tie, 1.0 is even
             one + 1.5 * ulp: one + 2 * ulp,        # tie, rounds up to even
             one + 0.49 * ulp: one,
             one + 0.51 * ulp: one + ulp,
             -(one + 1.5 * ulp): -(one + 2 * ulp)}
    for x, want in cases.items():
        assert oracle.round_to_bf16(np.array([x]))[0] == want


def test_bf16_bits_match_torch_rounding():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1, 1e3], 20000)).astype(np.float32)
    ours = oracle.f64_to_bf16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.bf16_to_f64(ref)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


# ------------------------------------------------------------------ affinities and gates
def test_affinity_closed_forms():
    l = np.array([[math.log(3.0), -math.log(3.0), 0.0]])
    np.testing.assert_allclose(oracle.affinity(l, oracle.SCORE_SIGMOID), [[0.75, 0.25, 0.5]], rtol=0, atol=1e-15)
    # softplus(log(e^c - 1)) = c, so sqrt gives sqrt(c)
    l = np.array([[math.log(math.e - 1.0), math.log(math.e ** 4 - 1.0), 0.0, -800.0, 800.0]])
    np.testing.assert_allclose(oracle.affinity(l, oracle.SCORE_SQRT_SOFTPLUS),
                               [[1.0, 2.0, math.sqrt(math.log(2.0)), 0.0, math.sqrt(800.0)]],
                               rtol=1e-14, atol=1e-300)
    l = np.array([[math.log(4.0), math.log(2.0), 0.0, 0.0]])
    np.testing.assert_allclose(oracle.affinity(l, oracle.SCORE_SOFTMAX), [[0.5, 0.25, 0.125, 0.125]],
                               rtol=1e-15)


@pytest.mark.parametrize("score,logits,want_ids,want_g", [
    (oracle.SCORE_SIGMOID, [-30.0, math.log(3.0), -30.0, -math.log(3.0)], [1, 3], [0.75, 0.25]),
    (oracle.SCORE_SQRT_SOFTPLUS, [math.log(math.e - 1.0), -30.0, math.log(math.e ** 4 - 1.0), -30.0],
     [2, 0], [2.0 / 3.0, 1.0 / 3.0]),
])
def test_renormalised_gates_closed_form(score, logits, want_ids, want_g):
    alpha = 2.5
    ids, G, _ = oracle.route_from_logits(np.array([logits]), None, score, 2, alpha, True)
    assert ids.tolist() == [want_ids]
    np.testing.assert_allclose(G[0], alpha * np.array(want_g), rtol=1e-12)
    assert abs(G.sum() - alpha) < 1e-12


def test_softmax_gate_closed_form():
    logits = np.array([[0.0, math.log(2.0), 0.0, math.log(4.0)]])
    ids, G, _ = oracle.route_from_logits(logits, None, oracle.SCORE_SOFTMAX, 2, 1.0, False)
    assert ids.tolist() == [[3, 1]]
    np.testing.assert_allclose(G[0], [0.5, 0.25], rtol=1e-15)


def test_bias_changes_selection_not_weights():
    # equal logits: every affinity is sigma(0) = 1/2, so the bias alone orders
    # the experts and the renormalised gates are alpha / k each.
    E, k, alpha = 7, 3, 2.5
    bias = np.array([0.1, -0.2, 0.5, 0.0, 0.3, -0.1, 0.2])
    ids, G, _ = oracle.route_from_logits(np.zeros((4, E)), bias, oracle.SCORE_SIGMOID, k, alpha, True)
    assert ids.tolist() == [[2, 4, 6]] * 4
    np.testing.assert_allclose(G, alpha / k, rtol=1e-15)


def test_gate_sums_and_k_equals_E():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((50, 9))
    b = rng.standard_normal(9) * 0.1
    for sf in (oracle.SCORE_SIGMOID, oracle.SCORE_SQRT_SOFTPLUS):
        _, G, _ = oracle.route_from_logits(l, b, sf, 4, 2.5, True)
        np.testing.assert_allclose(G.sum(1), 2.5, rtol=1e-13)
        ids, G, a = oracle.route_from_logits(l, None, sf, 9, 1.0, True)
        # k = E, alpha = 1: the gates are the affinities normalised over all experts
        full = np.take_along_axis(a / a.sum(1, keepdims=True), ids.astype(np.int64), 1)
        np.testing.assert_allclose(G, full, rtol=1e-13)
        assert all(sorted(r) == list(range(9)) for r in ids.tolist())
    _, G, _ = oracle.route_from_logits(l, None, oracle.SCORE_SOFTMAX, 4, 1.0, False)
    assert (G.sum(1) <= 1.0 + 1e-15).all() and (G > 0).all()


def test_topk_matches_python_sort_with_ties():
    rng = np.random.default_rng(2)
    s = rng.integers(0, 5, size=(200, 11)).astype(np.float64)  # many exact ties
    ids = oracle.select_topk(s, 4)
    for row, got in zip(s, ids):
        want = sorted(range(11), key=lambda e: (-row[e], e))[:4]
        assert got.tolist() == want


def test_tie_goes_to_lower_id_through_the_router():
    rng = np.random.default_rng(3)
    H, E = 64, 6
    X = _bits(rng.standard_normal((20, H)))
    Wg = rng.standard_normal((H, E)) / 8
    Wg[:, 4] = Wg[:, 1]  # experts 1 and 4 always have the same logit
    bias = np.zeros(E)
    bias[[1, 4]] = 1.0   # ... and the same, winning, selection score
    ids, _, l = oracle.route(X, _bits(Wg), bias, oracle.SCORE_SIGMOID, 3, 1.0, True)
    assert np.array_equal(l[:, 1], l[:, 4])
    assert (ids[:, 0] == 1).all() and (ids[:, 1] == 4).all()
    ids, G, _ = oracle.route(X, _bits(Wg), bias, oracle.SCORE_SIGMOID, 1, 1.0, True)
    assert (ids[:, 0] == 1).all() and np.allclose(G, 1.0)


def test_route_bruteforce_tiny():
    rng = np.random.default_rng(4)
    T, H, E, k, alpha = 5, 8, 6, 3, 2.5
    X = _bits(rng.standard_normal((T, H)))
    Wg = _bits(rng.standard_normal((H, E)) / 3)
    bias = rng.standard_normal(E) * 0.1
    xf = synth.f32_from_bf16_bits(X).astype(float).tolist()
    wf = synth.f32_from_bf16_bits(Wg).astype(float).tolist()
    for sf in (oracle.SCORE_SIGMOID, oracle.SCORE_SQRT_SOFTPLUS):
        ids, G, _ = oracle.route(X, Wg, bias, sf, k, alpha, True)
        for t in range(T):
            logit = [sum(xf[t][h] * wf[h][e] for h in range(H)) for e in range(E)]
            if sf == oracle.SCORE_SIGMOID:
                a = [1.0 / (1.0 + math.exp(-v)) for v in logit]
            else:
                a = [math.sqrt(math.log(1.0 + math.exp(v))) for v in logit]
            order = sorted(range(E), key=lambda e: (-(a[e] + bias[e]), e))[:k]
            assert ids[t].tolist() == order
            tot = sum(a[e] for e in order)
            np.testing.assert_allclose(G[t], [alpha * a[e] / tot for e in order], rtol=1e-12)


def test_hash_route_uses_table_rows():
    d = synth.make_inputs("c4s")
    c = d["cfg"]
    ids, G, l = oracle.route_hash(d["X"], d["Wg"], d["token_ids"], d["tid2eid"],
                                  c["score_fn"], c["alpha"], c["renorm"])
    assert np.array_equal(ids, d["tid2eid"][d["token_ids"]])
    np.testing.assert_allclose(G.sum(1), c["alpha"], rtol=1e-13)
    # same gate formula as the top-k router at those ids
    a = oracle.affinity(l, c["score_fn"])
    np.testing.assert_allclose(G, oracle.gates(a, ids, c["alpha"], True), rtol=0)


# ------------------------------------------------------------------ dispatch
def test_split_worked_example(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "megatron_split_example.json")))
    L = ex["experts_per_rank"]
    toks = ex["tokens"]
    E = 2 * L
    send = {}
    for r in ("0", "1"):
        E_ids = np.array([v["experts"] for v in toks.values() if str(v["rank"]) == r], dtype=np.int32)
        counts, offsets, perm, inv = oracle.dispatch(E_ids, E)
        assert counts.sum() == ex["assignments_per_rank"]
        # input_splits[j] = sum of count[e] over the experts that rank j holds
        send[r] = [int(counts[j * L:(j + 1) * L].sum()) for j in range(2)]
        assert send[r] == ex["send_rows"][r]
    for dst in ("0", "1"):
        out = [send[src][int(dst)] for src in ("0", "1")]
        assert out == ex["output_splits"][dst]
        assert sum(out) == ex["received_rows"][dst]
    # all four tokens on one device: counts and the expert blocks
    E_ids = np.array([v["experts"] for v in toks.values()], dtype=np.int32)
    counts, offsets, perm, inv = oracle.dispatch(E_ids, E)
    assert counts.tolist() == [2, 1, 3, 2] and offsets.tolist() == [0, 2, 3, 6, 8]
    # a = token 0, b = 1, c = 2, d = 3; flat index = token * 2 + slot
    assert perm.tolist() == [0, 4, 2, 1, 3, 6, 5, 7]


def test_dispatch_invariants():
    d = synth.make_inputs("c3s")
    c = d["cfg"]
    ids, _, _ = oracle.route(d["X"], d["Wg"], d["bias"], c["score_fn"], c["k"], c["alpha"], True)
    T, k, E = c["T"], c["k"], c["E"]
    assert all(len(set(r)) == k for r in ids.tolist())  # |I_t| = k
    counts, offsets, perm, inv = oracle.dispatch(ids, E)
    assert counts.sum() == T * k
    assert sorted(perm.tolist()) == list(range(T * k))
    flat = ids.reshape(-1)
    for e in range(E):
        blk = perm[offsets[e]:offsets[e + 1]]
        assert (flat[blk] == e).all() and (np.diff(blk) > 0).all()
    assert (perm[inv] == np.arange(T * k)).all()


def test_dispatch_drops_out_of_range_ids():
    E_ids = np.array([[0, 5], [-1, 2], [2, 1]], dtype=np.int32)
    counts, offsets, perm, inv = oracle.dispatch(E_ids, 3)
    assert counts.tolist() == [1, 1, 2]
    assert perm.tolist() == [0, 5, 3, 4]
    assert inv.tolist() == [0, -1, -1, 2, 3, 1]


# ------------------------------------------------------------------ FFN and combine
def _tiny_layer(rng, T=4, H=8, E=3, k=2, I=4, shared=True):
    X = _bits(rng.standard_normal((T, H)))
    W1 = _bits(rng.standard_normal((E, H, 2 * I)) / 3)
    W2 = _bits(rng.standard_normal((E, I, H)) / 2)
    Ws1 = _bits(rng.standard_normal((H, 2 * I)) / 3) if shared else None
    Ws2 = _bits(rng.standard_normal((I, H)) / 2) if shared else None
    E_ids = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)], dtype=np.int32)
    G = rng.random((T, k))
    return X, E_ids, G, W1, W2, Ws1, Ws2


def _ffn_loops(x, w1, w2):
    """F(x) = (SiLU(x W_gate) * x W_up) W_down with explicit loops."""
    H, twoI = len(w1), len(w1[0])
    I = twoI // 2
    h = [sum(x[r] * w1[r][c] for r in range(H)) for c in range(twoI)]
    act = [h[c] / (1.0 + math.exp(-h[c])) * h[I + c] for c in range(I)]
    return [sum(act[c] * w2[c][o] for c in range(I)) for o in range(len(w2[0]))]


def test_forward_bruteforce_tiny():
    rng = np.random.default_rng(6)
    X, E_ids, G, W1, W2, Ws1, Ws2 = _tiny_layer(rng)
    Y, _ = oracle.forward(X, E_ids, G, W1, W2, Ws1, Ws2)
    f = lambda b: synth.f32_from_bf16_bits(b).astype(float).tolist()  # noqa: E731
    x, w1, w2, s1, s2 = f(X), f(W1), f(W2), f(Ws1), f(Ws2)
    for t in range(X.shape[0]):
        want = _ffn_loops(x[t], s1, s2)
        for j in range(E_ids.shape[1]):
            ye = _ffn_loops(x[t], w1[E_ids[t, j]], w2[E_ids[t, j]])
            want = [a + G[t, j] * b for a, b in zip(want, ye)]
        np.testing.assert_allclose(Y[t], want, rtol=1e-12, atol=1e-12)


def _bf16_scalar(v):
    """Nearest bf16 value of a float, ties to even, written from the format:
    v = m * 2^e with 0.5 <= |m| < 1 (frexp); bf16 keeps 8 significant bits,
    so m * 2^8 is rounded to an integer (Python's round() takes halves to the
    even neighbour) and scaled back."""
    if v == 0.0:
        return 0.0
    m, e = math.frexp(v)
    return math.ldexp(round(m * 256.0), e - 8)


def test_bf16_scalar_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(16)
    x = (rng.standard_normal(4000) * 2.0 ** rng.integers(-20, 20, 4000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert [_bf16_scalar(float(v)) for v in x] == want.tolist()


def test_forward_with_bf16_swiglu_rows_matches_scalar_loops():
    """The oracle's forward with its SwiGLU rows rounded to bf16 (the rounding
    point of a path that keeps them in bf16 between the two GEMMs), against
    per-token loops that round each activation with _bf16_scalar; the rounding
    must also change the result, so the flag is not a no-op."""
    rng = np.random.default_rng(17)
    X, E_ids, G, W1, W2, Ws1, Ws2 = _tiny_layer(rng)
    Y, _ = oracle.forward(X, E_ids, G, W1, W2, Ws1, Ws2, act_round_bf16=True)
    Y0, _ = oracle.forward(X, E_ids, G, W1, W2, Ws1, Ws2)
    f = lambda b: synth.f32_from_bf16_bits(b).astype(float).tolist()  # noqa: E731
    x, w1, w2, s1, s2 = f(X), f(W1), f(W2), f(Ws1), f(Ws2)

    def ffn_rounded(xt, a, b):
        H, twoI = len(a), len(a[0])
        I = twoI // 2
        h = [sum(xt[r] * a[r][c] for r in range(H)) for c in range(twoI)]
        act = [_bf16_scalar(h[c] / (1.0 + math.exp(-h[c])) * h[I + c]) for c in range(I)]
        return [sum(act[c] * b[c][o] for c in range(I)) for o in range(len(b[0]))]

    for t in range(X.shape[0]):
        want = ffn_rounded(x[t], s1, s2)
        for j in range(E_ids.shape[1]):
            ye = ffn_rounded(x[t], w1[E_ids[t, j]], w2[E_ids[t, j]])
            want = [a + G[t, j] * b for a, b in zip(want, ye)]
        np.testing.assert_allclose(Y[t], want, rtol=1e-12, atol=1e-12)
    assert np.abs(Y - Y0).max() > 1e-6 * np.abs(Y0).max()


def _dense_ffn(X64, W1_64, W2_64):
    """Dense SwiGLU FFN with SiLU written through tanh: z*sigma(z) = z*(1+tanh(z/2))/2."""
    I = W2_64.shape[0]
    g = np.einsum("th,hi->ti", X64, W1_64[:, :I])
    u = np.einsum("th,hi->ti", X64, W1_64[:, I:])
    return np.einsum("ti,ih->th", g * (1.0 + np.tanh(g / 2.0)) / 2.0 * u, W2_64)


def test_single_expert_reduces_to_dense_ffn():
    rng = np.random.default_rng(7)
    X, _, _, W1, W2, _, _ = _tiny_layer(rng, T=9, H=16, E=1, k=1, I=8, shared=False)
    Y, _ = oracle.forward(X, np.zeros((9, 1), np.int32), np.ones((9, 1)), W1, W2)
    ref = _dense_ffn(oracle.bf16_to_f64(X), oracle.bf16_to_f64(W1[0]), oracle.bf16_to_f64(W2[0]))
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-13)


def test_zero_gates_leave_the_shared_expert():
    rng = np.random.default_rng(8)
    X, E_ids, G, W1, W2, Ws1, Ws2 = _tiny_layer(rng, T=6, H=16, E=4, k=2, I=8)
    Y, _ = oracle.forward(X, E_ids, np.zeros_like(G), W1, W2, Ws1, Ws2)
    ref = _dense_ffn(oracle.bf16_to_f64(X), oracle.bf16_to_f64(Ws1), oracle.bf16_to_f64(Ws2))
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-13)
    Y0, _ = oracle.forward(X, E_ids, np.zeros_like(G), W1, W2)
    assert (Y0 == 0).all()


def test_gates_act_linearly_and_identical_experts():
    rng = np.random.default_rng(9)
    X, E_ids, G, W1, W2, Ws1, Ws2 = _tiny_layer(rng, T=6, H=16, E=4, k=3, I=8)
    S = _dense_ffn(oracle.bf16_to_f64(X), oracle.bf16_to_f64(Ws1), oracle.bf16_to_f64(Ws2))
    Y1, _ = oracle.forward(X, E_ids, G, W1, W2, Ws1, Ws2)
    Y3, _ = oracle.forward(X, E_ids, 3.0 * G, W1, W2, Ws1, Ws2)
    np.testing.assert_allclose(Y3 - S, 3.0 * (Y1 - S), rtol=1e-11, atol=1e-12)
    # identical experts and gates summing to one give F(x) + F_s(x)
    W1s = np.repeat(W1[:1], 4, axis=0)
    W2s = np.repeat(W2[:1], 4, axis=0)
    Gn = G / G.sum(1, keepdims=True)
    Y, _ = oracle.forward(X, E_ids, Gn, W1s, W2s, Ws1, Ws2)
    F = _dense_ffn(oracle.bf16_to_f64(X), oracle.bf16_to_f64(W1[0]), oracle.bf16_to_f64(W2[0]))
    np.testing.assert_allclose(Y, F + S, rtol=1e-11, atol=1e-12)


def test_probability_before_linear2_equals_weighting_in_combine():
    # the page's fused placement of the gate: g * SwiGLU(.) then Linear2
    rng = np.random.default_rng(10)
    X, E_ids, G, W1, W2, _, _ = _tiny_layer(rng, T=5, H=16, E=3, k=2, I=8, shared=False)
    Y, _ = oracle.forward(X, E_ids, G, W1, W2)
    x = oracle.bf16_to_f64(X)
    want = np.zeros_like(Y)
    for t in range(5):
        for j in range(2):
            e = E_ids[t, j]
            w1 = oracle.bf16_to_f64(W1[e])
            h = x[t] @ w1
            act = G[t, j] * (h[:8] / (1 + np.exp(-h[:8])) * h[8:])
            want[t] += act @ oracle.bf16_to_f64(W2[e])
    np.testing.assert_allclose(Y, want, rtol=1e-12, atol=1e-13)


def test_forward_tokens_subset_matches_whole_layer():
    d = synth.make_inputs("c2s")
    Y, _ = oracle.forward(d["X"], d["E_ids"], d["G"], d["W1"], d["W2"])
    rows = np.array([0, 17, 100, 332])
    Ys = oracle.forward_tokens(rows, d["X"][rows], d["E_ids"][rows], d["G"][rows],
                               lambda e: d["W1"][e], lambda e: d["W2"][e], E=d["cfg"]["E"])
    np.testing.assert_allclose(Ys, Y[rows], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ A8W8-INT
def test_round_half_away_from_zero():
    z = np.array([0.5, -0.5, 1.5, 2.5, -2.5, 0.49999997, -1.4999999], dtype=np.float32)
    assert oracle.round_half_away(z).tolist() == [1, -1, 2, 3, -3, 0, -1]


def test_int8_row_quantisation_closed_forms():
    q, s = oracle.quantize_rows_int8(np.array([[127.0, 63.5, -63.5, 0.49], [0.0, 0.0, 0.0, 0.0]]))
    assert q.tolist() == [[127, 64, -64, 0], [0, 0, 0, 0]] and s.tolist() == [1.0, 0.0]
    rng = np.random.default_rng(20)
    x = rng.standard_normal((64, 300)) * rng.uniform(0.01, 100, size=(64, 1))
    for dt in (np.float32, np.float64):
        q, s = oracle.quantize_rows_int8(x.astype(dt), dt)
        assert (np.abs(q) <= 127).all()
        # the largest magnitude of each row becomes exactly +-127
        amax_idx = np.abs(x).argmax(1)
        assert (np.abs(q[np.arange(64), amax_idx]) == 127).all()
        # reconstruction within half a step
        assert (np.abs(x - q * s[:, None].astype(np.float64)) <= 0.5 * s[:, None] * (1 + 1e-6)).all()


def test_a8w8_expert_matches_integer_brute_force():
    rng = np.random.default_rng(21)
    N, H, I = 3, 8, 4
    q = rng.integers(-127, 128, size=(N, H))
    sx = rng.uniform(0.01, 0.1, size=N)
    W1q = rng.integers(-127, 128, size=(2 * I, H))   # weight1: one row per output channel
    S1 = rng.uniform(0.001, 0.01, size=2 * I)
    W2q = rng.integers(-127, 128, size=(H, I))       # weight2
    S2 = rng.uniform(0.001, 0.01, size=H)
    Y = oracle.swiglu_expert_a8w8(q, sx, W1q, S1, W2q, S2)
    for n in range(N):
        C = [sum(int(q[n, h]) * int(W1q[c, h]) for h in range(H)) for c in range(2 * I)]
        Hv = [C[c] * S1[c] * sx[n] for c in range(2 * I)]
        A = [Hv[c] / (1 + math.exp(-Hv[c])) * Hv[I + c] for c in range(I)]
        sA = max(abs(a) for a in A) / 127
        A8 = [int(math.copysign(math.floor(abs(a / sA) + 0.5), a)) for a in A]
        D = [sum(A8[i] * int(W2q[o, i]) for i in range(I)) for o in range(H)]
        np.testing.assert_allclose(Y[n], [D[o] * S2[o] * sA for o in range(H)], rtol=1e-12)


def test_a8w8_layer_within_the_activation_quantisation_bound():
    # Quantised token rows and weights that are exactly code * scale: then the
    # A8W8 layer differs from the plain float layer on the dequantised operands
    # only through the re-quantisation of the SwiGLU output, bounded per
    # element by sum_i |dA_i| |W2[i, o]| <= (s_A / 2) sum_i |W2[i, o]|.
    d = synth.make_inputs("c3s_q")
    c = d["cfg"]
    T, k, E, I = c["T"], c["k"], c["E"], c["I"]
    ids, G, _ = oracle.route(d["X"], d["Wg"], d["bias"], c["score_fn"], k, c["alpha"], True)
    Y = oracle.forward_a8w8_tokens(np.arange(T), d["X"], ids, G, d["W1"], d["S1"], d["W2"], d["S2"], E=E)
    x32 = oracle.bf16_to_f64(d["X"]).astype(np.float32)
    q, sx = oracle.quantize_rows_int8(x32, np.float32)
    Xd = q * sx[:, None].astype(np.float64)
    for t in (0, 5, T - 1):
        want = np.zeros(c["H"])
        bound = np.zeros(c["H"])
        for j in range(k):
            e = ids[t, j]
            W1 = d["W1"][e].T.astype(np.float64) * d["S1"][e][None, :].astype(np.float64)
            W2 = d["W2"][e].T.astype(np.float64) * d["S2"][e][None, :].astype(np.float64)
            h = Xd[t] @ W1
            a = h[:I] / (1 + np.exp(-h[:I])) * h[I:]
            want += G[t, j] * (a @ W2)
            bound += abs(G[t, j]) * (np.abs(a).max() / 127 / 2) * np.abs(W2).sum(0)
        assert (np.abs(Y[t] - want) <= bound * (1 + 1e-9) + 1e-12).all()


# ------------------------------------------------------------------ MXFP8
_TORCH_FP8 = {"e4m3": "float8_e4m3fn", "e5m2": "float8_e5m2"}


def _torch_fp8(fmt):
    torch = pytest.importorskip("torch")
    dt = getattr(torch, _TORCH_FP8[fmt], None)
    if dt is None:
        pytest.skip("this torch has no %s" % _TORCH_FP8[fmt])
    return torch, dt


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_decode_matches_torch_table(fmt):
    torch, dt = _torch_fp8(fmt)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(dt).to(torch.float64).numpy()
    ours = oracle.fp8_decode(np.arange(256), fmt)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_rounding_matches_torch_in_range(fmt):
    """Inside the finite range the rounding is the library's round-to-nearest-
    even conversion; the exact midpoints between neighbouring codes decide the
    tie rule."""
    torch, dt = _torch_fp8(fmt)
    vmax = oracle.FP8_FORMATS[fmt][3]
    grid = oracle.fp8_decode(np.arange(128), fmt)
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(11)
    rand = np.exp(rng.uniform(np.log(1e-7), np.log(vmax), 20000)) * rng.choice([-1, 1], 20000)
    v = np.concatenate([mids, -mids, grid, -grid, rand, [0.0, -0.0]]).astype(np.float32)
    assert np.all(np.abs(v) <= vmax)
    ref = torch.from_numpy(v).to(dt).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_encode(v.astype(np.float64), fmt), ref)


def test_fp8_saturates_to_the_largest_finite_value():
    # E4M3FN: S.1111.110 = 1.75 * 2^8 = 448; E5M2: S.11110.11 = 1.75 * 2^15
    for fmt, code in (("e4m3", 0x7E), ("e5m2", 0x7B)):
        vmax = oracle.FP8_FORMATS[fmt][3]
        v = np.array([vmax, vmax * 1.01, vmax * 1.2, 1e30, -vmax * 1.2, -1e30])
        got = oracle.fp8_encode(v, fmt)
        assert list(got) == [code, code, code, code, code | 0x80, code | 0x80]


def test_mx_quantize_worked_group():
    """Worked by hand: x = 1..32.  max 32 = 2^5, E4M3 emax = 8, so the shared
    exponent is 5 - 8 = -3 (scale code 124) and the elements are 8x.  In
    [128, 256) the E4M3 spacing is 2^(7-3) = 16: 136 = 8.5 steps rounds to
    the even 8 (128 -> 16), 152 = 9.5 steps to 10 (160 -> 20), 168 = 10.5
    to 10 (160 -> 20), 184 = 11.5 to 12 (192 -> 24), 200 = 12.5 to 12,
    216 = 13.5 to 14 (224 -> 28), 232 = 14.5 to 14, 248 = 15.5 to 16
    (256 -> 32); below 128 every 8x is on the grid."""
    x = np.arange(1, 33, dtype=np.float64)
    q, s = oracle.mx_quantize(x, "e4m3")
    assert list(s) == [124]
    want = list(range(1, 17)) + [16, 18, 20, 20, 20, 22, 24, 24, 24, 26, 28, 28, 28, 30, 32, 32]
    assert list(oracle.mx_dequantize(q, s, "e4m3")) == want


# FLOAT4_E2M1 values of the OCP Microscaling formats table, codes 0..7
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_codes_match_the_format_table():
    v = oracle.fp8_decode(np.arange(16), "e2m1")
    assert list(v[:8]) == E2M1_TABLE
    assert list(-v[8:]) == E2M1_TABLE and all(np.signbit(v[8:]))


def test_e2m1_rounding_ties_and_saturation():
    """Halfway cases go to the even code (mantissa bit 0): 0.25 -> 0,
    0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; beyond 6
    saturates; the sign of zero is kept."""
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0, -5.0, -0.0, 0.3])
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -4.0, -0.0, 0.5]
    got = oracle.fp8_decode(oracle.fp8_encode(v, "e2m1"), "e2m1")
    assert list(got) == want
    assert np.signbit(got[10])


def test_e2m1_unpacking_order():
    """Two codes per byte, the even element in the low nibble."""
    b = np.array([[0x21, 0xF0, 0x7A]], dtype=np.uint8)
    assert oracle.unpack_e2m1(b).tolist() == [[1, 2, 0, 15, 10, 7]]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
def test_mx_quantize_closed_forms(fmt):
    """The shared exponent from frexp (an independent route to floor(log2)),
    the rounding error bound of each element, exact round trips of values
    already on the MX grid, and a group of zeros."""
    eb, mb, bias, vmax = oracle.FP8_FORMATS[fmt]
    emax = {"e4m3": 8, "e5m2": 15, "e2m1": 2}[fmt]
    rng = np.random.default_rng(3)
    G = 400
    x = rng.standard_normal((G, 32)) * np.exp(rng.uniform(-20, 20, (G, 1)))
    q, s = oracle.mx_quantize(x, fmt)
    d = oracle.mx_dequantize(q, s, fmt)
    for g in range(G):
        amax = float(np.abs(x[g]).max())
        X = math.frexp(amax)[1] - 1 - emax
        assert int(s[g, 0]) == X + 127
        for v, dv in zip(x[g], d[g]):
            a = abs(v) / 2.0 ** X
            if a >= vmax:
                assert dv == math.copysign(vmax, v) * 2.0 ** X
                continue
            e = max(math.frexp(a)[1] - 1, 1 - bias) if a > 0 else 1 - bias
            assert abs(dv - v) <= 2.0 ** (e - mb - 1) * 2.0 ** X
    # values on the grid come back unchanged
    grid = oracle.mx_dequantize(q, s, fmt)
    q2, s2 = oracle.mx_quantize(grid, fmt)
    assert np.array_equal(oracle.mx_dequantize(q2, s2, fmt), grid)
    qz, sz = oracle.mx_quantize(np.zeros((1, 64)), fmt)
    assert list(sz[0]) == [0, 0] and not qz.any()


def _scalar_fp(fmt):
    """(decode(code), round(value)) for scalar brute force: FP8 through torch's
    float8 types; E2M1 through the format table, rounding by a search for the
    nearest table value with ties to the even code."""
    if fmt == "e2m1":
        def dec(code):
            v = E2M1_TABLE[code & 7]
            return -v if code & 8 else v

        def rnd(c):
            a = abs(c)
            best = min(range(8), key=lambda i: (abs(E2M1_TABLE[i] - a), i & 1))
            return math.copysign(E2M1_TABLE[best], c)
        return dec, rnd
    torch, dt = _torch_fp8(fmt)

    def dec(code):
        return torch.tensor([int(code)], dtype=torch.uint8).view(dt).to(torch.float64).item()

    def rnd(c):
        code = torch.tensor([c], dtype=torch.float32).to(dt).view(torch.uint8).item()
        return dec(code)
    return dec, rnd


def _bruteforce_mx_layer(X, E_ids, G, W1q, S1, W2q, S2, fmt, wfmt=None):
    """Per token, per expert, scalar loops: codes decoded by torch's float8
    types (E2M1 by the format table), scales 2^(code-127) by ldexp, shared
    exponents by frexp, element rounding by torch's conversion (E2M1 by a
    table search) after clamping to the finite range."""
    wfmt = fmt if wfmt is None else wfmt
    dec, rnd = _scalar_fp(fmt)
    wdec, _ = _scalar_fp(wfmt)
    vmax = oracle.FP8_FORMATS[fmt][3]
    emax = {"e4m3": 8, "e5m2": 15, "e2m1": 2}[fmt]

    def quant_row(v):
        out = []
        for g0 in range(0, len(v), 32):
            grp = v[g0:g0 + 32]
            amax = max(abs(t) for t in grp)
            X = max(-127, math.frexp(amax)[1] - 1 - emax) if amax > 0 else -127
            for t in grp:
                c = min(max(t / 2.0 ** X, -vmax), vmax)
                out.append(math.ldexp(rnd(c), X))
        return out

    T, k = E_ids.shape
    H = X.shape[1]
    I = W2q.shape[2]
    Y = np.zeros((T, H))
    for t in range(T):
        xd = quant_row([float(v) for v in X[t]])
        for j in range(k):
            e = int(E_ids[t, j])
            z = []
            for n in range(2 * I):
                acc = 0.0
                for h in range(H):
                    w = math.ldexp(wdec(W1q[e, n, h]), int(S1[e, n, h // 32]) - 127)
                    acc += xd[h] * w
                z.append(acc)
            u = [z[i] / (1.0 + math.exp(-z[i])) * z[I + i] for i in range(I)]
            ud = quant_row(u)
            for hh in range(H):
                acc = 0.0
                for i in range(I):
                    acc += ud[i] * math.ldexp(wdec(W2q[e, hh, i]), int(S2[e, hh, i // 32]) - 127)
                Y[t, hh] += float(G[t, j]) * acc
    return Y


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e2m1"),
                                      ("e2m1", "e2m1")])
def test_mx_layer_matches_scalar_bruteforce(fmt, wfmt):
    rng = np.random.default_rng(21)
    T, H, I, E, k = 4, 64, 32, 3, 2
    X = oracle.round_to_bf16(rng.standard_normal((T, H)))
    codes = np.arange(16 if wfmt == "e2m1" else 256)
    vals = oracle.fp8_decode(codes, wfmt)
    finite = codes[np.isfinite(vals) & (np.abs(vals) <= 4.0)]
    W1q = rng.choice(finite, (E, 2 * I, H)).astype(np.uint8)
    W2q = rng.choice(finite, (E, H, I)).astype(np.uint8)
    S1 = rng.integers(118, 124, (E, 2 * I, H // 32)).astype(np.uint8)
    S2 = rng.integers(118, 124, (E, H, I // 32)).astype(np.uint8)
    E_ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1]])
    G = rng.uniform(0.1, 1.0, (T, k))
    got = oracle.forward_mx_tokens(np.arange(T), oracle.f64_to_bf16_bits(X), E_ids, G,
                                   W1q, S1, W2q, S2, E, fmt, wfmt)
    want = _bruteforce_mx_layer(X, E_ids, G, W1q, S1, W2q, S2, fmt, wfmt)
    scale = np.abs(want).max()
    assert np.allclose(got, want, rtol=1e-9, atol=1e-12 * scale)


# ------------------------------------------------------------------ backward
def _bwd_case(seed, T, H, E, k, I, shared):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, H))
    Wg = rng.standard_normal((H, E)) / math.sqrt(H)
    W1 = rng.standard_normal((E, H, 2 * I)) / math.sqrt(H)
    W2 = rng.standard_normal((E, I, H)) / math.sqrt(I)
    Ws1 = rng.standard_normal((H, 2 * I)) / math.sqrt(H) if shared else None
    Ws2 = rng.standard_normal((I, H)) / math.sqrt(I) if shared else None
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    dY = rng.standard_normal((T, H))
    return X, Wg, W1, W2, Ws1, Ws2, ids, dY


def _layer_loss(X, Wg, W1, W2, Ws1, Ws2, ids, dY, score_fn, alpha, renorm):
    """sum(dY * Y) through the oracle's forward functions, routing ids fixed."""
    a = oracle.affinity(oracle.router_logits(X, Wg), score_fn)
    G = oracle.gates(a, ids, alpha, renorm)
    Y = oracle.forward_tokens(np.arange(X.shape[0]), X, ids, G, W1, W2, Ws1, Ws2, E=W1.shape[0])
    return float((dY * Y).sum())


@pytest.mark.parametrize("score_fn,renorm,shared", [(0, True, True), (1, True, False),
                                                     (2, False, True), (2, True, False),
                                                     (0, False, False)])
def test_backward_matches_central_differences(score_fn, renorm, shared):
    """Every parameter and input entry of a tiny layer: the oracle's gradient
    against (L(p + h) - L(p - h)) / 2h of the oracle's forward."""
    X, Wg, W1, W2, Ws1, Ws2, ids, dY = _bwd_case(4 + score_fn, T=3, H=6, E=4, k=2, I=3, shared=shared)
    alpha = 2.5 if renorm else 1.0
    g = oracle.backward(X, Wg, ids, dY, W1, W2, Ws1, Ws2, score_fn, alpha, renorm)
    params = {"dX": X, "dWg": Wg, "dW1": W1, "dW2": W2}
    if shared:
        params.update(dWs1=Ws1, dWs2=Ws2)
    h = 1e-6
    for name, P in params.items():
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            keep = P[idx]
            P[idx] = keep + h
            up = _layer_loss(X, Wg, W1, W2, Ws1, Ws2, ids, dY, score_fn, alpha, renorm)
            P[idx] = keep - h
            dn = _layer_loss(X, Wg, W1, W2, Ws1, Ws2, ids, dY, score_fn, alpha, renorm)
            P[idx] = keep
            fd[idx] = (up - dn) / (2 * h)
        assert np.allclose(g[name], fd, rtol=1e-6, atol=1e-7), name


def test_backward_matches_torch_autograd():
    """A larger layer against torch's reverse-mode differentiation (float64)
    of the same forward: sigmoid affinity, renormalised alpha-scaled gates,
    shared expert."""
    torch = pytest.importorskip("torch")
    X, Wg, W1, W2, Ws1, Ws2, ids, dY = _bwd_case(9, T=17, H=32, E=6, k=3, I=16, shared=True)
    alpha = 2.5
    g = oracle.backward(X, Wg, ids, dY, W1, W2, Ws1, Ws2, 0, alpha, True)
    t = {n: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for n, v in dict(X=X, Wg=Wg, W1=W1, W2=W2, Ws1=Ws1, Ws2=Ws2).items()}
    idt = torch.tensor(ids, dtype=torch.int64)
    a = torch.sigmoid(t["X"] @ t["Wg"])
    a_sel = torch.gather(a, 1, idt)
    G = alpha * a_sel / a_sel.sum(dim=1, keepdim=True)
    I = W2.shape[1]

    def ffn(x, w1, w2):
        h = x @ w1
        return (torch.nn.functional.silu(h[:, :I]) * h[:, I:]) @ w2

    Y = ffn(t["X"], t["Ws1"], t["Ws2"])
    for j in range(ids.shape[1]):
        rows = [G[r, j] * ffn(t["X"][r:r + 1], t["W1"][int(ids[r, j])], t["W2"][int(ids[r, j])])
                for r in range(X.shape[0])]
        Y = Y + torch.cat(rows, dim=0)
    (torch.tensor(dY) * Y).sum().backward()
    for n, key in dict(X="dX", Wg="dWg", W1="dW1", W2="dW2", Ws1="dWs1", Ws2="dWs2").items():
        assert np.allclose(g[key], t[n].grad.numpy(), rtol=1e-9, atol=1e-11), key


def _backward_loops_bf16(X, Wg, ids, dY, W1, W2, Ws1, Ws2, alpha):
    """Gradients of a tiny sigmoid-routed layer (renormalised gates, shared
    expert) by scalar loops, rounding to bf16 (_bf16_scalar) at the five
    points where a bf16 path keeps its tensors: the pre-activations H as the
    backward reads them, the SwiGLU output A (from the unrounded H), the
    gate-scaled row gradient g dY, the pre-activation gradient dH, and the
    logit gradient before its two products."""
    T, H = X.shape
    E, k, I = Wg.shape[1], ids.shape[1], W2.shape[1]
    bf, sig = _bf16_scalar, (lambda z: 1.0 / (1.0 + math.exp(-z)))
    silu = lambda z: z * sig(z)  # noqa: E731
    dsilu = lambda z: sig(z) * (1.0 + z * (1.0 - sig(z)))  # noqa: E731
    dX = np.zeros((T, H))
    dWg = np.zeros((H, E))
    dW1, dW2 = np.zeros((E, H, 2 * I)), np.zeros((E, I, H))
    dWs1, dWs2 = np.zeros((H, 2 * I)), np.zeros((I, H))
    dG = np.zeros((T, k))

    def branch(t, w1, w2, gate, dw1, dw2):
        """One expert FFN branch of token t: accumulates dX, dw1, dw2 and
        returns <dY_t, y> (y the branch output, A rounded)."""
        h = [sum(X[t, r] * w1[r, c] for r in range(H)) for c in range(2 * I)]
        hk = [bf(v) for v in h]
        act = [bf(silu(h[c]) * h[I + c]) for c in range(I)]
        y = [sum(act[c] * w2[c, o] for c in range(I)) for o in range(H)]
        dout = [bf(gate * dY[t, o]) for o in range(H)]
        dA = [sum(dout[o] * w2[c, o] for o in range(H)) for c in range(I)]
        dh = ([bf(dA[c] * hk[I + c] * dsilu(hk[c])) for c in range(I)]
              + [bf(dA[c] * silu(hk[c])) for c in range(I)])
        for c in range(I):
            for o in range(H):
                dw2[c, o] += act[c] * dout[o]
        for r in range(H):
            for c in range(2 * I):
                dw1[r, c] += X[t, r] * dh[c]
            dX[t, r] += sum(dh[c] * w1[r, c] for c in range(2 * I))
        return sum(dY[t, o] * y[o] for o in range(H))

    for t in range(T):
        l = [sum(X[t, r] * Wg[r, e] for r in range(H)) for e in range(E)]
        a = [sig(v) for v in l]
        S = sum(a[ids[t, j]] for j in range(k))
        g = [alpha * a[ids[t, j]] / S for j in range(k)]
        branch(t, Ws1, Ws2, 1.0, dWs1, dWs2)
        for j in range(k):
            e = ids[t, j]
            dG[t, j] = branch(t, W1[e], W2[e], g[j], dW1[e], dW2[e])
        # g_j = alpha a_j / S:  dL/da_i = alpha / S (dG_i - sum_j dG_j a_j / S)
        da = [0.0] * E
        ssum = sum(dG[t, j] * a[ids[t, j]] for j in range(k)) / S
        for j in range(k):
            da[ids[t, j]] += alpha / S * (dG[t, j] - ssum)
        dl = [bf(da[e] * a[e] * (1.0 - a[e])) for e in range(E)]
        for r in range(H):
            for e in range(E):
                dWg[r, e] += X[t, r] * dl[e]
            dX[t, r] += sum(dl[e] * Wg[r, e] for e in range(E))
    return dict(dX=dX, dWg=dWg, dW1=dW1, dW2=dW2, dWs1=dWs1, dWs2=dWs2, dG=dG)


def test_backward_with_bf16_rounding_points_matches_scalar_loops():
    X, Wg, W1, W2, Ws1, Ws2, ids, dY = _bwd_case(31, T=3, H=6, E=4, k=2, I=3, shared=True)
    X = oracle.round_to_bf16(X)
    alpha = 2.5
    got = oracle.backward(X, Wg, ids, dY, W1, W2, Ws1, Ws2, 0, alpha, True, round_bf16=True)
    want = _backward_loops_bf16(X, Wg, ids, dY, W1, W2, Ws1, Ws2, alpha)
    exact = oracle.backward(X, Wg, ids, dY, W1, W2, Ws1, Ws2, 0, alpha, True)
    for key, w in want.items():
        scale = np.abs(w).max()
        assert np.allclose(got[key], w, rtol=1e-12, atol=1e-12 * scale), key
        # the rounding points move every gradient, so none of them is a no-op
        assert np.abs(got[key] - exact[key]).max() > 1e-6 * scale, key


@pytest.mark.parametrize("name", ["c1s", "c3s", "c4s", "c5s"])
def test_backward_rounding_points_move_gradients_by_the_derived_rms(name):
    """The five bf16 rounding points of the rounded backward each move an
    operand by a relative error of RMS 2^-9 / sqrt(3) (uniform over half an
    ulp of 8 significant bits); a gradient depends on at most five of them,
    so its RMS distance from the exact gradient is at most 5 * 2^-9 / sqrt(3)
    of its RMS.  This is the bound the GPU backward tests use."""
    h = synth.make_inputs(name)
    c = h["cfg"]
    if c["routing"] == "hash":
        ids = h["tid2eid"][h["token_ids"]]
    else:
        ids, _, _ = oracle.route(h["X"], h["Wg"], h["bias"], c["score_fn"], c["k"], c["alpha"], c["renorm"])
    dY = oracle.bf16_to_f64(synth.upstream_grad(c["T"], c["H"]))
    args = (h["X"], h["Wg"], ids, dY, h["W1"], h["W2"], h["Ws1"], h["Ws2"], c["score_fn"], c["alpha"],
            c["renorm"])
    ref = oracle.backward(*args, round_bf16=True)
    exact = oracle.backward(*args)
    bound = 5 * 2.0 ** -9 / math.sqrt(3)
    for key in ("dX", "dWg", "dW1", "dW2", "dG") + (("dWs1", "dWs2") if c["shared"] else ()):
        rms = np.sqrt((exact[key] ** 2).mean())
        assert np.sqrt(((ref[key] - exact[key]) ** 2).mean()) <= bound * rms, key


# ------------------------------------------------------------------ decision margins
def _perturbed_mx_rows(xq, sx, W1q, S1, W2q, S2, fmt, wfmt, rng, rel):
    """swiglu_expert_mx with each pre-activation moved anywhere within rel
    times its product-magnitude sum (what a float32 accumulation may do)."""
    Xd = oracle.mx_dequantize(xq, sx, fmt)
    W1d = oracle.mx_dequantize(W1q, S1, wfmt)
    Z = Xd @ W1d.T
    Z = Z + rng.uniform(-1, 1, Z.shape) * rel * (np.abs(Xd) @ np.abs(W1d).T)
    I = W2q.shape[1]
    U = Z[:, :I] / (1 + np.exp(-Z[:, :I])) * Z[:, I:]
    Uq, SU = oracle.mx_quantize(U, fmt)
    return oracle.mx_dequantize(Uq, SU, fmt) @ oracle.mx_dequantize(W2q, S2, wfmt).T


@pytest.mark.parametrize("fmt,wfmt", [("e4m3", "e4m3"), ("e2m1", "e2m1")])
def test_mx_decision_margin_bounds_float32_moves(fmt, wfmt):
    """Moving the pre-activations within the assumed float32 error flips some
    activation codes (and so moves outputs); every move stays within the
    margin, and the margin is zero wherever no decision is within reach."""
    rng = np.random.default_rng(41)
    m, H, I = 24, 256, 128
    x = rng.standard_normal((m, H))
    xq, sx = oracle.mx_quantize(x, fmt)
    codes = np.arange(16 if wfmt == "e2m1" else 256)
    vals = oracle.fp8_decode(codes, wfmt)
    finite = codes[np.isfinite(vals) & (np.abs(vals) <= 4.0)]
    W1q = rng.choice(finite, (2 * I, H)).astype(np.uint8)
    W2q = rng.choice(finite, (H, I)).astype(np.uint8)
    S1 = rng.integers(118, 122, (2 * I, H // 32)).astype(np.uint8)
    S2 = rng.integers(118, 122, (H, I // 32)).astype(np.uint8)
    rel = 2.0 ** -7  # large, so that many decisions are within reach
    base = oracle.swiglu_expert_mx(xq, sx, W1q, S1, W2q, S2, fmt, wfmt)
    B = oracle.swiglu_margin_mx(xq, sx, W1q, S1, W2q, S2, fmt, wfmt, rel=rel)
    moved = 0
    for _ in range(8):
        d = np.abs(_perturbed_mx_rows(xq, sx, W1q, S1, W2q, S2, fmt, wfmt, rng, rel) - base)
        assert np.all(d <= B * (1 + 1e-9) + 1e-12)
        moved += int((d > 0).sum())
    assert moved > 0 and (B > 0).any()


def test_a8w8_decision_margin_bounds_float32_moves():
    rng = np.random.default_rng(42)
    m, H, I = 24, 128, 96
    x = rng.standard_normal((m, H)).astype(np.float32)
    q, sx = oracle.quantize_rows_int8(x, np.float32)
    W1q = rng.integers(-127, 128, (2 * I, H)).astype(np.int8)
    W2q = rng.integers(-127, 128, (H, I)).astype(np.int8)
    S1 = rng.uniform(0.5, 1.5, 2 * I) / 127 / np.sqrt(H)
    S2 = rng.uniform(0.5, 1.5, H) / 127 / np.sqrt(I)
    rel = 2.0 ** -9
    base = oracle.swiglu_expert_a8w8(q, sx, W1q, S1, W2q, S2)
    B = oracle.swiglu_margin_a8w8(q, sx, W1q, S1, W2q, S2, rel=rel)
    C = q.astype(np.int64) @ W1q.astype(np.int64).T
    Z0 = C * S1[None, :] * sx[:, None].astype(np.float64)
    moved = 0
    for _ in range(8):
        Z = Z0 * (1 + rng.uniform(-1, 1, Z0.shape) * rel)
        U = Z[:, :I] / (1 + np.exp(-Z[:, :I])) * Z[:, I:]
        U = U * (1 + rng.uniform(-1, 1, U.shape) * rel)
        s = np.abs(U).max(axis=1) / 127 * (1 + rng.uniform(-1, 1, m) * rel)
        A8 = oracle.round_half_away(U / s[:, None])
        out = (A8 @ W2q.astype(np.float64).T) * S2[None, :] * s[:, None]
        # the row scale moves every dequantised value by up to rel of itself:
        # a continuous change, bounded separately from the code flips
        cont = rel * 1.01 * (np.abs(A8) * s[:, None]) @ (np.abs(W2q.astype(np.float64)) * S2[:, None]).T
        d = np.abs(out - base)
        assert np.all(d <= B * (1 + 1e-9) + cont + 1e-12)
        moved += int((d > cont).sum())
    assert moved > 0 and (B > 0).any()
