"""The step (route + forward, bf16 and quantised forms) captured in a CUDA graph
and replayed: bit-identical to the same calls made eagerly, also after new
token rows are copied into the captured input buffer.  Every launch of the
path sizes itself from device memory (no host synchronisation), which is what
makes the capture possible."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle
import synth
from _gpu import DEV, bf, check_y_layer, params, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


def _route(p, dd, ws, E_ids, G):
    c = dd["cfg"]
    if c["routing"] == "hash":
        moe.moe_route(p, dd["X"], dd["Wg"], None, dd["token_ids"], dd["tid2eid"], c["V"], E_ids, G, ws)
    else:
        moe.moe_route(p, dd["X"], dd["Wg"], dd.get("bias"), None, None, 0, E_ids, G, ws)


def _forward(form, p, dd, ws, E_ids, G, Y):
    if form == "bf16":
        moe.moe_forward(p, dd["X"], E_ids, G, dd["W1"], dd["W2"], dd.get("Ws1"), dd.get("Ws2"), Y, ws)
    elif form == "a8w8":
        moe.moe_forward_a8w8(p, dd["X"], E_ids, G, dd["W1"], dd["S1"], dd["W2"], dd["S2"], Y, ws)
    else:
        c = dd["cfg"]
        moe.moe_forward_mx(p, moe.MX_FORMATS[synth.mx_format(c["quant"])], dd["X"], E_ids, G, dd["W1"], dd["S1"],
                           dd["W2"], dd["S2"], Y, ws, wfmt=moe.MX_FORMATS[synth.mx_weight_format(c["quant"])])


def _alloc(form, p):
    if form == "bf16":
        return moe.alloc_workspace(p, DEV)
    if form == "a8w8":
        return moe.alloc_workspace_a8w8(p, DEV)
    return moe.alloc_workspace_mx(p, DEV)


@pytest.mark.parametrize("name,form", [("c1", "bf16"), ("c3s", "bf16"), ("c4s", "bf16"), ("c3s_q", "a8w8"),
                                       ("c3s_mxa4", "mx")])
def test_step_replays_as_a_graph(name, form):
    h = synth.make_inputs(name)
    dd = to_device(h)
    c = h["cfg"]
    p = params(c)
    ws_r = moe.alloc_workspace(p, DEV)
    ws = _alloc(form, p)
    T, k, H = c["T"], c["k"], c["H"]
    E_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    G = torch.empty((T, k), dtype=torch.float32, device=DEV)
    Y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)

    def step():
        _route(p, dd, ws_r, E_ids, G)
        _forward(form, p, dd, ws, E_ids, G, Y)

    # eager, on a side stream that then also serves as the capture's warm-up
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    moe.moe_sync_status(ws)
    Y_eager, ids_eager = Y.clone(), E_ids.clone()

    graph = torch.cuda.CUDAGraph()
    Y.fill_(float("nan"))
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    moe.moe_sync_status(ws)
    assert torch.equal(E_ids, ids_eager)
    assert torch.equal(Y.view(torch.int16), Y_eager.view(torch.int16))

    # new token rows in the captured buffer: the replay routes and computes them
    h2 = synth.make_inputs(name, seed=4321)
    dd["X"].copy_(bf(h2["X"]))
    graph.replay()
    torch.cuda.synchronize()
    moe.moe_sync_status(ws)
    Y_graph, ids_graph = Y.clone(), E_ids.clone()
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(ids_graph, E_ids)
    assert torch.equal(Y_graph.view(torch.int16), Y.view(torch.int16))
    assert not torch.equal(Y_graph.view(torch.int16), Y_eager.view(torch.int16))
    if form == "bf16":
        x2 = h2["X"]
        ids, Gr, _ = (oracle.route_hash(x2, h["Wg"], h["token_ids"], h["tid2eid"], c["score_fn"], c["alpha"],
                                        c["renorm"])
                      if c["routing"] == "hash" else
                      oracle.route(x2, h["Wg"], h["bias"], c["score_fn"], k, c["alpha"], c["renorm"]))
        assert np.array_equal(ids_graph.cpu().numpy(), ids)
        check_y_layer(Y_graph, f"{name} graph replay", x2, ids, Gr, h["W1"], h["W2"], h.get("Ws1"),
                      h.get("Ws2"))
