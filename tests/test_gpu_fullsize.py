"""GPU parity at the workloads' full sizes: one or two seeded layers of each
workload, every output row compared with the oracle (which copies only the
experts it selects), and the union sweep byte-identical to the per-row mode.
Runs in the launch form the benchmark times: several layers captured in one
CUDA graph and replayed."""
import numpy as np
import pytest
import torch

from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


# (workload, layer, rows, activations): "wl" = the workload's own recipe,
# "corr" = rows correlated as in the verify workload (the prefill sub-chunk
# is also run that way, for comparison with its independent rows)
CASES = [
    ("decode_h2048_e128", 0, 1, "wl"),
    ("decode_h2048_e128", 47, 1, "wl"),
    ("verify_h4096_e256", 0, 2, "wl"),
    ("verify_h4096_e256", 1, 3, "wl"),
    ("verify_h4096_e256", 2, 4, "wl"),
    ("prefill8_h2048_e512", 0, 8, "wl"),
    ("prefill8_h2048_e512", 1, 8, "corr"),
    ("prefill8_h2048_e512", 2, 16, "wl"),     # two 8-row sub-chunks in one call
    ("sweep_h4096_e160", 0, 1, "wl"),
    ("sweep_h4096_e160", 5, 5, "wl"),
    ("sweep_h4096_e160", 47, 8, "wl"),
]


@pytest.mark.parametrize("name,layer,rows,acts", CASES)
def test_full_size_layer_vs_oracle(name, layer, rows, acts):
    wl = synth.WORKLOADS[name]
    corr = wl.corr if acts == "wl" else synth.WORKLOADS["verify_h4096_e256"].corr
    weights = synth.make_layer(wl.shape, wl.seed_base + layer, device="cuda")
    x = synth.make_rows(wl.shape, rows, seed=wl.seed_base + 500 + layer, device="cuda",
                        corr=corr)
    res = G.gpu_run(weights, x)
    st = G.check_parity(weights, x, res)
    print(name, layer, rows, acts, "U=%d" % res["uni"]["U"], st)
    if acts == "corr":
        assert res["uni"]["U"] < 48          # correlated rows share experts
    pr = G.gpu_run(weights, x, per_row=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("name,layer", [("decode_h2048_e128", 3), ("sweep_h4096_e160", 2),
                                        ("verify_h4096_e256", 4)])
def test_full_size_gemv_lever_one_row(name, layer):
    """The one-row CUDA-core GEMV variant at the workloads' full sizes."""
    wl = synth.WORKLOADS[name]
    weights = synth.make_layer(wl.shape, wl.seed_base + layer, device="cuda")
    x = synth.make_rows(wl.shape, 1, seed=wl.seed_base + 500 + layer, device="cuda", corr=wl.corr)
    res = G.gpu_run(weights, x, gemv=True)
    st = G.check_parity(weights, x, res)
    print(name, layer, "gemv", st)
    pr = G.gpu_run(weights, x, per_row=True, gemv=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


def test_full_size_graph_replay_matches_eager():
    wl = synth.WORKLOADS["prefill8_h2048_e512"]
    layers = [L.DeviceLayer(synth.make_layer(wl.shape, wl.seed_base + i, device="cuda"))
              for i in range(3)]
    xs = [synth.make_rows(wl.shape, 8, seed=wl.seed_base + 500 + i, device="cuda")
          for i in range(3)]
    ws = L.Workspace(wl.shape)
    eager = [L.forward(dl, x, ws).clone() for dl, x in zip(layers, xs)]
    outs = [torch.empty_like(x) for x in xs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for dl, x, o in zip(layers, xs, outs):
            L.forward(dl, x, ws, out=o)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="global"):
        for dl, x, o in zip(layers, xs, outs):
            L.forward(dl, x, ws, out=o)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert ws.status() == 0


@pytest.mark.parametrize("name,layer,rows", [("decode_h2048_e128", 0, 1),
                                             ("decode_h2048_e128", 47, 1),
                                             ("verify_h4096_e256", 3, 2),
                                             ("sweep_h4096_e160", 7, 1),
                                             ("prefill8_h2048_e512", 3, 1)])
def test_full_size_t_layout_vs_oracle(name, layer, rows):
    """Down projections in the t layout (the fused one-row form) at the
    workloads' full sizes; union mode byte-identical to per-row mode."""
    wl = synth.WORKLOADS[name]
    weights = synth.make_layer(wl.shape, wl.seed_base + layer, device="cuda")
    x = synth.make_rows(wl.shape, rows, seed=wl.seed_base + 500 + layer, device="cuda",
                        corr=wl.corr)
    dl = L.DeviceLayer(weights, t_layout=True)
    res = G.gpu_run(weights, x, dl=dl)
    st = G.check_parity(weights, x, res)
    print(name, layer, rows, "t layout", st)
    pr = G.gpu_run(weights, x, per_row=True, dl=dl)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))
