"""FP8 and BF16 expert matrices on the GPU: oracle parity (the oracle decodes
the same bytes in its own code), union mode byte-identical to per-row mode,
calls of several sub-chunks, degenerate routings, BF16 gate/up tiles taken in
two K-halves (hidden 3584 and 4096), BF16 down tiles in K-parts
(intermediates of 2048 to 4096), the full-size shapes, the refusal of BF16
gate/up tiles that do not fit the shared-memory ring, and CUDA-graph
replay."""
import pytest
import torch

import numpy as np

from oracle import oracle
from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import native as N
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G
from tests.test_gpu_parity import S

pytestmark = pytest.mark.gpu

FORMATS = ["fp8", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def F(fmt, **kw):
    return S(expert_fmt=fmt, **kw)


SHAPES = {
    "base": dict(),
    "tiny": dict(hidden=256, num_experts=16, top_k=4, moe_inter=128, shared_inter=128),
    "sigmoid_bias": dict(num_experts=64, top_k=6, moe_inter=256, shared_inter=256,
                         scoring="sigmoid", routed_scaling_factor=2.5),
    "nvfp4_router": dict(hidden=1024, num_experts=48, moe_inter=384, shared_inter=256,
                         router_fmt="nvfp4"),
    "no_norm_ungated": dict(norm_topk_prob=False, shared_gated=False),
    "no_shared": dict(has_shared=False),
    "wide_down_mixed": dict(hidden=512, num_experts=32, top_k=8, moe_inter=512, shared_inter=256),
    "split_down_mixed": dict(hidden=512, num_experts=16, top_k=4, moe_inter=1024,
                             shared_inter=2048),
    "h2048_maxc2": dict(hidden=2048, num_experts=16, top_k=4, moe_inter=256, shared_inter=128),
    "i1536_down_w6": dict(hidden=256, num_experts=16, top_k=4, moe_inter=1536, shared_inter=1536),
    # BF16: gate/up tiles in two K-halves; at 3584 (28 chunks) a warp's
    # chunks 8 + w straddle the halves
    "h4096_khalves": dict(hidden=4096, num_experts=16, top_k=4, moe_inter=128, shared_inter=256),
    "h3584_khalves": dict(hidden=3584, num_experts=16, top_k=4, moe_inter=256, shared_inter=128,
                          scoring="sigmoid", routed_scaling_factor=2.5),
    # BF16: down units in K-parts of 6 chunks (four 48 KB slots at hidden
    # 512): 32 chunks in parts of 6, 6, 6, 6, 6, 2 beside a 1-chunk shared
    # expert; 18 chunks in three parts; split units of 16 chunks (parts 6,
    # 6, 4) beside split units of 12
    "i4096_dparts": dict(hidden=512, num_experts=16, top_k=4, moe_inter=4096, shared_inter=128),
    "i2304_dparts": dict(hidden=512, num_experts=12, top_k=3, moe_inter=2304, shared_inter=2304),
    "split_dparts": dict(hidden=512, num_experts=16, top_k=2, moe_inter=2048, shared_inter=1536,
                         scoring="sigmoid", routed_scaling_factor=1.5),
}


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("rows", [1, 3, 8])
def test_small_shapes_vs_oracle(fmt, name, rows):
    shape = F(fmt, **SHAPES[name])
    rows = min(rows, 64 // shape.top_k)
    corr = 0.7 if shape.scoring == "sigmoid" else None
    weights, x = G.make_case(shape, rows, seed_w=201, seed_x=202, corr=corr)
    dl = L.DeviceLayer(weights)
    res = G.gpu_run(weights, x, dl=dl)
    G.check_parity(weights, x, res)
    pr = G.gpu_run(weights, x, per_row=True, dl=dl)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("variant", [dict(num_experts=16, top_k=16),
                                     dict(num_experts=1, top_k=1)])
def test_degenerate_routing_vs_oracle(fmt, variant):
    shape = F(fmt, hidden=256, moe_inter=128, shared_inter=128, **variant)
    weights, x = G.make_case(shape, 4, seed_w=211, seed_x=212)
    res = G.gpu_run(weights, x)
    G.check_parity(weights, x, res)
    assert res["uni"]["U"] == shape.num_experts
    pr = G.gpu_run(weights, x, per_row=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
def test_calls_of_several_sub_chunks(fmt):
    """16 rows at top_k 8: two 8-row sub-chunks, each row's bytes those of a
    call holding only its sub-chunk, the call's union that of all rows."""
    shape = F(fmt, num_experts=40, top_k=8)
    weights, x = G.make_case(shape, 16, seed_w=221, seed_x=222, corr=0.4)
    dl = L.DeviceLayer(weights)
    res = G.gpu_run(weights, x, dl=dl)
    G.check_parity(weights, x, res)
    assert res["uni"]["rows"] == 16
    for r0 in (0, 8):
        sub = G.gpu_run(weights, x[r0:r0 + 8].contiguous(), dl=dl)["out"]
        assert torch.equal(sub.view(torch.int16), res["out"][r0:r0 + 8].view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemv_lever_ignored(fmt):
    """The GEMV lever is an NVFP4 variant: other formats give the same bytes
    with it on or off."""
    shape = F(fmt)
    weights, x = G.make_case(shape, 1, seed_w=231, seed_x=232)
    dl = L.DeviceLayer(weights)
    a = G.gpu_run(weights, x, dl=dl)
    b = G.gpu_run(weights, x, dl=dl, gemv=True)
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))


@pytest.mark.parametrize("variant", [
    dict(hidden=3968, moe_inter=128, shared_inter=128),     # 31 chunks: no whole K-halves
])
def test_bf16_tiles_too_large_for_the_ring_are_refused(variant):
    shape = F("bf16", num_experts=8, top_k=2, **variant)
    weights, x = G.make_case(shape, 1, seed_w=241, seed_x=242)
    dl = L.DeviceLayer(weights)
    ws = L.Workspace(shape)
    with pytest.raises(N.MoeError) as ei:
        L.forward(dl, x, ws)
    assert ei.value.status == 2


def test_t_layout_refused_for_fp8():
    weights, _ = G.make_case(F("fp8"), 1, seed_w=251, seed_x=252)
    with pytest.raises(ValueError):
        L.DeviceLayer(weights, t_layout=True)


# full-size shapes of the workloads in the other formats (BF16 at hidden 4096
# with its gate/up tiles in K-halves)
FULL = [("decode_h2048_e128", "fp8", 1), ("decode_h2048_e128", "bf16", 1),
        ("prefill8_h2048_e512", "fp8", 8), ("prefill8_h2048_e512", "bf16", 8),
        ("verify_h4096_e256", "fp8", 3), ("sweep_h4096_e160", "fp8", 8),
        ("verify_h4096_e256", "bf16", 3), ("sweep_h4096_e160", "bf16", 8),
        ("sweep_h4096_e160", "bf16", 1)]


@pytest.mark.parametrize("name,fmt,rows", FULL)
def test_full_size_vs_oracle(name, fmt, rows):
    wl = synth.WORKLOADS[name]
    shape = synth.MoeShape(**{**wl.shape.__dict__, "expert_fmt": fmt})
    weights = synth.make_layer(shape, wl.seed_base + 7, device="cuda")
    x = synth.make_rows(shape, rows, seed=wl.seed_base + 507, device="cuda", corr=wl.corr)
    dl = L.DeviceLayer(weights)
    res = G.gpu_run(weights, x, dl=dl)
    st = G.check_parity(weights, x, res)
    print(name, fmt, rows, st)
    pr = G.gpu_run(weights, x, per_row=True, dl=dl)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
def test_cuda_graph_capture_matches_eager(fmt):
    shape = F(fmt, num_experts=64, top_k=6, moe_inter=256, shared_inter=256,
              scoring="sigmoid", routed_scaling_factor=2.5)
    layers = [L.DeviceLayer(synth.make_layer(shape, 260 + i, device="cuda")) for i in range(3)]
    ws = L.Workspace(shape)
    xs = [synth.make_rows(shape, r, seed=270 + r, device="cuda", corr=0.7) for r in (1, 4, 8)]
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
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert ws.status() == 0


@pytest.mark.parametrize("fmt", FORMATS)
def test_union_stage_with_scale_free_tables(fmt):
    """moe_union with FP8 / BF16 expert tables, whose scale arrays are NULL:
    the pointer entries are fetched without them, the table matches the
    oracle's union and no fault is recorded."""
    shape = F(fmt, num_experts=40, top_k=8)
    weights = synth.make_layer(shape, 281, device="cuda")
    dl = L.DeviceLayer(weights)
    assert dl.weights.gate.scales is None or dl.weights.gate.scales == 0
    ws = L.Workspace(shape)
    rng = np.random.default_rng(282)
    for rows in (1, 5, 16, 32):
        pool = rng.choice(40, size=12, replace=False)
        ids = np.stack([rng.choice(pool, 8, replace=False) for _ in range(rows)]).astype(np.int32)
        uni = L.union(dl, dl.cfg, torch.from_numpy(ids).cuda(), ws)
        G.check_union(uni, ids, 8, False, oracle.union(ids))
    torch.cuda.synchronize()
    assert ws.status() == 0
