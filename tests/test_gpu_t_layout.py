"""The t layout (down projections stored input-major) and the fused one-row
form that reads it: the conversion entry point bit-exact against a numpy
transposition of the codes and scales, the layer against the oracle (which
reads the untransposed matrices: the same weights), union mode
byte-identical to per-row mode, every row of a longer call byte-identical
to a one-row call, and the timeout and graph-capture paths."""
import numpy as np
import pytest
import torch

from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import native as N
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G
from tests.test_gpu_parity import DEGENERATE_SHAPES, SMALL_SHAPES, TINY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def t_layout_numpy(packed: np.ndarray, scales: np.ndarray):
    """[C, N, K/2] codes + [C, N, K/16] scales -> [C, K, N/2] + [C, K/16, N]."""
    codes = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), np.uint8)
    codes[..., 0::2] = packed & 0xF
    codes[..., 1::2] = packed >> 4
    ct = np.swapaxes(codes, -1, -2)
    return (ct[..., 0::2] | (ct[..., 1::2] << 4)).copy(), np.swapaxes(scales, -1, -2).copy()


@pytest.mark.parametrize("count,n_out,k_in", [(1, 16, 16), (3, 64, 128), (2, 48, 80),
                                              (5, 2048, 768)])
def test_conversion_bit_exact(count, n_out, k_in):
    g = torch.Generator().manual_seed(count * 1000 + n_out + k_in)
    pk = torch.randint(0, 256, (count, n_out, k_in // 2), generator=g, dtype=torch.uint8)
    sc = torch.randint(0, 256, (count, n_out, k_in // 16), generator=g, dtype=torch.uint8)
    pkd, scd = pk.cuda(), sc.cuda()
    pkt = torch.full((count, k_in, n_out // 2), 0xAA, dtype=torch.uint8, device="cuda")
    sct = torch.full((count, k_in // 16, n_out), 0xAA, dtype=torch.uint8, device="cuda")
    N.moe_nvfp4_to_t_layout(pkd.data_ptr(), scd.data_ptr(), count, n_out, k_in,
                            pkt.data_ptr(), sct.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want_pk, want_sc = t_layout_numpy(pk.numpy(), sc.numpy())
    assert np.array_equal(pkt.cpu().numpy(), want_pk)
    assert np.array_equal(sct.cpu().numpy(), want_sc)


@pytest.mark.parametrize("name", list(SMALL_SHAPES))
def test_small_shapes_one_row_vs_oracle(name):
    shape = SMALL_SHAPES[name]
    corr = 0.7 if shape.scoring == "sigmoid" else None
    for seed in range(2):
        weights, x = G.make_case(shape, 1, seed_w=111 + seed, seed_x=112 + seed, corr=corr)
        res = G.gpu_run(weights, x, t_layout=True)
        G.check_parity(weights, x, res)
        pr = G.gpu_run(weights, x, per_row=True, t_layout=True)
        assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "sigmoid_bias", "nvfp4_router", "no_shared",
                                  "h4096_maxc4", "wide_down_mixed"])
@pytest.mark.parametrize("rows", [3, 8])
def test_rows_are_one_row_calls(name, rows):
    """Each row of a t-layout call is a sub-chunk of its own: oracle parity on
    every row, the call's union that of all its rows, and every row's bytes
    those of a one-row call."""
    shape = SMALL_SHAPES[name]
    rows = min(rows, 256 // shape.top_k)
    weights, x = G.make_case(shape, rows, seed_w=121, seed_x=122, corr=0.7)
    dl = L.DeviceLayer(weights, t_layout=True)
    res = G.gpu_run(weights, x, dl=dl)
    G.check_parity(weights, x, res)
    assert res["uni"]["rows"] == rows
    pr = G.gpu_run(weights, x, per_row=True, dl=dl)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))
    for r in range(rows):
        one = G.gpu_run(weights, x[r:r + 1].contiguous(), dl=dl)["out"]
        assert torch.equal(one.view(torch.int16), res["out"][r:r + 1].view(torch.int16))


@pytest.mark.parametrize("name", list(DEGENERATE_SHAPES))
def test_degenerate_routing_vs_oracle(name):
    shape = DEGENERATE_SHAPES[name]
    weights, x = G.make_case(shape, 2, seed_w=131, seed_x=132)
    res = G.gpu_run(weights, x, t_layout=True)
    G.check_parity(weights, x, res)
    assert res["uni"]["U"] == shape.num_experts
    pr = G.gpu_run(weights, x, per_row=True, t_layout=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "sigmoid_bias", "nvfp4_router", "h4096_maxc4",
                                  "h3072_maxc3"])
def test_gemv_lever_with_t_layout_vs_oracle(name):
    shape = SMALL_SHAPES[name]
    weights, x = G.make_case(shape, 1, seed_w=141, seed_x=142, corr=0.7)
    res = G.gpu_run(weights, x, gemv=True, t_layout=True)
    G.check_parity(weights, x, res)
    pr = G.gpu_run(weights, x, per_row=True, gemv=True, t_layout=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


def test_t_layout_refuses_an_untransposed_sized_workspace():
    """The t layout needs the larger workspace (the per-CTA partial rows)."""
    weights, x = G.make_case(TINY, 1, seed_w=151, seed_x=152)
    dl = L.DeviceLayer(weights, t_layout=True)
    ws = L.Workspace(TINY)
    with pytest.raises(N.MoeError):
        L.forward(dl, x, ws)


def test_grid_barrier_timeout_sets_status_and_context_survives():
    """As for the output-major form: counter 0 of a fresh workspace skewed to
    G - 1, so the first launch's barrier waits run out (MOE_DEV_WAIT_TIMEOUT);
    then the same workspace computes the layer correctly twice more."""
    weights, x = G.make_case(TINY, 1, seed_w=161, seed_x=162)
    ws = L.Workspace(TINY, t_layout=True)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    torch.cuda.synchronize()
    assert int(ws.buf[16:24].view(torch.int64).item()) == 0
    ws.buf[24:32].view(torch.int64).fill_(grid - 1)
    dl = L.DeviceLayer(weights, t_layout=True)
    L.forward(dl, x, ws)
    torch.cuda.synchronize()
    assert ws.status() == 3
    assert ws.status() == 0
    assert int(ws.buf[16:24].view(torch.int64).item()) == grid
    for _ in range(2):
        res = G.gpu_run(weights, x, ws=ws, dl=dl)
        G.check_parity(weights, x, res)


def test_cuda_graph_capture_matches_eager():
    shape = SMALL_SHAPES["sigmoid_bias"]
    layers = [L.DeviceLayer(synth.make_layer(shape, 170 + i, device="cuda"), t_layout=True)
              for i in range(3)]
    ws = L.Workspace(shape, t_layout=True)
    xs = [synth.make_rows(shape, r, seed=180 + r, device="cuda", corr=0.7) for r in (1, 2, 1)]
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


def test_top_k_64_one_row():
    """64 slots: the top-k warp's lanes fetch the pointer entries of slots j
    and j + 32."""
    shape = synth.MoeShape(hidden=512, num_experts=128, top_k=64, moe_inter=128,
                           shared_inter=128)
    weights, x = G.make_case(shape, 1, seed_w=191, seed_x=192)
    res = G.gpu_run(weights, x, t_layout=True)
    G.check_parity(weights, x, res)
    pr = G.gpu_run(weights, x, per_row=True, t_layout=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))
