"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded bytes, plus the union-sweep == per-row byte identity the
forward_moe page reports for its probes.  Tolerances live in gpu_util."""
import numpy as np
import pytest
import torch

from oracle import oracle
from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import native as N
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def S(**kw):
    base = dict(hidden=512, num_experts=32, top_k=8, moe_inter=256, shared_inter=384)
    base.update(kw)
    return synth.MoeShape(**base)


TINY = synth.WORKLOADS["tiny_h256_e16"].shape

SMALL_SHAPES = {
    "tiny": TINY,
    "softmax_is_ne_i": S(),
    "sigmoid_bias": S(num_experts=64, top_k=6, moe_inter=256, shared_inter=256,
                      scoring="sigmoid", routed_scaling_factor=2.5),
    "nvfp4_router": S(hidden=1024, num_experts=48, moe_inter=384, shared_inter=256,
                      router_fmt="nvfp4"),
    "no_norm": S(norm_topk_prob=False),
    "ungated_shared": S(shared_gated=False),
    "no_shared": S(has_shared=False),
    "top1": S(top_k=1),
    "h4096_maxc4": S(hidden=4096, num_experts=16, top_k=4, moe_inter=128, shared_inter=128),
    "h3072_maxc3": S(hidden=3072, num_experts=16, top_k=2, moe_inter=256, shared_inter=128),
    "i1536_down_w6": S(hidden=256, num_experts=16, top_k=4, moe_inter=1536, shared_inter=1536),
    "i4096_down_max": S(hidden=256, num_experts=8, top_k=2, moe_inter=4096, shared_inter=128),
    "e1024_two_lists": S(hidden=256, num_experts=1024, top_k=8, moe_inter=128, shared_inter=128),
    "e600_sigmoid_no_norm": S(hidden=384, num_experts=600, top_k=6, moe_inter=128,
                              shared_inter=256, scoring="sigmoid", routed_scaling_factor=1.5,
                              norm_topk_prob=False),
    "e300_softmax_no_norm": S(hidden=256, num_experts=300, top_k=5, moe_inter=256,
                              shared_inter=128, norm_topk_prob=False),
    # 64-row down units with 4-chunk routed and 2-chunk shared intermediates
    "wide_down_mixed": S(hidden=512, num_experts=32, top_k=8, moe_inter=512, shared_inter=256),
    # 32-row down units split four chunk groups to a tile (8 and 16 chunks)
    "split_down_mixed": S(hidden=512, num_experts=16, top_k=4, moe_inter=1024, shared_inter=2048),
}


@pytest.mark.parametrize("name", list(SMALL_SHAPES))
@pytest.mark.parametrize("rows", [1, 3, 8])
def test_small_shapes_vs_oracle(name, rows):
    shape = SMALL_SHAPES[name]
    if rows * shape.top_k > 64:
        rows = 64 // shape.top_k
    corr = 0.7 if shape.scoring == "sigmoid" else None
    weights, x = G.make_case(shape, rows, seed_w=11, seed_x=12, corr=corr)
    res = G.gpu_run(weights, x)
    G.check_parity(weights, x, res)


@pytest.mark.parametrize("rows", range(1, 9))
@pytest.mark.parametrize("seed", range(4))
def test_tiny_all_rows_and_seeds(rows, seed):
    weights, x = G.make_case(TINY, rows, seed_w=seed, seed_x=500 + seed)
    res = G.gpu_run(weights, x)
    G.check_parity(weights, x, res)
    res_pr = G.gpu_run(weights, x, per_row=True)
    assert torch.equal(res["out"].view(torch.int16), res_pr["out"].view(torch.int16))


def test_top_k_64_single_row():
    shape = S(num_experts=128, top_k=64, moe_inter=128, shared_inter=128)
    weights, x = G.make_case(shape, 1, seed_w=3, seed_x=4)
    res = G.gpu_run(weights, x)
    G.check_parity(weights, x, res)


DEGENERATE_SHAPES = {
    # every expert selected: the union is all E experts, the weights the
    # whole normalised score vector in descending order
    "k_eq_e_softmax": S(hidden=256, num_experts=16, top_k=16, moe_inter=128, shared_inter=128),
    "k_eq_e_sigmoid_no_norm": S(hidden=256, num_experts=16, top_k=16, moe_inter=128,
                                shared_inter=256, scoring="sigmoid", routed_scaling_factor=2.5,
                                norm_topk_prob=False),
    # a single expert: weight exactly 1 (norm) or its score (no norm)
    "one_expert": S(hidden=256, num_experts=1, top_k=1, moe_inter=128, shared_inter=128),
    "one_expert_sigmoid_no_norm": S(hidden=256, num_experts=1, top_k=1, moe_inter=256,
                                    shared_inter=128, scoring="sigmoid",
                                    routed_scaling_factor=1.5, norm_topk_prob=False),
}


@pytest.mark.parametrize("name", list(DEGENERATE_SHAPES))
@pytest.mark.parametrize("rows", [1, 4, 8])
def test_degenerate_routing_vs_oracle(name, rows):
    """Routings with no choice left (k = E, or E = 1): oracle parity, every
    row's union is all E experts, and the union sweep is byte-identical to
    the per-row mode."""
    shape = DEGENERATE_SHAPES[name]
    rows = min(rows, 64 // shape.top_k)
    weights, x = G.make_case(shape, rows, seed_w=91, seed_x=92)
    res = G.gpu_run(weights, x)
    G.check_parity(weights, x, res)
    assert res["uni"]["U"] == shape.num_experts
    assert all(m == (1 << rows) - 1 for m in res["uni"]["rowmask"][:shape.num_experts])
    for r in range(rows):
        assert sorted(res["ids"][r]) == list(range(shape.num_experts))
    if shape.num_experts == 1 and shape.norm_topk_prob:
        assert np.all(res["wts"] == 1.0)
    pr = G.gpu_run(weights, x, per_row=True)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "sigmoid_bias", "nvfp4_router", "no_shared",
                                  "i1536_down_w6"])
@pytest.mark.parametrize("seed", range(6))
def test_union_sweep_byte_identical_to_per_row(name, seed):
    """The forward_moe page reports the union sweep byte-identical to the
    per-row path on six probes; here every seed is a probe."""
    shape = SMALL_SHAPES[name]
    rows = min(8, 64 // shape.top_k)
    weights, x = G.make_case(shape, rows, seed_w=100 + seed, seed_x=200 + seed, corr=0.8)
    a = G.gpu_run(weights, x)
    b = G.gpu_run(weights, x, per_row=True)
    assert a["uni"]["U"] < rows * shape.top_k or rows == 1
    assert b["uni"]["U"] == rows * shape.top_k
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["wts"], b["wts"])


def test_route_stage_logits_ids_weights():
    shape = SMALL_SHAPES["sigmoid_bias"]
    weights, x = G.make_case(shape, 5, seed_w=21, seed_x=22, corr=0.5)
    dl = L.DeviceLayer(weights)
    ws = L.Workspace(shape)
    ids, wts, logits = L.route(dl, x, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ol = oracle.OracleLayer(weights, experts=())
    o_logits, o_ids, o_wts = ol.route(x)
    bound = G.logit_error_bound(weights, x)
    err = np.abs(logits.cpu().numpy().astype(np.float64) - o_logits)
    assert np.all(err <= bound), (err / bound).max()
    same, _ = G.compare_ids(weights, x, ids.cpu().numpy(), o_ids, o_logits)
    w = wts.cpu().numpy().astype(np.float64)[same]
    assert np.all(np.abs(w - o_wts[same]) <= G.WTS_RTOL * np.abs(o_wts[same]))


@pytest.mark.parametrize("per_row", [False, True])
def test_union_stage_vs_oracle(per_row):
    """moe_union on up to 32 rows (256 ids, four blocks of 64): the union
    sequence, row masks and slot map bit-exact against the oracle's."""
    rng = np.random.default_rng(7)
    shape = S(num_experts=40, top_k=8)
    cfg = L.make_config(shape, per_row_mode=per_row)
    ws = L.Workspace(shape)
    for rows in list(range(1, 9)) + [9, 12, 16, 23, 32]:
        for _ in range(5):
            pool = rng.choice(40, size=12, replace=False)   # overlapping rows
            ids = np.stack([rng.choice(pool, 8, replace=False) for _ in range(rows)])
            ids = ids.astype(np.int32)
            uni = L.union(None, cfg, torch.from_numpy(ids).cuda(), ws)
            G.check_union(uni, ids, 8, per_row, None if per_row else oracle.union(ids))
    torch.cuda.synchronize()
    assert ws.status() == 0


def test_device_status_on_bad_expert_id():
    shape = S(num_experts=40, top_k=8)
    cfg = L.make_config(shape)
    ws = L.Workspace(shape)
    ids = torch.arange(16, dtype=torch.int32, device="cuda").reshape(2, 8)
    ids[1, 3] = 40 + 5
    L.union(None, cfg, ids, ws)
    torch.cuda.synchronize()
    assert ws.status() == 1          # MOE_DEV_BAD_EXPERT_ID, context still usable
    assert ws.status() == 0          # cleared by the read
    torch.zeros(1, device="cuda").add_(1)
    torch.cuda.synchronize()


def test_grid_barrier_timeout_sets_status_and_context_survives():
    """A bounded wait that runs out records MOE_DEV_WAIT_TIMEOUT and the
    context stays usable.  In a fresh workspace the first launch (ticket 0)
    runs its grid barriers on counter 0 (header offset 24), which is skewed
    to G - 1: the first CTA at barrier 1 completes it and the other G - 1
    wait for arrivals that never come; their waits run out after about two
    seconds, they skip the rest of the layer, and the launch ends.  The same
    workspace then computes the layer correctly twice more with no
    re-initialisation: the next launch uses counter 1, which the failed
    launch zeroed, and the one after it counter 0 again, zeroed by its
    predecessor."""
    weights, x = G.make_case(TINY, 2, seed_w=31, seed_x=32)
    ws = L.Workspace(TINY)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    torch.cuda.synchronize()
    assert int(ws.buf[16:24].view(torch.int64).item()) == 0      # launch ticket
    ws.buf[24:32].view(torch.int64).fill_(grid - 1)
    dl = L.DeviceLayer(weights)
    L.forward(dl, x, ws)
    torch.cuda.synchronize()
    assert ws.status() == 3          # MOE_DEV_WAIT_TIMEOUT
    assert ws.status() == 0          # cleared by the read
    assert int(ws.buf[16:24].view(torch.int64).item()) == grid  # one ticket per CTA
    for _ in range(2):
        res = G.gpu_run(weights, x, ws=ws, dl=dl)
        G.check_parity(weights, x, res)


def test_workspace_reuse_across_row_counts():
    shape = SMALL_SHAPES["softmax_is_ne_i"]
    weights = synth.make_layer(shape, 31, device="cuda")
    dl = L.DeviceLayer(weights)
    ws = L.Workspace(shape)
    outs = {}
    for rows in (8, 1, 5, 8, 1):
        x = synth.make_rows(shape, rows, seed=40 + rows, device="cuda")
        o = L.forward(dl, x, ws).clone()
        if rows in outs:
            assert torch.equal(o.view(torch.int16), outs[rows].view(torch.int16))
        outs[rows] = o
        fresh = G.gpu_run(weights, x, dl=dl)
        assert torch.equal(o.view(torch.int16), fresh["out"].view(torch.int16))
    torch.cuda.synchronize()
    assert ws.status() == 0


def test_cuda_graph_capture_matches_eager():
    """Three layers captured into one CUDA graph (global capture mode: any
    host synchronisation inside moe_forward would fail the capture) replay to
    the eager bytes."""
    shape = SMALL_SHAPES["sigmoid_bias"]
    layers = [L.DeviceLayer(synth.make_layer(shape, 50 + i, device="cuda")) for i in range(3)]
    ws = L.Workspace(shape)
    xs = [synth.make_rows(shape, 4, seed=60 + i, device="cuda", corr=0.7) for i in range(3)]
    eager = [L.forward(dl, x, ws).clone() for dl, x in zip(layers, xs)]
    outs = [torch.empty_like(x) for x in xs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for dl, x, o in zip(layers, xs, outs):      # warm up on the side stream
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


def test_layer_chain_on_one_stream_matches_single_calls():
    """Back-to-back layers on one stream (programmatic dependent launch
    overlaps each kernel's prologue with its predecessor) give the bytes of
    isolated calls, with each layer consuming the previous one's output."""
    shape = SMALL_SHAPES["nvfp4_router"]
    layers = [L.DeviceLayer(synth.make_layer(shape, 70 + i, device="cuda")) for i in range(4)]
    ws = L.Workspace(shape)
    x0 = synth.make_rows(shape, 6, seed=80, device="cuda")
    h = x0
    chain = []
    for dl in layers:
        h = L.forward(dl, h * 8, ws)         # rescale so routing stays informative
        chain.append(h)
    torch.cuda.synchronize()
    h = x0
    for dl, c in zip(layers, chain):
        torch.cuda.synchronize()
        h = L.forward(dl, h * 8, L.Workspace(shape))
        torch.cuda.synchronize()
        assert torch.equal(h.view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("name", list(SMALL_SHAPES))
def test_gemv_lever_one_row_vs_oracle(name):
    """The one-row CUDA-core GEMV variant (gemv_lever = 1, the forward_ep.rs
    page's runtime choice between its one-row GEMV kernels): oracle parity,
    and union mode byte-identical to per-row mode within the variant."""
    shape = SMALL_SHAPES[name]
    corr = 0.7 if shape.scoring == "sigmoid" else None
    for seed in range(2):
        weights, x = G.make_case(shape, 1, seed_w=61 + seed, seed_x=62 + seed, corr=corr)
        res = G.gpu_run(weights, x, gemv=True)
        G.check_parity(weights, x, res)
        pr = G.gpu_run(weights, x, per_row=True, gemv=True)
        assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))


def test_gemv_lever_ignored_above_one_row():
    shape = SMALL_SHAPES["softmax_is_ne_i"]
    weights, x = G.make_case(shape, 4, seed_w=63, seed_x=64)
    a = G.gpu_run(weights, x)
    b = G.gpu_run(weights, x, gemv=True)
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16))


def test_gemv_lever_applies_to_a_one_row_last_sub_chunk():
    """gemv_lever is taken per sub-chunk: in a 9-row call at top_k 8 (8-row
    sub-chunks) the first eight rows have the tensor-core bytes and the ninth
    row, a sub-chunk of its own, the bytes of a one-row GEMV call."""
    shape = PREFILL_SHAPES["k8"]
    weights, x = G.make_case(shape, 9, seed_w=65, seed_x=66, corr=0.4)
    dl = L.DeviceLayer(weights)
    lev = G.gpu_run(weights, x, dl=dl, gemv=True)
    G.check_parity(weights, x, lev)
    head = G.gpu_run(weights, x[:8].contiguous(), dl=dl)["out"]
    tail = G.gpu_run(weights, x[8:].contiguous(), dl=dl, gemv=True)["out"]
    tail_tc = G.gpu_run(weights, x[8:].contiguous(), dl=dl)["out"]
    assert torch.equal(lev["out"][:8].view(torch.int16), head.view(torch.int16))
    assert torch.equal(lev["out"][8:].view(torch.int16), tail.view(torch.int16))
    assert not torch.equal(tail.view(torch.int16), tail_tc.view(torch.int16))


PREFILL_SHAPES = {
    "k8": S(num_experts=40, top_k=8),
    "k4_sigmoid": S(num_experts=64, top_k=4, moe_inter=256, shared_inter=256,
                    scoring="sigmoid", routed_scaling_factor=2.5),
    "k3": S(num_experts=24, top_k=3, moe_inter=384, shared_inter=128),
}


@pytest.mark.parametrize("name", list(PREFILL_SHAPES))
@pytest.mark.parametrize("rows", [9, 16, 32])
def test_prefill_chunks_beyond_eight_rows(name, rows):
    """Calls of more than one 8-row sub-chunk: oracle parity on every row, the
    call's union (all rows, first-occurrence order across the sub-chunks)
    bit-exact against the oracle's, union mode byte-identical to per-row
    mode, and every row's bytes those of a call holding only its sub-chunk."""
    shape = PREFILL_SHAPES[name]
    rows = min(rows, 256 // shape.top_k)
    corr = 0.7 if shape.scoring == "sigmoid" else 0.4
    weights, x = G.make_case(shape, rows, seed_w=71, seed_x=72, corr=corr)
    dl = L.DeviceLayer(weights)
    res = G.gpu_run(weights, x, dl=dl)
    G.check_parity(weights, x, res)
    assert res["uni"]["rows"] == rows
    pr = G.gpu_run(weights, x, per_row=True, dl=dl)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))
    cr = min(8, 64 // shape.top_k)
    for r0 in range(0, rows, cr):
        sub_out = G.gpu_run(weights, x[r0:r0 + cr].contiguous(), dl=dl)["out"]
        assert torch.equal(sub_out.view(torch.int16),
                           res["out"][r0:r0 + cr].view(torch.int16))
