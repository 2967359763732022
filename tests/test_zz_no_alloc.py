"""moe_forward_static: the forward for callers that cannot allocate device
memory (for example a plug-in inside a host framework that owns every
device allocation, or a path that must never enter the CUDA allocator).  Its
scratch is the library's own static device array, so the caller passes only
inputs and outputs.

The test calls it through the C ABI twice in a row -- on two different layers
and row counts, so the second call runs on the array the first one left
behind -- and checks each output against moe_forward with a caller-owned
workspace.  Both run the same kernel on the same bytes, so the outputs must
be byte-identical (which is tighter than the parity tolerance the other GPU
tests use against the oracle).  This file
sorts last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process."""
import pytest
import torch

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


def test_static_workspace_forward_matches_workspace_forward_twice():
    cases = [(synth.WORKLOADS["verify_h4096_e256"].shape, 3, 2000),
             (synth.WORKLOADS["prefill8_h2048_e512"].shape, 8, 3000)]
    stream = torch.cuda.current_stream().cuda_stream
    for shape, rows, seed in cases:
        weights = synth.make_layer(shape, seed, device="cuda")
        x = synth.make_rows(shape, rows, seed=seed + 500, device="cuda", corr=0.7)
        dl = L.DeviceLayer(weights)
        ws = L.Workspace(shape)
        want = L.forward(dl, x, ws)
        assert ws.status() == 0          # the caller-owned workspace's forward
        got = torch.full_like(x, float("nan"))
        N.moe_forward_static(dl.cfg, dl.weights, x.data_ptr(), got.data_ptr(), rows, stream)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("case", ["t_layout_decode", "fp8_verify"])
def test_static_workspace_other_forms(case):
    """The static scratch also serves the t layout's fused one-row form and
    FP8 experts: byte-identical to moe_forward with a caller workspace."""
    import dataclasses
    if case == "t_layout_decode":
        shape, rows, t = synth.WORKLOADS["decode_h2048_e128"].shape, 1, True
    else:
        shape = dataclasses.replace(synth.WORKLOADS["verify_h4096_e256"].shape, expert_fmt="fp8")
        rows, t = 3, False
    weights = synth.make_layer(shape, 2100, device="cuda")
    x = synth.make_rows(shape, rows, seed=2600, device="cuda", corr=0.7)
    dl = L.DeviceLayer(weights, t_layout=t)
    ws = L.Workspace(shape, t_layout=t)
    want = L.forward(dl, x, ws)
    assert ws.status() == 0
    got = torch.full_like(x, float("nan"))
    N.moe_forward_static(dl.cfg, dl.weights, x.data_ptr(), got.data_ptr(), rows,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_static_workspace_refuses_bad_config():
    cfg = L.make_config(synth.WORKLOADS["tiny_h256_e16"].shape)
    cfg.top_k = 0
    with pytest.raises(N.MoeError):
        N.moe_forward_static(cfg, N.MoeWeights(), 0, 0, 1, 0)
