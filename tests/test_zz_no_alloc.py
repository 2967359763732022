"""moe_forward_static: the forward for callers that cannot allocate device
memory (for example a plug-in inside a host framework that owns every
device allocation, or a path that must never enter the CUDA allocator).  Its
scratch is the library's own static device array, so the caller passes only
inputs and outputs.

The test calls it through the C ABI twice in a row -- on two different layers
and row counts, so the second call runs on the array the first one left
behind -- and checks each output against moe_forward with a caller-owned
workspace, within the parity tolerance of the other GPU tests.  This file
sorts last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process."""
import numpy as np
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


def _close(a: torch.Tensor, b: torch.Tensor):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    assert rel <= G.OUT_REL_L2, rel
    assert np.abs(x - y).max() <= G.OUT_MAX_ABS


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
        got = torch.full_like(x, float("nan"))
        N.moe_forward_static(dl.cfg, dl.weights, x.data_ptr(), got.data_ptr(), rows, stream)
        torch.cuda.synchronize()
        assert ws.status() == 0
        _close(got, want)


def test_static_workspace_refuses_bad_config():
    cfg = L.make_config(synth.WORKLOADS["tiny_h256_e16"].shape)
    cfg.top_k = 0
    with pytest.raises(N.MoeError):
        N.moe_forward_static(cfg, N.MoeWeights(), 0, 0, 1, 0)
