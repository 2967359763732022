"""A seeded sweep of random layer configurations on the GPU: every feature at
once (hidden, experts, top-k, intermediate widths, softmax or sigmoid
scoring with or without renormalisation, bf16 or NVFP4 router, shared
expert gated, plain or absent, NVFP4 / FP8 / BF16 experts, the t layout, the
GEMV lever, 1 to 32 rows), each forward checked against the oracle and,
where the mode has a per-row twin, union mode byte-identical to per-row
mode.  The configuration draw uses Python's own seeded generator, so the
list of cases is fixed."""
import random

import pytest
import torch

from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

N_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def draw(seed: int):
    """(shape, rows, t_layout, gemv, corr) of case `seed`; all within the
    library's limits (FP8 / BF16 down tiles beyond the ring come in K-parts)."""
    rnd = random.Random(1000 + seed)
    fmt = rnd.choice(["nvfp4", "nvfp4", "fp8", "bf16"])
    H = rnd.choice([128, 256, 384, 512, 768, 1024, 2048])
    E = rnd.choice([1, 2, 5, 8, 16, 24, 40, 64, 100, 128, 160, 256, 300, 512])
    k = rnd.randint(1, min(E, 16))
    widths = [128, 256, 384, 512, 768, 1024, 1536, 2048]
    I, Is = rnd.choice(widths), rnd.choice(widths)
    sigm = rnd.random() < 0.4
    shape = synth.MoeShape(
        hidden=H, num_experts=E, top_k=k, moe_inter=I, shared_inter=Is,
        scoring="sigmoid" if sigm else "softmax",
        norm_topk_prob=rnd.random() < 0.7,
        routed_scaling_factor=rnd.choice([1.0, 1.5, 2.5]) if sigm else 1.0,
        router_fmt=rnd.choice(["bf16", "nvfp4"]),
        has_shared=rnd.random() < 0.8, shared_gated=rnd.random() < 0.7,
        expert_fmt=fmt)
    t_layout = fmt == "nvfp4" and rnd.random() < 0.3
    gemv = fmt == "nvfp4" and rnd.random() < 0.3
    rows = rnd.randint(1, min(32, 256 // k))
    if t_layout:
        rows = min(rows, 4)
    # keep the oracle's fp64 work per case to about a second
    while rows > 1 and rows * (k + 1) * 3 * H * max(I, Is) > 2e9:
        rows //= 2
    corr = rnd.choice([None, 0.5, 0.9])
    return shape, rows, t_layout, gemv, corr


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_config_vs_oracle(seed):
    shape, rows, t_layout, gemv, corr = draw(seed)
    weights, x = G.make_case(shape, rows, seed_w=3000 + seed, seed_x=4000 + seed, corr=corr)
    dl = L.DeviceLayer(weights, t_layout=t_layout)
    res = G.gpu_run(weights, x, dl=dl, gemv=gemv)
    # a random router can put two experts within the fp32 error bound of
    # each other; such a row is still checked at the GPU's own selection
    st = G.check_parity(weights, x, res, max_tied=1)
    print(seed, shape, rows, "t" if t_layout else "-", "gemv" if gemv else "-", st)
    pr = G.gpu_run(weights, x, dl=dl, per_row=True, gemv=gemv)
    assert torch.equal(res["out"].view(torch.int16), pr["out"].view(torch.int16))
