"""The benchmark's multi-process path on CPU: two gloo ranks run the
replica bookkeeping (barrier, max over ranks, whole-job aggregate) that
bench.py uses under torch.distributed.run."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_init("cpu")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier()
    elapsed = 10.0 + 5.0 * rank                 # rank 1 is the slowest
    mx = bench.max_over_ranks(elapsed, "cpu")
    value = bench.aggregate_us_per_unit(mx, units_per_rank=100, world=w)
    bench.barrier()
    q.put((rank, mx, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, value in res:
        assert mx == 15.0
        # 2 ranks x 100 units in 15 ms -> 75 us per unit for the whole job
        assert value == pytest.approx(75.0)


def test_single_process_defaults():
    import bench
    assert bench.dist_init("cpu") == (0, 1, 0)
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.aggregate_us_per_unit(2.0, 4, 1) == 500.0


def test_layer_bytes_decode_matches_closed_form():
    """decode_h2048_e128 at one row with U = 8: 8 experts + shared expert of
    3 * 2048 * 768 NVFP4 weights (9/16 byte each, +12 bytes of scale2), the
    NVFP4 router, the gate vector, x and out."""
    import bench
    from routed_moe_decode_router_gb300 import synth
    shape = synth.WORKLOADS["decode_h2048_e128"].shape
    per_expert = 3 * 2048 * 768 * 9 // 16 + 12
    want = 9 * per_expert + 128 * 2048 * 9 // 16 + 4 + 2048 * 2 + 2 * 2048 * 2
    assert bench.layer_bytes(shape, 1, 8) == want
    assert abs(want / 1e6 - 24.05) < 0.1            # 24.05 MB per decode layer-step


@pytest.mark.parametrize("workload,rows,U,want_mb", [
    # 8 independent rows over E = 512: mean union 60.6 -> 111.2 MB
    ("prefill8_h2048_e512", 8, 60.6, 111.2),
    # one row of the H 4096 / I 1536 sweep: 8 experts -> 96.9 MB
    ("sweep_h4096_e160", 1, 8, 96.9),
    # three verify rows with the live-trace union of 18.76 -> about 142 MB
    ("verify_h4096_e256", 3, 18.76, 142.0),
])
def test_layer_bytes_other_workloads(workload, rows, U, want_mb):
    """Byte counts of the other workloads against hand totals: per union
    expert 3*H*I weights at 9/16 byte plus three fp32 scale2, the shared
    expert likewise plus its bf16 gate vector, a bf16 router E*H*2, the fp32
    bias for sigmoid scoring, and x and out."""
    import bench
    from routed_moe_decode_router_gb300 import synth
    shape = synth.WORKLOADS[workload].shape
    lo, hi = int(U), int(U) + 1
    got = [bench.layer_bytes(shape, rows, u) for u in (lo, hi)]
    mb = (got[0] + (U - lo) * (got[1] - got[0])) / 1e6   # linear in U
    assert abs(mb - want_mb) < 0.15, (mb, want_mb)


def test_layer_bytes_variant_terms():
    """Each optional term enters exactly once: no shared expert, an ungated
    shared expert (no gate vector), an NVFP4 router (9/16 byte per weight +
    scale2), sigmoid scoring (E fp32 bias values)."""
    import bench
    from routed_moe_decode_router_gb300 import synth
    H, E, k, I, Is = 256, 16, 4, 128, 64
    base = synth.MoeShape(H, E, k, I, Is)
    b0 = bench.layer_bytes(base, 2, 5)
    expert = 3 * H * I * 9 // 16 + 12
    shared = 3 * H * Is * 9 // 16 + 12
    assert b0 == 5 * expert + shared + H * 2 + E * H * 2 + 2 * 2 * H * 2
    assert b0 - bench.layer_bytes(synth.MoeShape(H, E, k, I, Is, has_shared=False), 2, 5) \
        == shared + H * 2
    assert b0 - bench.layer_bytes(synth.MoeShape(H, E, k, I, Is, shared_gated=False), 2, 5) \
        == H * 2
    assert b0 - bench.layer_bytes(synth.MoeShape(H, E, k, I, Is, router_fmt="nvfp4"), 2, 5) \
        == E * H * 2 - (E * H * 9 // 16 + 4)
    assert bench.layer_bytes(synth.MoeShape(H, E, k, I, Is, scoring="sigmoid",
                                            routed_scaling_factor=2.5), 2, 5) - b0 == E * 4
    assert bench.layer_bytes(base, 2, 6) - b0 == expert
    assert bench.layer_bytes(base, 3, 5) - b0 == 2 * H * 2
