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
