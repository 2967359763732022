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


@pytest.mark.parametrize("fmt,per_weight", [("fp8", 1), ("bf16", 2)])
def test_layer_bytes_other_expert_formats(fmt, per_weight):
    """FP8 / BF16 experts: 1 / 2 bytes per weight and no block scales; the
    router and the rest are unchanged."""
    import dataclasses

    import bench
    from routed_moe_decode_router_gb300 import synth
    shape = dataclasses.replace(synth.WORKLOADS["decode_h2048_e128"].shape, expert_fmt=fmt)
    per_expert = 3 * 2048 * 768 * per_weight + 12
    want = 9 * per_expert + 128 * 2048 * 9 // 16 + 4 + 2048 * 2 + 2 * 2048 * 2
    assert bench.layer_bytes(shape, 1, 8) == want


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


class _FakeSmi:
    """Stands in for the nvidia-smi child process of ClockSampler."""

    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def kill(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_sampler_median_max_and_reasons():
    import bench
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi(
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1980, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 2070, 2070, 1000.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "a truncated line\n")
    assert s.stop() == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                        "reasons": ["sw_power_cap"], "samples": 3}
    s.proc = _FakeSmi(
        "0, 1410, 2070, 700.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n"
        "0, 1395, 2070, 690.0, 0x0000000000000048, Active, Active, Not Active, Not Active\n")
    r = s.stop()
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"] and r["sm_mhz"] == 1402.5
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_committed_traffic_keyed_to_kernel_workload_rows_and_sources(tmp_path, monkeypatch):
    import bench
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        "text\nbench-traffic: kernel=moe_layer_kernel workload=decode_h2048_e128 rows=1 "
        "bytes_per_launch=24182016 src=abc123\n"
        "bench-traffic: kernel=moe_layer_kernel workload=decode_h2048_e128 rows=1 layout=t "
        "bytes_per_launch=24100000 src=abc123\n"
        "bench-traffic: kernel=moe_layer_kernel workload=decode_h2048_e128 rows=1 layout=t "
        "variant=no_shared bytes_per_launch=21500000 src=abc123\n")
    (tmp_path / "profiles" / "raw.ncu-rep").write_text(
        "bench-traffic: kernel=moe_layer_kernel workload=w rows=1 bytes_per_launch=1 src=abc123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc123")
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1) == 24182016
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1, True) == 24100000
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1, True, "nvfp4",
                                   "no_shared") == 21500000
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1, True, "nvfp4",
                                   "ungated_shared") is None
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1, False, "fp8") is None
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 8) is None
    assert bench.committed_traffic("moe_layer_kernel", "prefill8_h2048_e512", 1) is None
    assert bench.committed_traffic("moe_route_kernel", "decode_h2048_e128", 1) is None
    assert bench.committed_traffic("moe_layer_kernel", "w", 1) is None   # only .md / .txt
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "def456")  # sources changed
    assert bench.committed_traffic("moe_layer_kernel", "decode_h2048_e128", 1) is None


def test_reference_arm_json_line_on_cpu():
    """`bench.py --impl reference` times the CPU oracle and prints one JSON
    line with the contract's keys; it needs no GPU, so it runs here on the
    small workload."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_h256_e16", "--steps", "3", "--warmup", "3"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is False
    assert d["unit"] == "us/layer-step" and d["value"] > 0
    assert abs(d["ms_per_step"] - d["value"] / 1000.0) < 1e-3
    assert d["config"]["workload"] == "tiny_h256_e16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"],
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    """With two ranks, rank 0 alone times the oracle and prints the line
    (n_gpus = 2); the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    p = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(root, "bench.py"),
                        "--gpus", "2", "--impl", "reference", "--workload", "tiny_h256_e16",
                        "--steps", "3", "--warmup", "3"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_parity_verdict_bar():
    """The bench's parity verdict applies the parity tests' bar: rel-L2 <= 5e-3
    and max-abs <= 3e-2 of the bf16 output against the fp64 oracle."""
    import numpy as np
    import torch
    import bench
    want = np.linspace(-1.0, 1.0, 256).reshape(2, 128)
    ok = bench.parity_verdict([(torch.from_numpy(want).to(torch.bfloat16), want)])
    assert ok["ok"] and ok["layers_checked"] == 1 and ok["max_rel_l2"] < 5e-3
    bad = want.copy()
    bad[1, 7] += 0.05
    v = bench.parity_verdict([(torch.from_numpy(want).to(torch.bfloat16), want),
                              (torch.from_numpy(bad).to(torch.bfloat16), want)])
    assert not v["ok"] and v["max_abs"] > 3e-2


def test_launches_per_layer():
    import bench
    from routed_moe_decode_router_gb300 import synth
    dec = synth.WORKLOADS["decode_h2048_e128"].shape       # top_k 8: 8-row sub-chunks
    assert bench.launches_per_layer(dec, 1, True) == 1
    assert bench.launches_per_layer(dec, 8, False) == 1
    assert bench.launches_per_layer(dec, 16, False) == 3  # two sub-chunks + the union kernel
    assert bench.launches_per_layer(dec, 3, True) == 4    # one launch per row + the union


def test_extra_and_variant_configs_are_well_formed():
    """Every further measured workload names a known workload, a row count the
    library takes (at most 32 rows, rows * top_k <= 256), real MoeShape
    fields, and enough layers that one step streams more distinct weight
    bytes than the 129 MB L2 (so no flush is needed between steps)."""
    import dataclasses

    import bench
    from routed_moe_decode_router_gb300 import synth
    fields = {f.name for f in dataclasses.fields(synth.MoeShape)}
    names = set()
    for ex in bench.EXTRA_CONFIGS + bench.VARIANT_CONFIGS:
        wl = synth.WORKLOADS[ex.workload]
        assert all(k in fields for k, _ in ex.shape)
        shape = dataclasses.replace(wl.shape, expert_fmt=ex.fmt, **dict(ex.shape))
        assert 1 <= ex.rows <= 32 and ex.rows * shape.top_k <= 256
        assert not (ex.t_layout and ex.fmt != "nvfp4")
        weights = ex.layers * (bench.layer_bytes(shape, ex.rows, shape.top_k)
                               - 2 * ex.rows * shape.hidden * 2)
        assert weights > 129e6, ex
        key = (ex.workload, ex.rows, ex.t_layout, ex.fmt, ex.gemv, ex.shape, ex.corr_from)
        assert key not in names
        names.add(key)
    assert all(ex.variant for ex in bench.VARIANT_CONFIGS)
    assert not any(ex.variant for ex in bench.EXTRA_CONFIGS)
