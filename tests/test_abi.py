"""Host-side tests of the C ABI (no GPU needed): the library loads and
exports every entry point the header declares, the ctypes structures match
the C layout, and every refusal happens on the host before any launch."""
import ctypes as C
import os
import re
import subprocess

import pytest

from routed_moe_decode_router_gb300 import build as B
from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import native as N
from routed_moe_decode_router_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_router.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.lib()


def header_functions():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_library_exports_every_declared_function(lib):
    declared = header_functions()
    assert len(declared) == 13
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(moe_\w+)", out))
    assert set(declared) == exported
    assert set(declared) == set(N.EXPORTS)
    for name in declared:
        assert hasattr(lib, name)


def test_abi_version(lib):
    assert N.moe_abi_version() == 3


def test_ctypes_layout_matches_c_header(tmp_path):
    structs = {"moe_nvfp4": N.Nvfp4Desc, "moe_config": N.MoeConfig,
               "moe_expert_table": N.ExpertTable, "moe_weights": N.MoeWeights,
               "moe_union_table": N.UnionTable}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_router.h"',
             'int main(void) {']
    for cname, py in structs.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (cname, cname))
        for fname, _ in py._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));'
                         % (cname, fname, cname, fname))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True,
                                                  text=True, check=True).stdout.splitlines())
    for cname, py in structs.items():
        assert int(got[cname]) == C.sizeof(py), cname
        for fname, _ in py._fields_:
            assert int(got["%s.%s" % (cname, fname)]) == getattr(py, fname).offset, fname


def good_cfg(**kw):
    c = L.make_config(synth.WORKLOADS["tiny_h256_e16"].shape)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    ("num_experts", 0, N.MoeError),
    ("router_width", 17, N.MoeError),
    ("hidden", 200, N.MoeError),
    ("hidden", 8192, N.MoeError),
    ("top_k", 0, N.MoeError),
    ("top_k", 17, N.MoeError),
    ("moe_inter", 96, N.MoeError),
    ("shared_inter", 64, N.MoeError),
    ("routed_scaling_factor", 2.5, N.MoeError),
    ("scoring", 7, N.MoeError),
    ("router_fmt", 3, N.MoeError),
    ("per_row_mode", 2, N.MoeError),
    ("gemv_lever", 2, N.MoeError),
    ("t_layout", 2, N.MoeError),
    ("expert_fmt", 3, N.MoeError),
    ("expert_fmt", -1, N.MoeError),
])
def test_config_refusals(lib, field, value, status):
    cfg = good_cfg(**{field: value})
    with pytest.raises(status):
        N.moe_check_config(cfg)
    assert N.lib().moe_workspace_size(C.byref(cfg)) == 0


def test_top_k_beyond_one_union_block_refused(lib):
    """A row's top_k ids must fit one 64-id union block."""
    cfg = good_cfg(num_experts=128, router_width=128, top_k=65)
    with pytest.raises(N.MoeError):
        N.moe_check_config(cfg)
    N.moe_check_config(good_cfg(num_experts=128, router_width=128, top_k=64))


def test_zero_computation_router_refused_as_unsupported(lib):
    cfg = good_cfg(router_width=20)
    with pytest.raises(N.MoeError) as ei:
        N.moe_check_config(cfg)
    assert ei.value.status == 2
    assert "zero-computation" in str(ei.value)


def test_sigmoid_accepts_scaling_factor(lib):
    N.moe_check_config(good_cfg(scoring=1, routed_scaling_factor=2.5))


def test_workspace_size_independent_of_rows_and_positive(lib):
    for name, wl in synth.WORKLOADS.items():
        n = N.moe_workspace_size(L.make_config(wl.shape))
        assert n > 0 and n % 256 == 0, name


def test_t_layout_workspace_holds_one_partial_row_per_cta(lib):
    """The t layout adds room for 256 CTAs' partial output rows (fp32)."""
    for name, wl in synth.WORKLOADS.items():
        a = N.moe_workspace_size(L.make_config(wl.shape))
        b = N.moe_workspace_size(L.make_config(wl.shape, t_layout=True))
        assert b - a == 256 * wl.shape.hidden * 4, name


def test_t_layout_needs_nvfp4_experts(lib):
    for fmt in (N.MOE_EXPERT_FP8, N.MOE_EXPERT_BF16):
        N.moe_check_config(good_cfg(expert_fmt=fmt))
        with pytest.raises(N.MoeError) as ei:
            N.moe_check_config(good_cfg(expert_fmt=fmt, t_layout=1))
        assert ei.value.status == 2


def test_fp8_and_bf16_expert_tables_need_no_scales(lib):
    """FP8 / BF16 experts: NULL scale arrays pass the host checks (the call
    then stops at the NULL workspace); NVFP4 experts refuse them."""
    shape = synth.WORKLOADS["tiny_h256_e16"].shape
    for fmt, ok in ((N.MOE_EXPERT_NVFP4, False), (N.MOE_EXPERT_FP8, True),
                    (N.MOE_EXPERT_BF16, True)):
        cfg = good_cfg(expert_fmt=fmt)
        w = fake_weights()
        w.gate = w.up = w.down = N.ExpertTable(FAKE, 0, FAKE)
        d = N.Nvfp4Desc(FAKE, 0, 1.0)
        w.shared_gate_proj = w.shared_up_proj = w.shared_down_proj = d
        with pytest.raises(N.MoeError) as ei:
            N.moe_forward(cfg, w, FAKE, FAKE + (1 << 20), 1, 0, 1 << 20, 0)
        assert ("workspace" in str(ei.value)) == ok, (fmt, str(ei.value))


def test_largest_config_fits_the_static_workspace(lib):
    for t in (0, 1):
        cfg = good_cfg(hidden=4096, num_experts=1024, router_width=1024, top_k=64,
                       moe_inter=4096, shared_inter=4096, t_layout=t)
        N.moe_check_config(cfg)
        assert N.moe_workspace_size(cfg) <= N.MOE_STATIC_WORKSPACE_BYTES


FAKE = 0x10000   # never dereferenced: every check below fails on the host


def fake_weights():
    w = N.MoeWeights()
    w.router_bf16 = FAKE
    tab = N.ExpertTable(FAKE, FAKE, FAKE)
    w.gate = w.up = w.down = tab
    d = N.Nvfp4Desc(FAKE, FAKE, 1.0)
    w.shared_gate_proj = w.shared_up_proj = w.shared_down_proj = d
    w.shared_expert_gate = FAKE
    return w


# case -> (expected status, text the error message must contain)
FORWARD_REFUSALS = {
    "rows0": (1, "rows=0"),
    "rows33": (1, "rows=33"),
    "ids257": (2, "rows*top_k=272 exceeds 256"),
    "x_null": (1, "x: NULL"),
    "x_misaligned": (1, "x: NULL or not 16-byte aligned"),
    "out_null": (1, "out is NULL"),
    "out_misaligned": (1, "out: not 16-byte aligned"),
    "overlap": (1, "x and out overlap"),
    "ws_null": (3, "workspace is NULL"),
    "ws_small": (3, "needs"),
    "ws_misaligned": (3, "256-byte aligned"),
    "router_misaligned": (1, "router_bf16"),
    "nvfp4_router_null": (1, "router_nvfp4: NULL pointer"),
    "table_null": (1, "gate expert table: NULL array"),
    "table_misaligned": (1, "up expert table: misaligned array"),
    "shared_misaligned": (1, "shared_down_proj: packed/scales must be 16-byte aligned"),
    "shared_gate_missing": (1, "shared_gate=1 needs"),
    "bias_missing": (1, "correction_bias"),
}


@pytest.mark.parametrize("case", sorted(FORWARD_REFUSALS))
def test_forward_refusals_on_host(lib, case):
    """Each bad argument is refused by its own check, with its own status and
    message, before anything touches the device (the pointers are fake)."""
    cfg = good_cfg()
    w = fake_weights()
    need = N.moe_workspace_size(cfg)
    x, out, rows, ws, nbytes = 0x200000, 0x400000, 2, 0x800000, need
    if case == "rows0":
        rows = 0
    elif case == "rows33":
        rows = 33
    elif case == "ids257":
        cfg = good_cfg(top_k=16, num_experts=16, router_width=16)
        rows = 17
    elif case == "x_null":
        x = 0
    elif case == "x_misaligned":
        x += 2
    elif case == "out_null":
        out = 0
    elif case == "out_misaligned":
        out += 8
    elif case == "overlap":
        out = x + 256
    elif case == "ws_null":
        ws = 0
    elif case == "ws_small":
        nbytes = need - 1
    elif case == "ws_misaligned":
        ws += 16
    elif case == "router_misaligned":
        w.router_bf16 = FAKE + 2
    elif case == "nvfp4_router_null":
        cfg = good_cfg(router_fmt=1)
        nbytes = N.moe_workspace_size(cfg)
        w.router_nvfp4 = N.Nvfp4Desc(0, FAKE, 1.0)
    elif case == "table_null":
        w.gate = N.ExpertTable(0, FAKE, FAKE)
    elif case == "table_misaligned":
        w.up = N.ExpertTable(FAKE + 4, FAKE, FAKE)
    elif case == "shared_misaligned":
        w.shared_down_proj = N.Nvfp4Desc(FAKE + 8, FAKE, 1.0)
    elif case == "shared_gate_missing":
        w.shared_expert_gate = 0
    elif case == "bias_missing":
        cfg = good_cfg(scoring=1, routed_scaling_factor=2.5)
        nbytes = N.moe_workspace_size(cfg)
    status, text = FORWARD_REFUSALS[case]
    with pytest.raises(N.MoeError) as ei:
        N.moe_forward(cfg, w, x, out, rows, ws, nbytes, 0)
    assert ei.value.status == status, str(ei.value)
    assert text in N.lib().moe_last_error().decode()


@pytest.mark.parametrize("case", ["rows0", "rows33", "x_null", "out_null", "overlap",
                                  "table_null", "shared_misaligned"])
def test_static_forward_refuses_before_any_device_call(lib, case):
    """moe_forward_static checks every argument before it looks up or clears
    its library-owned workspace, so a bad argument comes back as its own
    refusal even on a machine without a GPU (a device call there would fail
    with MOE_ERR_CUDA instead)."""
    cfg = good_cfg()
    w = fake_weights()
    x, out, rows = 0x200000, 0x400000, 2
    if case == "rows0":
        rows = 0
    elif case == "rows33":
        rows = 33
    elif case == "x_null":
        x = 0
    elif case == "out_null":
        out = 0
    elif case == "overlap":
        out = x + 256
    elif case == "table_null":
        w.gate = N.ExpertTable(0, FAKE, FAKE)
    elif case == "shared_misaligned":
        w.shared_down_proj = N.Nvfp4Desc(FAKE + 8, FAKE, 1.0)
    status, text = FORWARD_REFUSALS[case]
    with pytest.raises(N.MoeError) as ei:
        N.moe_forward_static(cfg, w, x, out, rows, 0)
    assert ei.value.status == status, str(ei.value)
    assert text in N.lib().moe_last_error().decode()


def test_route_and_union_refusals_on_host(lib):
    cfg = good_cfg()
    w = fake_weights()
    need = N.moe_workspace_size(cfg)
    with pytest.raises(N.MoeError):
        N.moe_route(cfg, w, 0x200000, 0, 0, 0, 0, 0x800000, need, 0)
    with pytest.raises(N.MoeError):
        N.moe_route(cfg, w, 0x200000, 1, 0x1002, 0, 0, 0x800000, need, 0)
    with pytest.raises(N.MoeError):
        N.moe_union(cfg, None, 0, 1, 0, 0x800000, need, 0)
    with pytest.raises(N.MoeError):
        N.moe_union(cfg, None, 0x1000, 17, 0, 0x800000, need, 0)
    with pytest.raises(N.MoeError):
        N.moe_read_routing(cfg, 0x800001, need, 1, 0, 0, 0, 0)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(N, "_lib", None)
    monkeypatch.setattr(N, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        N.lib()


def _cpu_layer_and_workspaces():
    import types
    import torch
    shape = synth.WORKLOADS["tiny_h256_e16"].shape
    dl = L.DeviceLayer(synth.make_layer(shape, 0), device="cpu")
    # stand-ins with the attributes the helpers read; nothing reaches a GPU
    ws_cpu = types.SimpleNamespace(buf=torch.empty(256, dtype=torch.uint8), ptr=0x800000,
                                   nbytes=1 << 20)
    ws_cuda = types.SimpleNamespace(buf=types.SimpleNamespace(device=torch.device("cuda:0")),
                                    ptr=0x800000, nbytes=1 << 20)
    return shape, dl, ws_cpu, ws_cuda


def test_python_helpers_refuse_host_memory_before_calling_the_library(monkeypatch):
    """layer.forward / route / union refuse tensors that are not in the
    layer's CUDA memory, of the wrong dtype or width, or not contiguous,
    before any pointer reaches the library (a host pointer in a kernel
    would fault the GPU rather than raise)."""
    import torch
    shape, dl, ws_cpu, ws_cuda = _cpu_layer_and_workspaces()
    called = []
    for name in ("moe_forward", "moe_route", "moe_union"):
        monkeypatch.setattr(N, name, lambda *a, _n=name: called.append(_n))
    x = synth.make_rows(shape, 2, seed=1)
    # a workspace in host memory
    with pytest.raises(ValueError, match="CUDA device memory"):
        L.forward(dl, x, ws_cpu)
    # layer on the host, workspace on a CUDA device
    with pytest.raises(ValueError, match="the layer is on cpu"):
        L.forward(dl, x, ws_cuda)
    dl.device = torch.device("cuda:0")          # as if the layer were resident
    with pytest.raises(ValueError, match="x is on cpu"):
        L.forward(dl, x, ws_cuda)
    with pytest.raises(ValueError, match="dtype"):
        L.forward(dl, x.float(), ws_cuda)
    with pytest.raises(ValueError, match="expected \\[rows, 256\\]"):
        L.forward(dl, x[:, :128], ws_cuda)
    with pytest.raises(ValueError, match="expected \\[rows, 256\\]"):
        L.route(dl, x.reshape(-1), ws_cuda)
    with pytest.raises(ValueError, match="contiguous"):
        L.forward(dl, torch.empty((256, 2), dtype=torch.bfloat16).t(), ws_cuda)
    with pytest.raises(ValueError, match="ids has dtype"):
        L.union(None, dl.cfg, torch.zeros((2, 4), dtype=torch.int64), ws_cuda)
    with pytest.raises(ValueError, match="ids is on cpu"):
        L.union(None, dl.cfg, torch.zeros((2, 4), dtype=torch.int32), ws_cuda)
    assert called == []


@pytest.mark.parametrize("case", ["count0", "n_not16", "k_not16", "k_big", "null",
                                  "misaligned", "overlap"])
def test_t_layout_conversion_refusals(lib, case):
    """moe_nvfp4_to_t_layout refuses bad arguments on the host, before any
    CUDA call."""
    A, B, C_, D = 0x100000, 0x200000, 0x300000, 0x400000
    args = dict(packed=A, scales=B, count=2, n_out=64, k_in=128, packed_t=C_, scales_t=D)
    if case == "count0":
        args["count"] = 0
    elif case == "n_not16":
        args["n_out"] = 40
    elif case == "k_not16":
        args["k_in"] = 72
    elif case == "k_big":
        args["k_in"] = 65536 + 16
    elif case == "null":
        args["scales_t"] = 0
    elif case == "misaligned":
        args["packed_t"] = C_ + 8
    elif case == "overlap":
        args["packed_t"] = A + 16
    with pytest.raises(N.MoeError) as ei:
        N.moe_nvfp4_to_t_layout(**args)
    assert ei.value.status == 1
