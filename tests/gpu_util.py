"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded bytes.

Tolerances (written here, used by every parity test):
  ids      bit-exact; a position may differ only where the oracle's own fp64
           selection keys of the two experts lie within the fp32 error bound
           of the GPU router (a near tie).  Each case states how many such
           rows it allows (0 unless stated), and at least one row must match
           the oracle exactly.
  unions   bit-exact (sequence, row masks, slot map) against the oracle's
           union of the GPU's ids.
  weights  relative error <= 1e-6 on every row: a row that matches the
           oracle's selection against the oracle's weights, a near-tie row
           against the oracle evaluated at the GPU's selection.
  output   bf16 out vs the oracle's fp64 out on every row (near-tie rows
           against the oracle at the GPU's selection): relative L2 <= 5e-3
           and max-abs <= 3e-2.
"""
import os

import numpy as np
import torch

from oracle import oracle
from routed_moe_decode_router_gb300 import layer as L
from routed_moe_decode_router_gb300 import synth
from tests import refdecode as ref

WTS_RTOL = 1e-6
OUT_REL_L2 = 5e-3
OUT_MAX_ABS = 3e-2
NTHREADS = max(1, min(16, os.cpu_count() or 1))


def gpu_run(weights, x, per_row=False, ws=None, dl=None, gemv=False, t_layout=False):
    dl = dl or L.DeviceLayer(weights, t_layout=t_layout)
    ws = ws or L.Workspace(weights.shape, t_layout=dl.t_layout)
    rows = x.shape[0]
    out = L.forward(dl, x, ws, per_row_mode=per_row, gemv=gemv)
    ids, wts, uni = L.read_routing(dl, ws, rows, per_row_mode=per_row)
    torch.cuda.synchronize()
    status = ws.status()
    return {"out": out, "ids": ids.cpu().numpy(), "wts": wts.cpu().numpy(), "uni": uni,
            "status": status}


def router_dense(weights):
    s = weights.shape
    if s.router_fmt == "nvfp4":
        m = weights.router_nvfp4
        return ref.nvfp4_dense(m.packed, m.scales, m.scale2)
    return ref.bf16_decode(ref.to_np(weights.router_bf16))


def logit_error_bound(weights, x):
    """Per (row, expert) bound on |fp32 GPU logit - exact logit|: the GPU
    accumulates H/32 products per lane in fp32, then a 5-level shuffle tree
    (plus one rounding of scale2 for an NVFP4 router)."""
    H = weights.shape.hidden
    W = router_dense(weights)
    xd = ref.bf16_decode(ref.to_np(x))
    mag = np.abs(xd) @ np.abs(W).T
    depth = H // 32 + 8
    return depth * 2.0 ** -24 * mag


def oracle_keys(weights, logits):
    s = weights.shape
    if s.scoring == "softmax":
        return logits.copy()
    bias = ref.to_np(weights.bias).astype(np.float64)
    return 1.0 / (1.0 + np.exp(-logits)) + bias


def compare_ids(weights, x, gpu_ids, orc_ids, orc_logits):
    """Rows whose ids match exactly, and the rows that differ only by a
    near tie.  Any other difference fails."""
    bound = logit_error_bound(weights, x)
    keys = oracle_keys(weights, orc_logits)
    sig = weights.shape.scoring == "sigmoid"
    same, tied = [], []
    for r in range(gpu_ids.shape[0]):
        if np.array_equal(gpu_ids[r], orc_ids[r]):
            same.append(r)
            continue
        for j in range(gpu_ids.shape[1]):
            a, b = int(gpu_ids[r, j]), int(orc_ids[r, j])
            if a == b:
                continue
            tol = bound[r, a] + bound[r, b]
            if sig:
                tol = 0.25 * tol + 4e-7
            tol += 2.0 ** -23 * max(abs(keys[r, a]), abs(keys[r, b]))
            assert abs(keys[r, a] - keys[r, b]) <= tol, (
                "row %d slot %d: GPU picked %d, oracle %d; keys %.9g vs %.9g (tol %.3g)"
                % (r, j, a, b, keys[r, a], keys[r, b], tol))
        tied.append(r)
    return same, tied


def first_occurrence_union(ids, per_row):
    flat = [int(v) for v in np.asarray(ids).ravel()]
    if per_row:
        return flat
    return list(dict.fromkeys(flat))


def check_union(gpu_uni, ids, k, per_row, orc_union=None):
    rows = ids.shape[0]
    exp = first_occurrence_union(ids, per_row)
    assert gpu_uni["U"] == len(exp)
    assert gpu_uni["expert"] == exp
    for p in range(rows * k):
        u = gpu_uni["slot2u"][p]
        assert gpu_uni["expert"][u] == int(ids.ravel()[p])
        assert gpu_uni["uslot"][u][p // k] == p % k
    for u in range(gpu_uni["U"]):
        if per_row:
            want = 1 << (u // k)
        else:
            want = sum(1 << r for r in range(rows) if exp[u] in ids[r])
        assert gpu_uni["rowmask"][u] == want
    if orc_union is not None:
        U, uni, slot2u, rowmask = orc_union
        assert gpu_uni["U"] == U
        assert gpu_uni["expert"] == [int(v) for v in uni]
        assert gpu_uni["rowmask"] == [int(v) for v in rowmask]
        assert gpu_uni["slot2u"] == [int(v) for v in slot2u.ravel()]


def oracle_run(weights, x, extra_experts=()):
    """Oracle forward that copies only the experts it (or the GPU) selects."""
    o_route = oracle.OracleLayer(weights, experts=())
    _, ids, _ = o_route.route(x)
    subset = set(int(v) for v in ids.ravel()) | set(int(v) for v in np.ravel(extra_experts))
    ol = oracle.OracleLayer(weights, experts=subset)
    return ol.forward(x, nthreads=NTHREADS)


def oracle_at_ids(weights, x, ids):
    """Oracle forward of rows x with their experts given (ids [rows, k])."""
    ids = np.asarray(ids, dtype=np.int32)
    ol = oracle.OracleLayer(weights, experts=set(int(v) for v in ids.ravel()))
    return ol.forward_ids(x, ids, nthreads=NTHREADS)


def check_parity(weights, x, res, orc=None, max_tied=0):
    """Full comparison of one GPU forward with the oracle; returns stats.
    `max_tied` bounds the rows allowed to differ from the oracle's selection
    by a near tie; those rows' weights and outputs are checked against the
    oracle evaluated at the GPU's selection."""
    assert res["status"] == 0, "device status %d" % res["status"]
    if orc is None:
        orc = oracle_run(weights, x, res["ids"])
    s = weights.shape
    same, tied = compare_ids(weights, x, res["ids"], orc["ids"], orc["logits"])
    assert len(tied) <= max_tied, "near-tie rows %s (this case allows %d)" % (tied, max_tied)
    assert same, "no row matches the oracle's selection"
    per_row = res["uni"]["per_row_mode"] == 1
    check_union(res["uni"], res["ids"], s.top_k, per_row,
                None if per_row else oracle.union(res["ids"]))
    want_w = np.array(orc["wts"], dtype=np.float64, copy=True)
    want_out = np.array(orc["out"], dtype=np.float64, copy=True)
    if tied:
        at = oracle_at_ids(weights, x[tied], res["ids"][tied])
        want_w[tied] = at["wts"]
        want_out[tied] = at["out"]
    w_g = res["wts"].astype(np.float64)
    rel = np.abs(w_g - want_w) / np.abs(want_w)
    assert rel.max() <= WTS_RTOL, "routing weight rel err %.3g" % rel.max()
    got = res["out"].float().cpu().numpy().astype(np.float64)
    rel_l2 = np.linalg.norm(got - want_out) / max(np.linalg.norm(want_out), 1e-30)
    max_abs = np.abs(got - want_out).max()
    assert rel_l2 <= OUT_REL_L2, "out rel-L2 %.3g" % rel_l2
    assert max_abs <= OUT_MAX_ABS, "out max-abs %.3g" % max_abs
    return {"tied_rows": tied, "rows": x.shape[0], "wts_rel": float(rel.max()),
            "out_rel_l2": float(rel_l2), "out_max_abs": float(max_abs)}


def make_case(shape, rows, seed_w, seed_x, corr=None, device="cuda"):
    weights = synth.make_layer(shape, seed_w, device=device)
    x = synth.make_rows(shape, rows, seed_x, device=device, corr=corr)
    return weights, x
