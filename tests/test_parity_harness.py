"""The GPU parity checker (tests/gpu_util.py) on the CPU.

The GPU tests pass or fail on check_parity / compare_ids / check_union.
These tests give the checker the oracle's own result dressed as a GPU
result, which it must accept, and then that result with one planted error
(a wrong expert, a routing weight or an output just past its tolerance, a
wrong union entry or row mask, a device status), which it must reject.  A
swap of two experts whose keys tie exactly is accepted as a near tie only
where the case allows one, and that row's weights and output are then still
compared, with the oracle evaluated at the swapped selection."""
import copy

import numpy as np
import pytest
import torch

from oracle import oracle
from routed_moe_decode_router_gb300 import synth
from tests import gpu_util as G

SHAPE = synth.MoeShape(hidden=128, num_experts=16, top_k=4, moe_inter=128, shared_inter=128)


def _as_gpu_result(weights, x):
    orc = G.oracle_run(weights, x)
    ids = orc["ids"]
    U, uni, slot2u, rowmask = oracle.union(ids)
    rows, k = ids.shape
    uslot = [[0xFF] * 8 for _ in range(U)]
    for r in range(rows):
        for j in range(k):
            uslot[slot2u[r, j]][r] = j
    res = {
        "out": torch.from_numpy(orc["out"]).to(torch.bfloat16),
        "ids": ids.copy(),
        "wts": orc["wts"].astype(np.float32),
        "uni": {"U": int(U), "expert": [int(v) for v in uni],
                "rowmask": [int(v) for v in rowmask],
                "slot2u": [int(v) for v in slot2u.ravel()], "uslot": uslot,
                "rows": rows, "top_k": k, "per_row_mode": 0},
        "status": 0,
    }
    return res, orc


@pytest.fixture(scope="module")
def case():
    weights = synth.make_layer(SHAPE, seed=41)
    x = synth.make_rows(SHAPE, 3, seed=42)
    res, orc = _as_gpu_result(weights, x)
    return weights, x, res, orc


def test_accepts_the_oracle_result(case):
    weights, x, res, orc = case
    st = G.check_parity(weights, x, res, orc)
    assert st["tied_rows"] == [] and st["out_rel_l2"] < 5e-3


def _rejects(case, mutate):
    weights, x, res, orc = case
    bad = copy.deepcopy(res)
    mutate(bad, orc)
    with pytest.raises(AssertionError):
        G.check_parity(weights, x, bad, orc)


def test_rejects_a_wrong_expert(case):
    def m(bad, orc):
        keys = G.oracle_keys(case[0], orc["logits"])
        bad["ids"][1, 2] = int(np.argmin(keys[1]))     # far from any tie
    _rejects(case, m)


def test_rejects_a_routing_weight_past_1e6(case):
    def m(bad, orc):
        bad["wts"][0, 1] = np.float32(orc["wts"][0, 1] * (1 + 3e-6))
    _rejects(case, m)


def test_rejects_an_output_past_max_abs(case):
    def m(bad, orc):
        bad["out"][2, 5] += 0.05
    _rejects(case, m)


def test_rejects_an_output_past_rel_l2(case):
    def m(bad, orc):
        bad["out"] = (bad["out"].float() * 1.01).to(torch.bfloat16)
    _rejects(case, m)


def test_rejects_a_wrong_union(case):
    def m(bad, orc):
        e = bad["uni"]["expert"]
        e[0], e[1] = e[1], e[0]
    _rejects(case, m)


def test_rejects_a_wrong_rowmask(case):
    def m(bad, orc):
        bad["uni"]["rowmask"][0] ^= 0b100
    _rejects(case, m)


def test_rejects_a_device_status(case):
    def m(bad, orc):
        bad["status"] = 1
    _rejects(case, m)


def test_near_tie_accepted_only_when_keys_tie():
    """Experts 3 and 9 get identical router rows, so their logits tie
    exactly and the oracle orders them 3 then 9; a GPU result with 9 then 3
    is a near tie.  Swapping two experts whose keys differ is an error."""
    weights, x, res, orc, r = _tied_case()
    ids = res["ids"].copy()
    a, b = list(ids[r]).index(3), list(ids[r]).index(9)
    ids[r, a], ids[r, b] = 9, 3
    same, tied = G.compare_ids(weights, x, ids, orc["ids"], orc["logits"])
    assert tied == [r] and r not in same
    keys = G.oracle_keys(weights, orc["logits"])
    j0, j1 = 0, 1
    if {int(ids[r, j0]), int(ids[r, j1])} == {3, 9}:
        j0, j1 = 1, 2
    ids2 = res["ids"].copy()
    ids2[r, j0], ids2[r, j1] = ids2[r, j1], ids2[r, j0]
    assert keys[r, ids2[r, j0]] != keys[r, ids2[r, j1]]
    with pytest.raises(AssertionError):
        G.compare_ids(weights, x, ids2, orc["ids"], orc["logits"])


def _tied_case():
    weights = synth.make_layer(SHAPE, seed=43)
    weights.router_bf16[3] = weights.router_bf16[3] * 4   # make both likely winners
    weights.router_bf16[9] = weights.router_bf16[3]
    x = synth.make_rows(SHAPE, 2, seed=44)
    res, orc = _as_gpu_result(weights, x)
    rows_with_both = [r for r in range(2) if {3, 9} <= set(int(v) for v in orc["ids"][r])]
    assert rows_with_both, orc["ids"]
    return weights, x, res, orc, rows_with_both[0]


def _swap_tied(res, r):
    """The result with experts 3 and 9 (and their weights) swapped in row r,
    as an fp32 router that resolved the exact tie the other way would give."""
    bad = copy.deepcopy(res)
    ids = bad["ids"]
    a, b = list(ids[r]).index(3), list(ids[r]).index(9)
    ids[r, a], ids[r, b] = 9, 3
    bad["wts"][r, a], bad["wts"][r, b] = res["wts"][r, b], res["wts"][r, a]
    U, uni, slot2u, rowmask = oracle.union(ids)
    uslot = [[0xFF] * 8 for _ in range(U)]
    for rr in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            uslot[slot2u[rr, j]][rr] = j
    bad["uni"].update(U=int(U), expert=[int(v) for v in uni], rowmask=[int(v) for v in rowmask],
                      slot2u=[int(v) for v in slot2u.ravel()], uslot=uslot)
    return bad


def test_near_tie_row_is_still_compared():
    """The swapped row passes only where the case allows a near tie, and its
    weights and output are compared with the oracle at the GPU's selection:
    a wrong output or weight on that row is rejected."""
    weights, x, res, orc, r = _tied_case()
    tied = _swap_tied(res, r)
    st = G.check_parity(weights, x, tied, orc, max_tied=1)
    assert st["tied_rows"] == [r]
    with pytest.raises(AssertionError):
        G.check_parity(weights, x, tied, orc)           # this case allows none
    bad = copy.deepcopy(tied)
    bad["out"][r, 7] += 0.05
    with pytest.raises(AssertionError):
        G.check_parity(weights, x, bad, orc, max_tied=1)
    bad = copy.deepcopy(tied)
    a = list(bad["ids"][r]).index(9)
    bad["wts"][r, a] = np.float32(bad["wts"][r, a] * (1 + 3e-6))
    with pytest.raises(AssertionError):
        G.check_parity(weights, x, bad, orc, max_tied=1)
