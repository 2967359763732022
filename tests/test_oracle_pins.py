"""Pins of the CPU oracle against references other than itself.

Each test checks one oracle function against a library routine (torch's
float8/bfloat16 decoders, numpy/torch fp64 matmul, scipy's softmax and
expit, numpy's lexsort), a published value table, a closed form or an
invariant, so that a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special as sps
import torch

from routed_moe_decode_router_gb300 import synth
from tests import refdecode as ref


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_e2m1_matches_published_table(orc):
    tab = ref.e2m1_table()
    for code in range(16):
        v = orc.e2m1(code)
        assert v == tab[code]
        assert math.copysign(1.0, v) == math.copysign(1.0, tab[code])


def test_e4m3_exhaustive_vs_torch(orc):
    want = ref.e4m3_decode(np.arange(256))
    for code in range(256):
        got = orc.e4m3(code)
        if np.isnan(want[code]):
            assert np.isnan(got), code
        else:
            assert got == want[code], (code, got, want[code])


def test_bf16_decode_exhaustive_vs_torch(orc):
    bits = np.arange(65536, dtype=np.uint32)
    want = ref.bf16_decode(bits.astype(np.uint16))
    got = np.array([orc.bf16(int(b)) for b in bits[::7]])
    w = want[::7]
    nan = np.isnan(w)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], w[~nan])


def test_round_bf16_matches_torch_on_floats(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-38).astype(np.float32),
        (rng.standard_normal(1000) * 1e30).astype(np.float32),
    ])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.round_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_no_double_rounding(orc):
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1 + 2^-7; a hair above
    # it must round up, although rounding to float first would land on the
    # midpoint and tie down to 1.0.
    assert orc.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert orc.round_bf16(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even
    assert orc.round_bf16(-2.5) == 0xC020
    assert orc.round_bf16(1e39) == 0x7F80


def test_round_bf16_edges_vs_torch(orc):
    """The ends of the bf16 range against torch's float32 -> bfloat16
    rounding: the subnormal grid (quantum 2^-133), the largest finite value
    and the ties above it that overflow to infinity, infinities and NaN."""
    sub = np.arange(0, 600, dtype=np.float64) * 2.0 ** -135          # 1/4 of the quantum
    top = np.array([float.fromhex(h) for h in (
        "0x1.fcp127", "0x1.fdp127", "0x1.fep127", "0x1.fe7ffep127", "0x1.fe8p127",
        "0x1.ffp127", "0x1.fffffep127")])
    rng = np.random.default_rng(2)
    tiny = rng.uniform(0, 2.0 ** -125, 2000)
    vals = np.concatenate([sub, -sub, top, -top, tiny, [np.inf, -np.inf]])
    vals = vals.astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.round_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    # NaN stays NaN (all exponent bits set, mantissa not zero); its sign and
    # payload carry no meaning
    b = orc.round_bf16(float("nan"))
    assert b & 0x7F80 == 0x7F80 and b & 0x007F != 0


def test_nvfp4_elem_vs_library_decode(orc):
    rng = np.random.default_rng(2)
    N, K = 24, 96
    packed = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, size=(N, K // 16), dtype=np.uint8)
    scales[(scales & 0x7F) == 0x7F] = 0x38          # keep NaN codes out
    s2 = np.float32(0.0123)
    m = orc.HostMat(packed, scales, s2)
    want = ref.nvfp4_dense(packed, scales, s2)
    got = np.array([[orc.nvfp4_elem(m, n, k) for k in range(K)] for n in range(N)])
    assert np.array_equal(got, want)


def test_fp8_elem_vs_library_decode(orc):
    """FP8 experts: one E4M3 code per weight, row-major, times scale2 (fp32)."""
    rng = np.random.default_rng(4)
    N, K = 24, 80
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x41             # keep NaN codes out
    s2 = np.float32(0.0371)
    m = orc.HostMat(codes, None, s2, "fp8")
    want = ref.fp8_dense(codes, s2)
    got = np.array([[orc.mat_elem(m, n, k) for k in range(K)] for n in range(N)])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("s2", [1.0, 0.73])
def test_bf16_elem_vs_library_decode(orc, s2):
    """BF16 experts: one little-endian bfloat16 per weight, row-major, times
    scale2 (fp32)."""
    rng = np.random.default_rng(5)
    N, K = 16, 48
    bits = rng.integers(0, 1 << 16, size=(N, K), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF         # keep infinities and NaNs out
    raw = bits.astype("<u2").view(np.uint8).reshape(N, 2 * K)
    m = orc.HostMat(raw, None, np.float32(s2), "bf16")
    want = ref.bf16_dense(raw, np.float32(s2))
    got = np.array([[orc.mat_elem(m, n, k) for k in range(K)] for n in range(N)])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", ["fp8", "bf16"])
def test_other_formats_roundtrip(orc, fmt):
    """The FP8 encoder is within half an E4M3 step of the weights and the
    BF16 one within half a bfloat16 step: what the oracle reads back is the
    value the generator meant."""
    g = torch.Generator().manual_seed(6)
    w = torch.randn((8, 64), generator=g) * 0.02
    q = synth.ENCODERS[fmt](w)
    m = orc.HostMat(q.packed, q.scales, q.scale2, fmt)
    deq = np.array([[orc.mat_elem(m, n, k) for k in range(64)] for n in range(8)])
    err = np.abs(deq - w.double().numpy())
    rel = 2.0 ** -4 if fmt == "fp8" else 2.0 ** -8
    assert np.all(err <= rel * np.abs(w.double().numpy()) + 2.0 ** -9 * float(q.scale2))


def test_quantizer_roundtrip_within_grid_step(orc):
    """dequant(quantize(W)) stays within one block step of W; a wrong nibble
    order or scale index would give errors of the size of W itself."""
    g = torch.Generator().manual_seed(3)
    w = torch.randn((16, 128), generator=g) * 0.02
    q = synth.quantize_nvfp4(w)
    m = orc.HostMat(q.packed, q.scales, q.scale2)
    deq = np.array([[orc.nvfp4_elem(m, n, k) for k in range(128)] for n in range(16)])
    step = ref.e4m3_decode(q.scales.numpy()) * float(q.scale2)
    step = np.repeat(step, 16, axis=1)
    err = np.abs(deq - w.double().numpy())
    assert np.all(err <= step * 1.0001 + 1e-12)
    assert err.mean() < 0.25 * np.abs(w.numpy()).mean()


# ---------------------------------------------------------------------------
# Small layers for the routing and expert pins
# ---------------------------------------------------------------------------

def small_shape(**kw):
    base = dict(hidden=96, num_experts=8, top_k=3, moe_inter=64, shared_inter=32)
    base.update(kw)
    return synth.MoeShape(**base)


def dense_mats(layer):
    """All matrices of a layer dequantised through the library decoders."""
    s = layer.shape
    d = {}
    if s.router_fmt == "nvfp4":
        m = layer.router_nvfp4
        d["router"] = ref.nvfp4_dense(m.packed, m.scales, m.scale2)
    else:
        d["router"] = ref.bf16_decode(ref.to_np(layer.router_bf16))
    for name in ("gate", "up", "down"):
        src = getattr(layer, name)
        d[name] = [ref.expert_dense(s.expert_fmt, src.packed[e], src.scales[e], src.scale2[e])
                   for e in range(s.num_experts)]
    if s.has_shared:
        for name in ("sh_gate", "sh_up", "sh_down"):
            m = getattr(layer, name)
            d[name] = ref.expert_dense(s.expert_fmt, m.packed, m.scales, m.scale2)
        d["sh_vec"] = ref.bf16_decode(ref.to_np(layer.sh_gate_vec))
    return d


def swiglu64(x, wg, wu, wd):
    x = torch.as_tensor(x, dtype=torch.float64)
    g = torch.as_tensor(wg) @ x
    u = torch.as_tensor(wu) @ x
    return (torch.as_tensor(wd) @ (torch.nn.functional.silu(g) * u)).numpy()


def brute_route(shape, logits_row, bias):
    """Routing of one row by library routines: softmax / expit from scipy,
    selection by a stable lexsort on fp32 keys (key desc, id asc)."""
    E, k = shape.num_experts, shape.top_k
    if shape.scoring == "softmax":
        score = sps.softmax(logits_row)
        key = logits_row.astype(np.float32)
    else:
        score = sps.expit(logits_row)
        key = (score + bias.astype(np.float64)).astype(np.float32)
    order = np.lexsort((np.arange(E), -key.astype(np.float64)))
    ids = order[:k]
    w = score[ids]
    if shape.norm_topk_prob:
        w = w / w.sum()
    if shape.scoring == "sigmoid":
        w = w * shape.routed_scaling_factor
    return ids, w


def brute_forward(layer, x_bits):
    """Dense brute force: every expert evaluated for every row, then the
    selected ones gathered; independent of the oracle's code."""
    s = layer.shape
    d = dense_mats(layer)
    x = ref.bf16_decode(x_bits)
    logits = x @ d["router"].T
    bias = ref.to_np(layer.bias) if layer.bias is not None else None
    outs, all_ids, all_w = [], [], []
    for r in range(x.shape[0]):
        ys = np.stack([swiglu64(x[r], d["gate"][e], d["up"][e], d["down"][e])
                       for e in range(s.num_experts)])
        ids, w = brute_route(s, logits[r], bias)
        out = (w[:, None] * ys[ids]).sum(0)
        if s.has_shared:
            ysh = swiglu64(x[r], d["sh_gate"], d["sh_up"], d["sh_down"])
            gate = sps.expit(x[r] @ d["sh_vec"]) if s.shared_gated else 1.0
            out = out + gate * ysh
        outs.append(out)
        all_ids.append(ids)
        all_w.append(w)
    return np.stack(outs), np.stack(all_ids), np.stack(all_w), logits


# ---------------------------------------------------------------------------
# Router
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_router_onehot_picks_weight_column(orc, fmt):
    layer = synth.make_layer(small_shape(router_fmt=fmt), seed=5)
    ol = orc.OracleLayer(layer)
    d = dense_mats(layer)
    H = layer.shape.hidden
    for h in (0, 1, 17, H - 1):
        x = torch.zeros((1, H), dtype=torch.bfloat16)
        x[0, h] = 1.0
        lg = ol.router_logits(x)
        assert np.array_equal(lg[0], d["router"][:, h])


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_router_vs_numpy_matmul(orc, fmt):
    shape = small_shape(router_fmt=fmt)
    layer = synth.make_layer(shape, seed=6)
    x = synth.make_rows(shape, 4, seed=7)
    lg = orc.OracleLayer(layer).router_logits(x)
    want = ref.bf16_decode(ref.to_np(x)) @ dense_mats(layer)["router"].T
    np.testing.assert_allclose(lg, want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Top-k and routing weights
# ---------------------------------------------------------------------------

def test_topk_vs_lexsort_with_planted_ties(orc):
    rng = np.random.default_rng(8)
    for trial in range(300):
        E = int(rng.integers(4, 17))
        k = int(rng.integers(1, E + 1))
        keys = rng.integers(-3, 4, size=E).astype(np.float64)   # many ties
        if trial % 2:
            keys = keys + rng.standard_normal(E) * 1e-3
        want = np.lexsort((np.arange(E), -keys))[:k]
        assert np.array_equal(orc.topk(keys, k), want), (keys, k)


def test_softmax_weights_vs_scipy(orc):
    rng = np.random.default_rng(9)
    for norm in (True, False):
        shape = small_shape(num_experts=16, top_k=4, norm_topk_prob=norm)
        ol = orc.OracleLayer(synth.make_layer(shape, seed=10))
        for _ in range(50):
            lg = rng.standard_normal(16) * 2
            ids, w = ol.topk_row(lg)
            p = sps.softmax(lg)
            assert np.array_equal(ids, np.argsort(-lg, kind="stable")[:4])
            want = p[ids] / (p[ids].sum() if norm else 1.0)
            np.testing.assert_allclose(w, want, rtol=1e-13)
            if norm:
                assert abs(w.sum() - 1.0) < 1e-13


def test_selection_decided_on_fp32_keys(orc):
    """The top-k decision is taken on keys rounded to fp32, the precision of
    the kernel's logits: keys that differ only below fp32 resolution tie,
    and the tie goes to the lower expert id."""
    shape = small_shape(num_experts=8, top_k=2)
    ol = orc.OracleLayer(synth.make_layer(shape, seed=31))
    ids, _ = ol.topk_row(np.array([0.5, 0.5 + 2.0 ** -40, 0.1, 0, 0, 0, 0, 0]))
    assert list(ids) == [0, 1]
    # sigmoid(0) = 0.5 and sigmoid(1e-9) = 0.5 + 2.5e-10 round to the same fp32
    shape = small_shape(num_experts=8, top_k=2, scoring="sigmoid")
    layer = synth.make_layer(shape, seed=32)
    layer.bias = torch.zeros(8, dtype=torch.float32)
    ids, _ = orc.OracleLayer(layer).topk_row(np.array([0.0, 1e-9, -3, -3, -3, -3, -3, -3]))
    assert list(ids) == [0, 1]


def test_softmax_equal_logits_uniform(orc):
    shape = small_shape(num_experts=16, top_k=4)
    ol = orc.OracleLayer(synth.make_layer(shape, seed=11))
    ids, w = ol.topk_row(np.full(16, 0.37))
    assert list(ids) == [0, 1, 2, 3]
    np.testing.assert_allclose(w, 0.25, rtol=1e-15)


def test_sigmoid_bias_selection_and_weights(orc):
    rng = np.random.default_rng(12)
    shape = small_shape(num_experts=16, top_k=4, scoring="sigmoid",
                        routed_scaling_factor=2.5)
    layer = synth.make_layer(shape, seed=13)
    ol = orc.OracleLayer(layer)
    bias = ref.to_np(layer.bias)
    for _ in range(50):
        lg = rng.standard_normal(16)
        ids, w = ol.topk_row(lg)
        want_ids, want_w = brute_route(shape, lg, bias)
        assert np.array_equal(ids, want_ids)
        np.testing.assert_allclose(w, want_w, rtol=1e-13)
        assert abs(w.sum() - 2.5) < 1e-12
        # the bias steers the selection but not the weights
        s = sps.expit(lg[ids])
        np.testing.assert_allclose(w, 2.5 * s / s.sum(), rtol=1e-13)


def test_sigmoid_bias_changes_selection(orc):
    shape = small_shape(num_experts=8, top_k=2, scoring="sigmoid")
    layer = synth.make_layer(shape, seed=14)
    layer.bias = torch.tensor([0, 0, 0, 0, 0, 0, 0.9, 0.8], dtype=torch.float32)
    ol = orc.OracleLayer(layer)
    ids, _ = ol.topk_row(np.array([1.0, 0.9, 0, 0, 0, 0, 0, 0]))
    assert list(ids) == [6, 7]


# ---------------------------------------------------------------------------
# Union
# ---------------------------------------------------------------------------

def test_union_vs_python_first_occurrence(orc):
    rng = np.random.default_rng(15)
    for _ in range(300):
        rows = int(rng.integers(1, 9))
        k = int(rng.integers(1, 9))
        E = int(rng.integers(k, 40))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(rows)]).astype(np.int32)
        U, uni, slot2u, rowmask = orc.union(ids)
        want = list(dict.fromkeys(ids.ravel().tolist()))
        assert U == len(want) and list(uni) == want
        assert U <= min(rows * k, E)
        for r in range(rows):
            for j in range(k):
                assert uni[slot2u[r, j]] == ids[r, j]
        for u in range(U):
            rows_with = {r for r in range(rows) if uni[u] in ids[r]}
            assert {r for r in range(8) if rowmask[u] >> r & 1} == rows_with
        if rows == 1:
            assert U == k


def test_union_of_32_rows_vs_python_first_occurrence(orc):
    """Prefill chunks wider than one 8-row sub-chunk: the union of up to 32
    rows (256 ids) is the same first-occurrence scan, with 32-bit row masks."""
    rng = np.random.default_rng(13)
    for rows, k, E in ((32, 8, 160), (16, 8, 512), (24, 4, 40), (32, 2, 7)):
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(rows)])
        U, uni, slot2u, rowmask = orc.union(ids)
        first = list(dict.fromkeys(int(v) for v in ids.ravel()))
        assert U == len(first) and [int(v) for v in uni] == first
        for u, e in enumerate(first):
            rows_with = {r for r in range(rows) if e in ids[r]}
            assert {r for r in range(32) if int(rowmask[u]) >> r & 1} == rows_with
        for r in range(rows):
            for j in range(k):
                assert first[slot2u[r, j]] == ids[r, j]


def test_union_ignores_prior_buffer_contents(orc):
    """The union fills its output arrays whatever they held before."""
    ids = np.array([[3, 1], [1, 4]], dtype=np.int32)
    uni = np.full(4, -7, dtype=np.int32)
    slot2u = np.full((2, 2), 0xEE, dtype=np.uint8)
    rowmask = np.full(4, 0xFF, dtype=np.uint32)
    U = orc.lib().orc_union(ids.ctypes.data, 2, 2, uni.ctypes.data, slot2u.ctypes.data,
                            rowmask.ctypes.data)
    assert U == 3 and list(uni[:3]) == [3, 1, 4]
    assert list(rowmask[:3]) == [0b01, 0b11, 0b10]
    assert slot2u.tolist() == [[0, 1], [1, 2]]


def test_union_mean_matches_independent_routing_closed_form(orc):
    """E[U] = E * (1 - (1 - k/E)^R) for rows that each draw k distinct
    experts uniformly: E=512, k=8, R=8 -> 60.6."""
    rng = np.random.default_rng(16)
    E, k, R = 512, 8, 8
    tot = 0
    n = 2000
    for _ in range(n):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(R)])
        tot += orc.union(ids.astype(np.int32))[0]
    want = E * (1 - (1 - k / E) ** R)
    assert abs(tot / n - want) < 0.15, (tot / n, want)


# ---------------------------------------------------------------------------
# Expert MLP and the whole layer
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "bf16"])
def test_expert_mlp_vs_torch_swiglu(orc, fmt):
    shape = small_shape(expert_fmt=fmt)
    layer = synth.make_layer(shape, seed=17)
    d = dense_mats(layer)
    x = np.random.default_rng(18).standard_normal(shape.hidden)
    for e in (0, 5):
        g = orc.HostMat(layer.gate.packed[e], layer.gate.scales[e], layer.gate.scale2[e], fmt)
        u = orc.HostMat(layer.up.packed[e], layer.up.scales[e], layer.up.scale2[e], fmt)
        dn = orc.HostMat(layer.down.packed[e], layer.down.scales[e], layer.down.scale2[e], fmt)
        y = orc.expert_mlp(g, u, dn, x)
        want = swiglu64(x, d["gate"][e], d["up"][e], d["down"][e])
        np.testing.assert_allclose(y, want, rtol=1e-11, atol=1e-14)


def test_forward_reduces_to_swiglu(orc):
    """top_k = 1 with norm_topk_prob (weight exactly 1) and an all-zero
    shared down projection: the layer is the selected expert's SwiGLU MLP."""
    shape = small_shape(top_k=1)
    layer = synth.make_layer(shape, seed=19)
    layer.sh_down = synth.zero_nvfp4_like(layer.sh_down)
    x = synth.make_rows(shape, 3, seed=20)
    res = orc.OracleLayer(layer).forward(x)
    d = dense_mats(layer)
    xd = ref.bf16_decode(ref.to_np(x))
    for r in range(3):
        e = int(res["ids"][r, 0])
        assert e == int(np.argmax(res["logits"][r]))
        assert res["wts"][r, 0] == 1.0
        want = swiglu64(xd[r], d["gate"][e], d["up"][e], d["down"][e])
        np.testing.assert_allclose(res["out"][r], want, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("variant", [
    dict(),
    dict(scoring="sigmoid", routed_scaling_factor=2.5),
    dict(router_fmt="nvfp4"),
    dict(norm_topk_prob=False),
    dict(shared_gated=False),
    dict(has_shared=False),
    dict(moe_inter=32, shared_inter=96),      # shared expert wider than the routed ones
    dict(expert_fmt="fp8"),
    dict(expert_fmt="bf16"),
    dict(expert_fmt="fp8", scoring="sigmoid", routed_scaling_factor=2.5, router_fmt="nvfp4"),
    dict(expert_fmt="bf16", shared_gated=False, norm_topk_prob=False),
])
def test_forward_vs_dense_bruteforce(orc, variant):
    shape = small_shape(**variant)
    layer = synth.make_layer(shape, seed=21)
    x = synth.make_rows(shape, 4, seed=22)
    res = orc.OracleLayer(layer).forward(x, nthreads=3)
    out, ids, w, logits = brute_forward(layer, ref.to_np(x))
    assert np.array_equal(res["ids"], ids)
    np.testing.assert_allclose(res["wts"], w, rtol=1e-12)
    np.testing.assert_allclose(res["logits"], logits, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(res["out"], out, rtol=1e-10, atol=1e-13)
    # bf16 view is the round-to-nearest-even of the fp64 result
    rb = torch.from_numpy(res["out"]).to(torch.float32)
    exact = rb.double().numpy() == res["out"]
    want_b = rb.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(res["out_bf16"][exact], want_b[exact])


@pytest.mark.parametrize("variant", [
    dict(num_experts=1, top_k=1),                          # one expert, weight 1
    dict(num_experts=5, top_k=5),                          # every expert selected
    dict(num_experts=5, top_k=5, scoring="sigmoid", routed_scaling_factor=2.5,
         norm_topk_prob=False),
])
def test_forward_degenerate_routing_vs_dense_bruteforce(orc, variant):
    """Routing with no choice left: a single expert, or k = E so that every
    expert is selected and the weights are the whole (normalised) score
    vector in descending order."""
    shape = small_shape(**variant)
    layer = synth.make_layer(shape, seed=29)
    x = synth.make_rows(shape, 3, seed=30)
    res = orc.OracleLayer(layer).forward(x)
    out, ids, w, _ = brute_forward(layer, ref.to_np(x))
    assert np.array_equal(res["ids"], ids)
    for r in range(3):
        assert sorted(res["ids"][r]) == list(range(shape.num_experts))
    np.testing.assert_allclose(res["wts"], w, rtol=1e-12)
    np.testing.assert_allclose(res["out"], out, rtol=1e-10, atol=1e-13)
    if shape.num_experts == 1:
        assert np.all(res["wts"] == 1.0)
    U, uni, _, rowmask = orc.union(res["ids"])
    assert U == shape.num_experts and np.all(rowmask == 0b111)


def _bf16_nearest(v: float) -> float:
    """Nearest bfloat16 to a (normal-range) double, ties to even, by exact
    rational arithmetic."""
    from fractions import Fraction
    if v == 0.0:
        return 0.0
    e = math.frexp(abs(v))[1]                 # |v| = f * 2^e, f in [0.5, 1)
    quantum = Fraction(2) ** (e - 8)          # 8 significant bits
    return float(round(Fraction(v) / quantum) * quantum)


def _bf16_bits(val: float) -> int:
    return int(np.array([val], dtype=np.float32).view(np.uint32)[0]) >> 16


def test_forward_output_rounded_once_to_bf16(orc):
    """The layer's bf16 output is the nearest bf16 of the fp64 result, not of
    its fp32 rounding.  One expert, top-1 with norm (weight exactly 1), no
    shared expert, and a down matrix whose only non-zero weight per row sits
    at input 0 with value scale2: every output is scale2 * h[0].  scale2 is
    the fp32 value that puts the product inside the narrow band where fp32
    rounding lands on a bf16 midpoint, so the two roundings differ."""
    shape = small_shape(num_experts=1, top_k=1, has_shared=False)
    layer = synth.make_layer(shape, seed=33)
    x = synth.make_rows(shape, 1, seed=34)
    d = dense_mats(layer)
    xd = torch.as_tensor(ref.bf16_decode(ref.to_np(x))[0], dtype=torch.float64)
    g = torch.as_tensor(d["gate"][0][0]) @ xd
    u = torch.as_tensor(d["up"][0][0]) @ xd
    h0 = float(torch.nn.functional.silu(g) * u)
    assert abs(h0) > 1e-6
    found = None
    for k in range(1, 400):
        b = _bf16_nearest(abs(h0) * (1 + k / 512))
        m = b + 2.0 ** (math.frexp(b)[1] - 9)          # midpoint above b
        c = np.float32(m / abs(h0))
        for _ in range(4):
            v = float(c) * h0
            if (np.float32(v) == np.float32(math.copysign(m, h0)) and abs(v) != m
                    and abs(abs(v) - m) > 2.0 ** -45 * m
                    and _bf16_nearest(v) != _bf16_nearest(float(np.float32(v)))):
                found = (c, v)
                break
            c = np.nextafter(c, np.float32(np.inf))
        if found:
            break
    assert found, "no fp32 scale puts the product in the double-rounding band"
    c, v = found
    H, I = shape.hidden, shape.moe_inter
    dn = layer.down
    dn.packed[0].zero_()
    dn.scales[0].zero_()
    dn.packed[0][:, 0] = 2                 # E2M1 code of 1.0 at input 0 (low nibble)
    dn.scales[0][:, 0] = 0x38              # E4M3 code of 1.0 for inputs 0..15
    dn.scale2[0] = float(c)
    res = orc.OracleLayer(layer).forward(x)
    assert res["wts"][0, 0] == 1.0
    np.testing.assert_allclose(res["out"][0], v, rtol=1e-13)
    want = _bf16_bits(_bf16_nearest(v))
    assert want != _bf16_bits(_bf16_nearest(float(np.float32(v))))
    assert np.all(res["out_bf16"][0] == want)


def test_forward_identical_experts_closed_form(orc):
    """Every routed expert has the same weights: the weighted sum collapses
    to (sum of weights) * y = y (softmax with norm), so
    out = y + sigmoid(x . gs) * ys."""
    shape = small_shape()
    layer = synth.make_layer(shape, seed=23)
    for name in ("gate", "up", "down"):
        m = getattr(layer, name)
        for t in (m.packed, m.scales, m.scale2):
            t[:] = t[0:1].clone()
    x = synth.make_rows(shape, 2, seed=24)
    res = orc.OracleLayer(layer).forward(x)
    d = dense_mats(layer)
    xd = ref.bf16_decode(ref.to_np(x))
    for r in range(2):
        y = swiglu64(xd[r], d["gate"][0], d["up"][0], d["down"][0])
        ys = swiglu64(xd[r], d["sh_gate"], d["sh_up"], d["sh_down"])
        gate = sps.expit(xd[r] @ d["sh_vec"])
        np.testing.assert_allclose(res["out"][r], y + gate * ys, rtol=1e-11, atol=1e-14)


def test_forward_thread_count_invariant(orc):
    shape = small_shape()
    layer = synth.make_layer(shape, seed=25)
    x = synth.make_rows(shape, 4, seed=26)
    ol = orc.OracleLayer(layer)
    a = ol.forward(x, nthreads=1)
    b = ol.forward(x, nthreads=5)
    assert np.array_equal(a["out"], b["out"])


def test_forward_union_sweep_equals_per_row(orc):
    """Evaluating each union expert once for the rows of its rowmask and
    summing in slot order gives the oracle's per-row result exactly."""
    shape = small_shape(num_experts=6, top_k=3)
    layer = synth.make_layer(shape, seed=27)
    x = synth.make_rows(shape, 4, seed=28, corr=0.9)
    ol = orc.OracleLayer(layer)
    res = ol.forward(x)
    U, uni, slot2u, rowmask = orc.union(res["ids"])
    assert U < 4 * 3                      # correlated rows share experts
    xd = ref.bf16_decode(ref.to_np(x))
    ysw = {}
    for u in range(U):
        e = int(uni[u])
        g = orc.HostMat(layer.gate.packed[e], layer.gate.scales[e], layer.gate.scale2[e])
        up = orc.HostMat(layer.up.packed[e], layer.up.scales[e], layer.up.scale2[e])
        dn = orc.HostMat(layer.down.packed[e], layer.down.scales[e], layer.down.scale2[e])
        for r in range(4):
            if rowmask[u] >> r & 1:
                ysw[(u, r)] = orc.expert_mlp(g, up, dn, xd[r])
    sg = orc.HostMat(layer.sh_gate.packed, layer.sh_gate.scales, layer.sh_gate.scale2)
    su = orc.HostMat(layer.sh_up.packed, layer.sh_up.scales, layer.sh_up.scale2)
    sd = orc.HostMat(layer.sh_down.packed, layer.sh_down.scales, layer.sh_down.scale2)
    gs = ref.bf16_decode(ref.to_np(layer.sh_gate_vec))
    for r in range(4):
        ys = orc.expert_mlp(sg, su, sd, xd[r])
        dot = 0.0
        for h in range(shape.hidden):
            dot += xd[r, h] * gs[h]
        gate = 1.0 / (1.0 + math.exp(-dot))
        for o in range(shape.hidden):
            acc = 0.0
            for j in range(3):
                acc += res["wts"][r, j] * ysw[(int(slot2u[r, j]), r)][o]
            acc += gate * ys[o]
            assert acc == res["out"][r, o]


# ---------------------------------------------------------------------------
# The layer at caller-given experts (used to evaluate a near-tie row at the
# GPU's selection)
# ---------------------------------------------------------------------------

def _given_ids(rng, E, k, rows):
    """Distinct ids per row in a random order, deliberately not the top-k."""
    return np.stack([rng.permutation(E)[:k] for _ in range(rows)]).astype(np.int32)


@pytest.mark.parametrize("variant", [
    dict(),
    dict(norm_topk_prob=False),
    dict(scoring="sigmoid", routed_scaling_factor=2.5),
    dict(scoring="sigmoid", routed_scaling_factor=1.5, norm_topk_prob=False),
])
def test_weights_for_given_ids_vs_scipy(orc, variant):
    shape = small_shape(num_experts=12, top_k=4, **variant)
    layer = synth.make_layer(shape, seed=41)
    ol = orc.OracleLayer(layer, experts=())
    rng = np.random.default_rng(42)
    for _ in range(20):
        lg = rng.normal(0.0, 2.0, shape.num_experts)
        sel = rng.permutation(shape.num_experts)[:shape.top_k]
        score = sps.softmax(lg) if shape.scoring == "softmax" else sps.expit(lg)
        want = score[sel]
        if shape.norm_topk_prob:
            want = want / want.sum()
        if shape.scoring == "sigmoid":
            want = want * shape.routed_scaling_factor
        np.testing.assert_allclose(ol.weights_for_ids(lg, sel), want, rtol=1e-13)


@pytest.mark.parametrize("variant", [
    dict(),
    dict(scoring="sigmoid", routed_scaling_factor=2.5),
    dict(norm_topk_prob=False, shared_gated=False),
])
def test_forward_at_given_ids_vs_dense_bruteforce(orc, variant):
    """Every row evaluated at experts that are not its top-k, in a random
    slot order: weights and output against the dense brute force at the
    same experts."""
    shape = small_shape(num_experts=9, top_k=3, **variant)
    layer = synth.make_layer(shape, seed=43)
    x = synth.make_rows(shape, 4, seed=44)
    sel = _given_ids(np.random.default_rng(45), shape.num_experts, shape.top_k, 4)
    res = orc.OracleLayer(layer).forward_ids(x, sel, nthreads=2)
    d = dense_mats(layer)
    xd = ref.bf16_decode(ref.to_np(x))
    logits = xd @ d["router"].T
    for r in range(4):
        score = sps.softmax(logits[r]) if shape.scoring == "softmax" else sps.expit(logits[r])
        w = score[sel[r]]
        if shape.norm_topk_prob:
            w = w / w.sum()
        if shape.scoring == "sigmoid":
            w = w * shape.routed_scaling_factor
        np.testing.assert_allclose(res["wts"][r], w, rtol=1e-12)
        out = sum(w[j] * swiglu64(xd[r], d["gate"][e], d["up"][e], d["down"][e])
                  for j, e in enumerate(sel[r]))
        gate = sps.expit(xd[r] @ d["sh_vec"]) if shape.shared_gated else 1.0
        out = out + gate * swiglu64(xd[r], d["sh_gate"], d["sh_up"], d["sh_down"])
        np.testing.assert_allclose(res["out"][r], out, rtol=1e-10, atol=1e-13)


def test_forward_at_given_ids_refuses_repeated_ids(orc):
    shape = small_shape(num_experts=9, top_k=3)
    layer = synth.make_layer(shape, seed=43)
    x = synth.make_rows(shape, 1, seed=44)
    with pytest.raises(ValueError):
        orc.OracleLayer(layer).forward_ids(x, np.array([[1, 1, 2]], dtype=np.int32))
