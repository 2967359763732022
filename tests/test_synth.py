"""The seeded input generator: determinism, the router-only shortcut, the
row-correlation recipe and the NVFP4 encoder's code ranges.  CPU only."""
import numpy as np
import pytest
import torch

from routed_moe_decode_router_gb300 import synth

SHAPES = [
    synth.MoeShape(256, 16, 4, 128, 128),
    synth.MoeShape(256, 24, 3, 128, 128, scoring="sigmoid", routed_scaling_factor=2.5),
    synth.MoeShape(256, 16, 4, 128, 128, router_fmt="nvfp4"),
]


def _tensors(layer):
    out = {}
    for name in ("router_bf16", "bias", "sh_gate_vec"):
        t = getattr(layer, name, None)
        if t is not None:
            out[name] = t
    for name in ("router_nvfp4", "gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        m = getattr(layer, name, None)
        if m is not None:
            out[name + ".packed"] = m.packed
            out[name + ".scales"] = m.scales
            out[name + ".scale2"] = m.scale2
    return out


@pytest.mark.parametrize("shape", SHAPES)
def test_make_layer_is_deterministic_and_seed_dependent(shape):
    a = _tensors(synth.make_layer(shape, seed=7))
    b = _tensors(synth.make_layer(shape, seed=7))
    c = _tensors(synth.make_layer(shape, seed=8))
    assert a.keys() == b.keys() == c.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert any(not torch.equal(a[k], c[k]) for k in a)


@pytest.mark.parametrize("shape", SHAPES)
def test_router_only_draws_the_full_layers_routing_weights(shape):
    """The router-only shortcut (used to calibrate the row correlation on
    the routing alone) must give the same router and bias as the full
    layer of the same seed."""
    full = synth.make_layer(shape, seed=11)
    ro = synth.make_layer(shape, seed=11, router_only=True)
    if shape.router_fmt == "nvfp4":
        for f in ("packed", "scales", "scale2"):
            assert torch.equal(getattr(full.router_nvfp4, f), getattr(ro.router_nvfp4, f))
    else:
        assert torch.equal(full.router_bf16, ro.router_bf16)
    if shape.scoring == "sigmoid":
        assert torch.equal(full.bias, ro.bias)
        assert float(full.bias.abs().max()) <= 0.1


def test_make_rows_deterministic_and_correlated():
    shape = synth.MoeShape(2048, 16, 4, 128, 128)
    a = synth.make_rows(shape, 4, seed=3)
    assert a.dtype == torch.bfloat16 and a.shape == (4, 2048)
    assert torch.equal(a, synth.make_rows(shape, 4, seed=3))
    ind = synth.make_rows(shape, 8, seed=4).float()
    cor = synth.make_rows(shape, 8, seed=4, corr=0.8).float()
    c_ind = np.corrcoef(ind.numpy())[np.triu_indices(8, 1)]
    c_cor = np.corrcoef(cor.numpy())[np.triu_indices(8, 1)]
    # x_t = a*s + sqrt(1 - a^2)*n_t: unit variance, pairwise correlation a^2
    assert abs(c_ind).max() < 0.1
    assert abs(c_cor.mean() - 0.64) < 0.05
    assert abs(float(cor.std()) - 1.0) < 0.05


def test_quantizer_codes_and_zero_blocks():
    g = torch.Generator().manual_seed(5)
    w = torch.randn((8, 64), generator=g) * 0.02
    w[3, 16:32] = 0.0                       # one all-zero block of 16
    q = synth.quantize_nvfp4(w)
    assert q.packed.shape == (8, 32) and q.scales.shape == (8, 4)
    assert q.packed.dtype == torch.uint8 and q.scales.dtype == torch.uint8
    # E4M3 scales of amax/(6*scale2) <= 448 are finite positive codes (no NaN
    # code 0x7F/0xFF, no sign bit), except the zero block's 0
    s = q.scales.numpy()
    assert np.all(s & 0x80 == 0) and np.all((s & 0x7F) != 0x7F)
    assert s[3, 1] == 0 and np.all(q.packed.numpy()[3, 8:16] == 0)
    # the largest element of the matrix maps to the E2M1 code of magnitude 6
    n, k = np.unravel_index(int(w.abs().argmax()), w.shape)
    byte = int(q.packed[n, k // 2])
    code = (byte >> 4) if k % 2 else (byte & 15)
    assert code & 7 == 7
    assert float(q.scale2) == pytest.approx(float(w.abs().max()) / (6 * 448), rel=1e-6)
