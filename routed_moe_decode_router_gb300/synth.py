"""Seeded synthetic inputs for the routed MoE layer.

This module only draws random numbers and stores them in the layer's storage
formats: bf16 activations and router weights, and the expert matrices in
NVFP4 (FP4 E2M1 codes, one FP8 E4M3 scale per 16 contiguous inputs, one fp32
scale per matrix), FP8 (one E4M3 code per weight, one fp32 scale per matrix)
or BF16 (one bfloat16 per weight, scale 1).  It holds none of the layer's own arithmetic, and both the CUDA
path and the CPU oracle read the bytes it writes.

Every draw comes from a ``torch.Generator`` seeded per layer (weights) or per
step (activations), so a workload is reproducible on one device; the CUDA
path and the oracle always read the same bytes, so the two devices' random
streams never need to agree.

Workloads (names carry the shapes):

``tiny_h256_e16``        1 row, H=256, E=16, top_k=4, I=Is=128, softmax + norm,
                         bf16 router, sigmoid-gated shared expert, seed 0.
``decode_h2048_e128``    1 row, H=2048, E=128, top_k=8, I=Is=768, softmax +
                         norm, NVFP4 router, 48 distinct layers.
``verify_h4096_e256``    2..4 correlated rows, H=4096, E=256, top_k=8,
                         I=Is=1024, sigmoid + correction bias U(-0.1, 0.1),
                         norm, routed_scaling_factor 2.5, 16 distinct layers.
``prefill8_h2048_e512``  8 independent rows, H=2048, E=512, top_k=8,
                         I=Is=512, softmax + norm, 16 distinct layers.
``sweep_h4096_e160``     1..8 correlated rows, H=4096, E=160, top_k=8,
                         I=Is=1536, sigmoid + bias, rsf 2.5, 48 distinct layers.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

# Correlation ``a`` of consecutive rows, x_t = a*s + sqrt(1-a^2)*n_t, for the
# verify and sweep workloads.  Written by tests/golden/make_corr_calibration.py
# (which bisects ``a`` on the oracle's routing of the verify workload so that
# the mean union over K = 2..4 rows tracks the live-trace curve the forward_moe
# page quotes: 8.00 / 13.74 / 18.76 / 23.35 at K = 1..4); its output is
# tests/golden/corr_calibration.json.
CORR_A = 0.706

E4M3_MAX = 448.0
E2M1_MAX = 6.0


@dataclasses.dataclass(frozen=True)
class MoeShape:
    hidden: int
    num_experts: int
    top_k: int
    moe_inter: int
    shared_inter: int
    scoring: str = "softmax"          # "softmax" or "sigmoid"
    norm_topk_prob: bool = True
    routed_scaling_factor: float = 1.0
    router_fmt: str = "bf16"          # "bf16" or "nvfp4"
    has_shared: bool = True
    shared_gated: bool = True
    expert_fmt: str = "nvfp4"         # "nvfp4", "fp8" or "bf16" (routed and shared experts)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: MoeShape
    rows: Sequence[int]
    layers: int
    seed_base: int
    corr: Optional[float]             # None = independent rows


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_h256_e16",
                 MoeShape(256, 16, 4, 128, 128), rows=(1,), layers=1,
                 seed_base=0, corr=None),
        Workload("decode_h2048_e128",
                 MoeShape(2048, 128, 8, 768, 768, router_fmt="nvfp4"),
                 rows=(1,), layers=48, seed_base=1000, corr=None),
        Workload("verify_h4096_e256",
                 MoeShape(4096, 256, 8, 1024, 1024, scoring="sigmoid",
                          routed_scaling_factor=2.5),
                 rows=(1, 2, 3, 4), layers=16, seed_base=2000, corr=CORR_A),
        Workload("prefill8_h2048_e512",
                 MoeShape(2048, 512, 8, 512, 512), rows=(8,), layers=16,
                 seed_base=3000, corr=None),
        Workload("sweep_h4096_e160",
                 MoeShape(4096, 160, 8, 1536, 1536, scoring="sigmoid",
                          routed_scaling_factor=2.5),
                 rows=(1, 2, 3, 4, 5, 6, 7, 8), layers=48, seed_base=4000,
                 corr=CORR_A),
    ]
}


@dataclasses.dataclass
class Nvfp4:
    """One expert matrix [N][K] (or a stack [..., N, K] of them).  NVFP4:
    packed uint8 [..., N, K/2] (low nibble = even input), scales uint8
    [..., N, K/16] (E4M3 bit patterns).  The other expert formats use the
    same holder: FP8, packed uint8 [..., N, K] (E4M3 codes); BF16, packed
    uint8 [..., N, 2K] (the little-endian bfloat16 bytes); both with empty
    scales [..., N, 0]."""
    packed: torch.Tensor
    scales: torch.Tensor
    scale2: torch.Tensor   # float32 [...]; one per matrix

    def to(self, device) -> "Nvfp4":
        return Nvfp4(self.packed.to(device), self.scales.to(device),
                     self.scale2.to(device))

    def select(self, i: int) -> "Nvfp4":
        return Nvfp4(self.packed[i], self.scales[i], self.scale2[i])


@dataclasses.dataclass
class MoeLayerWeights:
    shape: MoeShape
    router_bf16: Optional[torch.Tensor]   # bf16 [E, H]
    router_nvfp4: Optional[Nvfp4]         # [E, H]
    bias: Optional[torch.Tensor]          # float32 [E] (sigmoid scoring)
    gate: Nvfp4                           # [E, I, H]
    up: Nvfp4                             # [E, I, H]
    down: Nvfp4                           # [E, H, I]
    sh_gate: Optional[Nvfp4]              # [Is, H]
    sh_up: Optional[Nvfp4]                # [Is, H]
    sh_down: Optional[Nvfp4]              # [H, Is]
    sh_gate_vec: Optional[torch.Tensor]   # bf16 [H]

    @property
    def device(self):
        return self.gate.packed.device

    def to(self, device) -> "MoeLayerWeights":
        def mv(t):
            return None if t is None else t.to(device)
        return MoeLayerWeights(self.shape, mv(self.router_bf16),
                               mv(self.router_nvfp4), mv(self.bias),
                               self.gate.to(device), self.up.to(device),
                               self.down.to(device), mv(self.sh_gate),
                               mv(self.sh_up), mv(self.sh_down),
                               mv(self.sh_gate_vec))


def _e2m1_code(v: torch.Tensor) -> torch.Tensor:
    """Nearest FP4 E2M1 code of v (|v| saturates at 6); a tie goes to the code
    with the even magnitude index.  Magnitudes by code 0..7:
    0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    a = v.abs()
    mag = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
           + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
           + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    neg = ((v < 0) & (mag > 0)).to(torch.uint8)
    return mag | (neg << 3)


def quantize_nvfp4(w: torch.Tensor) -> Nvfp4:
    """Encode float weights [..., N, K] (K a multiple of 32) into NVFP4.

    scale2 = amax(|W|) / (6 * 448) per matrix; the E4M3 block scale is the
    round-to-nearest-even E4M3 value of amax(block) / (6 * scale2); each
    element is the nearest E2M1 code of w / (block scale * scale2).  An
    all-zero block gets scale 0 and zero codes."""
    w = w.float()
    *lead, N, K = w.shape
    assert K % 32 == 0, "K must be a multiple of 32"
    amax = w.abs().amax(dim=(-2, -1))
    scale2 = torch.where(amax > 0, amax / (E2M1_MAX * E4M3_MAX),
                         torch.ones_like(amax))
    blk = w.reshape(*lead, N, K // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    s2 = scale2.reshape(*lead, 1, 1)
    sval = (bmax / (E2M1_MAX * s2)).clamp(max=E4M3_MAX)
    s8 = sval.to(torch.float8_e4m3fn)
    denom = s8.float() * s2
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    v = torch.where(denom[..., None] > 0, blk / safe[..., None],
                    torch.zeros_like(blk))
    code = _e2m1_code(v).reshape(*lead, N, K)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return Nvfp4(packed.contiguous(), s8.view(torch.uint8).contiguous(),
                 scale2.float().contiguous())


def quantize_fp8(w: torch.Tensor) -> Nvfp4:
    """Encode float weights [..., N, K] into FP8: scale2 = amax(|W|) / 448 per
    matrix, each element the round-to-nearest-even E4M3 code of w / scale2."""
    w = w.float()
    *lead, N, K = w.shape
    amax = w.abs().amax(dim=(-2, -1))
    scale2 = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    v = (w / scale2.reshape(*lead, 1, 1)).clamp(-E4M3_MAX, E4M3_MAX)
    codes = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return Nvfp4(codes.contiguous(),
                 torch.zeros((*lead, N, 0), dtype=torch.uint8, device=w.device),
                 scale2.float().contiguous())


def store_bf16(w: torch.Tensor) -> Nvfp4:
    """Store float weights [..., N, K] as bfloat16 (round to nearest even),
    scale2 = 1."""
    *lead, N, K = w.shape
    b = w.float().to(torch.bfloat16).contiguous()
    return Nvfp4(b.view(torch.uint8).reshape(*lead, N, 2 * K).contiguous(),
                 torch.zeros((*lead, N, 0), dtype=torch.uint8, device=w.device),
                 torch.ones(tuple(lead), dtype=torch.float32, device=w.device))


ENCODERS = {"nvfp4": quantize_nvfp4, "fp8": quantize_fp8, "bf16": store_bf16}


def _normal(gen, shape, std, device):
    return torch.randn(shape, generator=gen, device=device,
                       dtype=torch.float32) * std


def make_layer(shape: MoeShape, seed: int, device="cpu",
               std: float = 0.02, router_only: bool = False) -> MoeLayerWeights:
    """Random-init weights of one routed MoE layer, N(0, std) everywhere,
    experts encoded in the shape's expert format (NVFP4, FP8 or BF16; the
    same draws for every format).  Draw order: router, correction bias (sigmoid
    scoring only, U(-0.1, 0.1)), shared-expert gate vector, shared gate / up
    / down, then the routed experts in fixed-size chunks (gate, up, down per
    chunk).  ``router_only`` stops after the routing weights (router and
    bias) and leaves every expert matrix empty."""
    s = shape
    H, E, I, Is = s.hidden, s.num_experts, s.moe_inter, s.shared_inter
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    router_bf16 = router_nvfp4 = None
    wr = _normal(gen, (E, H), std, device)
    if s.router_fmt == "nvfp4":
        router_nvfp4 = quantize_nvfp4(wr)
    else:
        router_bf16 = wr.to(torch.bfloat16)
    del wr

    bias = None
    if s.scoring == "sigmoid":
        bias = (torch.rand((E,), generator=gen, device=device,
                           dtype=torch.float32) * 0.2 - 0.1)

    def empty(*shape):
        return Nvfp4(torch.zeros(shape + (0,), dtype=torch.uint8, device=device),
                     torch.zeros(shape + (0,), dtype=torch.uint8, device=device),
                     torch.zeros(shape[:-1], dtype=torch.float32, device=device))

    if router_only:
        return MoeLayerWeights(s, router_bf16, router_nvfp4, bias,
                               empty(E, I), empty(E, I), empty(E, H),
                               None, None, None, None)

    sh_gate = sh_up = sh_down = sh_vec = None
    enc = ENCODERS[s.expert_fmt]
    if s.has_shared:
        sh_vec = _normal(gen, (H,), std, device).to(torch.bfloat16)
        sh_gate = enc(_normal(gen, (Is, H), std, device))
        sh_up = enc(_normal(gen, (Is, H), std, device))
        sh_down = enc(_normal(gen, (H, Is), std, device))

    chunk = max(1, min(E, (1 << 25) // (I * H)))
    gp, gs_, g2, up_, us, u2, dp, ds, d2 = ([] for _ in range(9))
    for e0 in range(0, E, chunk):
        c = min(chunk, E - e0)
        q = enc(_normal(gen, (c, I, H), std, device))
        gp.append(q.packed); gs_.append(q.scales); g2.append(q.scale2)
        q = enc(_normal(gen, (c, I, H), std, device))
        up_.append(q.packed); us.append(q.scales); u2.append(q.scale2)
        q = enc(_normal(gen, (c, H, I), std, device))
        dp.append(q.packed); ds.append(q.scales); d2.append(q.scale2)
    gate = Nvfp4(torch.cat(gp), torch.cat(gs_), torch.cat(g2))
    up = Nvfp4(torch.cat(up_), torch.cat(us), torch.cat(u2))
    down = Nvfp4(torch.cat(dp), torch.cat(ds), torch.cat(d2))
    return MoeLayerWeights(s, router_bf16, router_nvfp4, bias, gate, up, down,
                           sh_gate, sh_up, sh_down, sh_vec)


def make_rows(shape: MoeShape, rows: int, seed: int, device="cpu",
              corr: Optional[float] = None) -> torch.Tensor:
    """Activations x [rows, H] in bf16.  Independent N(0, 1) rows, or rows
    correlated within the step: x_t = a*s + sqrt(1 - a^2)*n_t with one shared
    s ~ N(0, 1) and independent n_t ~ N(0, 1)."""
    H = shape.hidden
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if corr is None:
        x = torch.randn((rows, H), generator=gen, device=device)
    else:
        sh = torch.randn((1, H), generator=gen, device=device)
        n = torch.randn((rows, H), generator=gen, device=device)
        x = corr * sh + math.sqrt(1.0 - corr * corr) * n
    return x.to(torch.bfloat16)


def zero_nvfp4_like(m: Nvfp4) -> Nvfp4:
    """An all-zero NVFP4 matrix of the same geometry (zero codes, zero
    scales)."""
    return Nvfp4(torch.zeros_like(m.packed), torch.zeros_like(m.scales),
                 m.scale2.clone())
