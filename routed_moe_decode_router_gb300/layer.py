"""PyTorch-facing wrapper of the C ABI: holds one layer's device tensors and
their C descriptors, and calls the library on the current CUDA stream.
PyTorch provides device memory and streams only; every step runs in the
CUDA library.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import native as N
from .synth import MoeLayerWeights, MoeShape, Nvfp4


def make_config(shape: MoeShape, per_row_mode: bool = False, gemv: bool = False,
                t_layout: bool = False) -> N.MoeConfig:
    return N.MoeConfig(
        hidden=shape.hidden, num_experts=shape.num_experts,
        router_width=shape.num_experts, top_k=shape.top_k,
        moe_inter=shape.moe_inter, shared_inter=shape.shared_inter,
        scoring=N.MOE_SCORING_SIGMOID if shape.scoring == "sigmoid" else N.MOE_SCORING_SOFTMAX,
        norm_topk_prob=int(shape.norm_topk_prob),
        routed_scaling_factor=float(shape.routed_scaling_factor),
        router_fmt=N.MOE_ROUTER_NVFP4 if shape.router_fmt == "nvfp4" else N.MOE_ROUTER_BF16,
        has_shared=int(shape.has_shared), shared_gate=int(shape.shared_gated),
        per_row_mode=int(per_row_mode), gemv_lever=int(gemv), t_layout=int(t_layout),
        expert_fmt={"nvfp4": N.MOE_EXPERT_NVFP4, "fp8": N.MOE_EXPERT_FP8,
                    "bf16": N.MOE_EXPERT_BF16}[shape.expert_fmt])


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _device_of(dl: Optional["DeviceLayer"], ws: "Workspace") -> torch.device:
    dev = ws.buf.device
    if dev.type != "cuda":
        raise ValueError("the workspace is on %s; it must be in CUDA device memory" % dev)
    if dl is not None and dl.device != dev:
        raise ValueError("the layer is on %s but the workspace on %s" % (dl.device, dev))
    return dev


def _check_rows(t, name: str, dtype: torch.dtype, cols: int, device: torch.device):
    """Refuse, before any pointer reaches the library, a [rows, cols] tensor
    the kernels would misread: wrong dtype or width, not contiguous, or not
    in memory of the layer's CUDA device (a host pointer handed to a kernel
    faults the GPU instead of raising).  Reads tensor attributes only, so it
    is safe inside CUDA graph capture.  The row count itself is checked by
    the library."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if t.dim() != 2 or t.shape[1] != cols:
        raise ValueError("%s has shape %s, expected [rows, %d]" % (name, tuple(t.shape), cols))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.device != device:
        raise ValueError("%s is on %s; the layer and workspace are on %s"
                         % (name, t.device, device))


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class DeviceLayer:
    """One routed MoE layer resident on a CUDA device.

    ``layer`` holds the weights (moved to ``device`` if needed).  The
    per-expert pointer tables (device arrays of pointers, indexed by expert
    id) are built here once.  With ``t_layout`` the down projections (routed
    and shared) are converted once, by the library, into the t layout, and
    the layer's calls run the fused one-row form; the layer then holds the
    converted copies (the original down tensors stay in ``layer``)."""

    def __init__(self, layer: MoeLayerWeights, device="cuda", t_layout: bool = False):
        if layer.device != torch.device(device) and str(layer.device) != str(device):
            layer = layer.to(device)
        self.layer = layer
        self.shape = layer.shape
        self.device = layer.gate.packed.device
        self.t_layout = bool(t_layout)
        s = self.shape
        E = s.num_experts
        self._tables = {}
        down = layer.down
        sh_down = layer.sh_down if s.has_shared else None
        if self.t_layout:
            if s.expert_fmt != "nvfp4":
                raise ValueError("the t layout holds NVFP4 down projections only")
            stream = _stream(None)
            down = self._to_t(down, E, s.hidden, s.moe_inter, stream)
            if s.has_shared:
                sh_down = self._to_t(sh_down, 1, s.hidden, s.shared_inter, stream)
        # the converted copies must live as long as the layer: the pointer
        # tables and descriptors below point into them
        self.down, self.sh_down = down, sh_down
        w = N.MoeWeights()
        if s.router_fmt == "nvfp4":
            m = layer.router_nvfp4
            w.router_nvfp4 = N.Nvfp4Desc(m.packed.data_ptr(), m.scales.data_ptr(),
                                         float(m.scale2))
        else:
            w.router_bf16 = layer.router_bf16.data_ptr()
        if layer.bias is not None:
            w.correction_bias = layer.bias.data_ptr()
        for name in ("gate", "up", "down"):
            m = down if name == "down" else getattr(layer, name)
            pk = m.packed.reshape(E, -1)
            sc = m.scales.reshape(E, -1)
            pk_ptrs = (pk.data_ptr() + torch.arange(E, dtype=torch.int64) *
                       pk.stride(0)).to(device)
            # FP8 / BF16 experts have no block scales: NULL scale arrays
            sc_ptrs = (sc.data_ptr() + torch.arange(E, dtype=torch.int64) *
                       sc.stride(0)).to(device) if s.expert_fmt == "nvfp4" else None
            s2 = m.scale2.float().contiguous()
            self._tables[name] = (pk_ptrs, sc_ptrs, s2)
            setattr(w, name, N.ExpertTable(pk_ptrs.data_ptr(), _ptr(sc_ptrs),
                                           s2.data_ptr()))
        if s.has_shared:
            for name, field in (("sh_gate", "shared_gate_proj"),
                                ("sh_up", "shared_up_proj"),
                                ("sh_down", "shared_down_proj")):
                m = sh_down if name == "sh_down" else getattr(layer, name)
                setattr(w, field, N.Nvfp4Desc(
                    m.packed.data_ptr(), m.scales.data_ptr() if s.expert_fmt == "nvfp4" else 0,
                    float(m.scale2)))
            if s.shared_gated:
                w.shared_expert_gate = layer.sh_gate_vec.data_ptr()
        self.weights = w
        self._cfgs = {(pr, gv): make_config(s, per_row_mode=pr, gemv=gv, t_layout=self.t_layout)
                      for pr in (False, True) for gv in (False, True)}
        self.cfg = self._cfgs[(False, False)]
        self.cfg_per_row = self._cfgs[(True, False)]

    def config(self, per_row_mode: bool = False, gemv: bool = False) -> N.MoeConfig:
        return self._cfgs[(bool(per_row_mode), bool(gemv))]

    @staticmethod
    def _to_t(m, count: int, n_out: int, k_in: int, stream: int):
        """The t-layout copy of `count` stacked [n_out][k_in] NVFP4 matrices."""
        pk = torch.empty((count, k_in, n_out // 2), dtype=torch.uint8, device=m.packed.device)
        sc = torch.empty((count, k_in // 16, n_out), dtype=torch.uint8, device=m.packed.device)
        N.moe_nvfp4_to_t_layout(m.packed.data_ptr(), m.scales.data_ptr(), count, n_out, k_in,
                                pk.data_ptr(), sc.data_ptr(), stream)
        shape = m.packed.shape[:-2]
        return Nvfp4(pk.view(*shape, k_in, n_out // 2), sc.view(*shape, k_in // 16, n_out),
                     m.scale2)


class Workspace:
    """Caller-owned device workspace for one layer shape (zeroed once)."""

    def __init__(self, shape: MoeShape, device="cuda",
                 stream: Optional[torch.cuda.Stream] = None, t_layout: bool = False):
        self.nbytes = N.moe_workspace_size(make_config(shape, t_layout=t_layout))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        N.moe_workspace_init(self.buf.data_ptr(), self.nbytes, _stream(stream))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, stream=None) -> int:
        """Synchronise and read (then clear) the device status word."""
        return N.moe_read_device_status(self.ptr, self.nbytes, _stream(stream))


def forward(dl: DeviceLayer, x: torch.Tensor, ws: Workspace,
            out: Optional[torch.Tensor] = None, per_row_mode: bool = False,
            stream=None, gemv: bool = False) -> torch.Tensor:
    """out[rows, H] (bf16) = routed MoE layer of x[rows, H] (bf16)."""
    dev = _device_of(dl, ws)
    _check_rows(x, "x", torch.bfloat16, dl.shape.hidden, dev)
    rows = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    _check_rows(out, "out", torch.bfloat16, dl.shape.hidden, dev)
    if out.shape[0] != rows:
        raise ValueError("out has %d rows, x has %d" % (out.shape[0], rows))
    N.moe_forward(dl.config(per_row_mode, gemv), dl.weights, x.data_ptr(), out.data_ptr(),
                  rows, ws.ptr, ws.nbytes, _stream(stream))
    return out


def route(dl: DeviceLayer, x: torch.Tensor, ws: Workspace, stream=None):
    """Router + top-k: (ids [rows, k] int32, wts [rows, k] fp32,
    logits [rows, E] fp32)."""
    _check_rows(x, "x", torch.bfloat16, dl.shape.hidden, _device_of(dl, ws))
    rows = x.shape[0]
    k, E = dl.shape.top_k, dl.shape.num_experts
    ids = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    wts = torch.empty((rows, k), dtype=torch.float32, device=x.device)
    logits = torch.empty((rows, E), dtype=torch.float32, device=x.device)
    N.moe_route(dl.cfg, dl.weights, x.data_ptr(), rows, ids.data_ptr(), wts.data_ptr(),
                logits.data_ptr(), ws.ptr, ws.nbytes, _stream(stream))
    return ids, wts, logits


def _union_from_bytes(raw: torch.Tensor) -> dict:
    t = N.UnionTable.from_buffer_copy(bytes(raw.cpu().numpy().tobytes()))
    U = t.num_union
    n = t.rows * t.top_k
    return {
        "U": U,
        "expert": [t.expert[i] for i in range(U)],
        "rowmask": [t.rowmask[i] for i in range(U)],
        "slot2u": [t.slot2u[i] for i in range(n)],
        "uslot": [[t.uslot[u][r] for r in range(N.MOE_MAX_ROWS)] for u in range(U)],
        "rows": t.rows, "top_k": t.top_k, "per_row_mode": t.per_row_mode,
    }


def union(dl: Optional[DeviceLayer], cfg: N.MoeConfig, ids: torch.Tensor,
          ws: Workspace, stream=None) -> dict:
    """Union of ids [rows, k] (device int32) built on the device."""
    _check_rows(ids, "ids", torch.int32, cfg.top_k, _device_of(dl, ws))
    rows = ids.shape[0]
    raw = torch.empty(C.sizeof(N.UnionTable), dtype=torch.uint8, device=ids.device)
    N.moe_union(cfg, dl.weights if dl is not None else None, ids.data_ptr(), rows,
                raw.data_ptr(), ws.ptr, ws.nbytes, _stream(stream))
    return _union_from_bytes(raw)


def read_routing(dl: DeviceLayer, ws: Workspace, rows: int, per_row_mode=False,
                 stream=None):
    """(ids, wts, union dict) of the last call on this workspace."""
    k = dl.shape.top_k
    dev = ws.buf.device
    ids = torch.empty((rows, k), dtype=torch.int32, device=dev)
    wts = torch.empty((rows, k), dtype=torch.float32, device=dev)
    raw = torch.empty(C.sizeof(N.UnionTable), dtype=torch.uint8, device=dev)
    N.moe_read_routing(dl.config(per_row_mode), ws.ptr, ws.nbytes, rows, ids.data_ptr(),
                       wts.data_ptr(), raw.data_ptr(), _stream(stream))
    return ids, wts, _union_from_bytes(raw)
