"""ctypes binding of the CPU oracle in moe_oracle.c.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product path never does.  It
compiles moe_oracle.c with gcc on first use (plain IEEE arithmetic: no fast
math, no fused multiply-add contraction) into oracle/_build/.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's shared library (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_SO)
                and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
            return _SO
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off",
             "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
             "-lpthread"])
        os.replace(tmp, _SO)
        return _SO


FMT = {"nvfp4": 0, "fp8": 1, "bf16": 2}


class Mat(C.Structure):
    """orc_mat: one matrix of any of the formats (FMT)."""
    _fields_ = [("packed", C.c_void_p), ("scales", C.c_void_p),
                ("scale2", C.c_float), ("fmt", C.c_int)]


class Cfg(C.Structure):
    _fields_ = [("hidden", C.c_int), ("num_experts", C.c_int),
                ("top_k", C.c_int), ("moe_inter", C.c_int),
                ("shared_inter", C.c_int), ("scoring", C.c_int),
                ("norm_topk_prob", C.c_int),
                ("routed_scaling_factor", C.c_double),
                ("router_nvfp4", C.c_int), ("has_shared", C.c_int),
                ("shared_gated", C.c_int)]


class Weights(C.Structure):
    _fields_ = [("router_bf16", C.c_void_p), ("router_fp4", Mat),
                ("bias", C.c_void_p), ("gate", C.c_void_p),
                ("up", C.c_void_p), ("down", C.c_void_p),
                ("sh_gate", Mat), ("sh_up", Mat), ("sh_down", Mat),
                ("sh_gate_vec", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        L.orc_e2m1.restype = C.c_double
        L.orc_e2m1.argtypes = [C.c_int]
        L.orc_e4m3.restype = C.c_double
        L.orc_e4m3.argtypes = [C.c_int]
        L.orc_bf16.restype = C.c_double
        L.orc_bf16.argtypes = [C.c_uint16]
        L.orc_round_bf16.restype = C.c_uint16
        L.orc_round_bf16.argtypes = [C.c_double]
        L.orc_nvfp4_elem.restype = C.c_float
        L.orc_nvfp4_elem.argtypes = [C.POINTER(Mat), C.c_int, C.c_int,
                                     C.c_int]
        L.orc_mat_elem.restype = C.c_float
        L.orc_mat_elem.argtypes = [C.POINTER(Mat), C.c_int, C.c_int, C.c_int]
        L.orc_router_logits.argtypes = [C.POINTER(Cfg), C.POINTER(Weights),
                                        C.c_void_p, C.c_int, C.c_void_p]
        L.orc_topk.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p]
        L.orc_topk_row.argtypes = [C.POINTER(Cfg), C.POINTER(Weights),
                                   C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_route.argtypes = [C.POINTER(Cfg), C.POINTER(Weights), C.c_void_p,
                                C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_union.restype = C.c_int
        L.orc_union.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                C.c_void_p, C.c_void_p]
        L.orc_expert_mlp.argtypes = [C.c_int, C.c_int, C.POINTER(Mat),
                                     C.POINTER(Mat), C.POINTER(Mat),
                                     C.c_void_p, C.c_void_p]
        L.orc_forward.argtypes = [C.POINTER(Cfg), C.POINTER(Weights),
                                  C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                  C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.c_void_p]
        L.orc_weights_for_ids.argtypes = [C.POINTER(Cfg), C.c_void_p,
                                          C.c_void_p, C.c_void_p]
        L.orc_forward_ids.argtypes = [C.POINTER(Cfg), C.POINTER(Weights),
                                      C.c_void_p, C.c_int, C.c_void_p,
                                      C.c_int, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _np(t):
    """torch tensor (any device) or numpy array -> contiguous host numpy."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.uint16)
        t = t.numpy()
    return np.ascontiguousarray(t)


# ---------------------------------------------------------------------------
# Scalar helpers
# ---------------------------------------------------------------------------

def e2m1(code: int) -> float:
    return lib().orc_e2m1(code)


def e4m3(code: int) -> float:
    return lib().orc_e4m3(code)


def bf16(bits: int) -> float:
    return lib().orc_bf16(bits)


def round_bf16(v: float) -> int:
    return lib().orc_round_bf16(v)


class HostMat:
    """One matrix held in host memory for the oracle: NVFP4 (packed [N][K/2]
    codes, scales [N][K/16]), FP8 (packed [N][K] E4M3 codes) or BF16 (packed
    [N][2K] bytes, little-endian bfloat16); scale2 one fp32 per matrix."""

    def __init__(self, packed, scales, scale2, fmt: str = "nvfp4"):
        self.packed = _np(packed).astype(np.uint8, copy=False)
        self.fmt = fmt
        self.scale2 = float(np.asarray(_np(scale2)).reshape(()))
        self.N, width = self.packed.shape
        self.K = {"nvfp4": 2 * width, "fp8": width, "bf16": width // 2}[fmt]
        if fmt == "nvfp4":
            self.scales = _np(scales).astype(np.uint8, copy=False)
            assert self.scales.shape == (self.N, self.K // 16)
        else:
            self.scales = np.zeros(1, dtype=np.uint8)   # not read

    def c(self) -> Mat:
        return Mat(_ptr(self.packed), _ptr(self.scales), self.scale2, FMT[self.fmt])


def nvfp4_elem(m: HostMat, n: int, k: int) -> float:
    cm = m.c()
    return lib().orc_nvfp4_elem(C.byref(cm), m.K, n, k)


def mat_elem(m: HostMat, n: int, k: int) -> float:
    cm = m.c()
    return lib().orc_mat_elem(C.byref(cm), m.K, n, k)


def topk(keys, k: int) -> np.ndarray:
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.float64))
    ids = np.zeros(k, dtype=np.int32)
    lib().orc_topk(_ptr(keys), keys.size, k, _ptr(ids))
    return ids


def union(ids: np.ndarray):
    """Union of ids [rows, k] -> (U, union[U], slot2u[rows, k],
    rowmask[U])."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    rows, k = ids.shape
    uni = np.zeros(rows * k, dtype=np.int32)
    slot2u = np.zeros((rows, k), dtype=np.uint8)
    assert rows <= 32, "row masks are 32 bits wide"
    rowmask = np.zeros(rows * k, dtype=np.uint32)
    U = lib().orc_union(_ptr(ids), rows, k, _ptr(uni), _ptr(slot2u),
                        _ptr(rowmask))
    return U, uni[:U].copy(), slot2u, rowmask[:U].copy()


def expert_mlp(g: HostMat, u: HostMat, d: HostMat, x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    H, I = g.K, g.N
    y = np.zeros(H, dtype=np.float64)
    cg, cu, cd = g.c(), u.c(), d.c()
    lib().orc_expert_mlp(H, I, C.byref(cg), C.byref(cu), C.byref(cd),
                         _ptr(x), _ptr(y))
    return y


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

class OracleLayer:
    """Host copy of one layer's weights in the oracle's own descriptors.

    ``experts`` restricts which routed experts are copied to the host (the
    others stay NULL): the oracle only ever reads the experts it selects, so
    a caller that already knows the selection can avoid copying a whole
    multi-GB layer."""

    def __init__(self, layer, experts=None):
        s = layer.shape
        self.shape = s
        self.cfg = Cfg(s.hidden, s.num_experts, s.top_k, s.moe_inter,
                       s.shared_inter, 1 if s.scoring == "sigmoid" else 0,
                       int(s.norm_topk_prob), float(s.routed_scaling_factor),
                       1 if s.router_fmt == "nvfp4" else 0, int(s.has_shared),
                       int(s.shared_gated))
        self._keep = []
        w = Weights()
        if s.router_fmt == "nvfp4":
            m = layer.router_nvfp4
            self.router = HostMat(m.packed, m.scales, m.scale2)
            w.router_fp4 = self.router.c()
        else:
            self.router_bf16 = _np(layer.router_bf16)
            w.router_bf16 = _ptr(self.router_bf16)
        if layer.bias is not None:
            self.bias = _np(layer.bias).astype(np.float32)
            w.bias = _ptr(self.bias)
        E = s.num_experts
        self._subset = None if experts is None else set(int(e) for e in experts)
        sel = range(E) if experts is None else sorted(self._subset)
        arrs = {}
        for name in ("gate", "up", "down"):
            arr = (Mat * E)()
            src = getattr(layer, name)
            s2 = _np(src.scale2).astype(np.float32)
            for e in sel:
                hm = HostMat(src.packed[e], src.scales[e], s2[e], s.expert_fmt)
                self._keep.append(hm)
                arr[e] = hm.c()
            arrs[name] = arr
            self._keep.append(arr)
        w.gate = C.cast(arrs["gate"], C.c_void_p)
        w.up = C.cast(arrs["up"], C.c_void_p)
        w.down = C.cast(arrs["down"], C.c_void_p)
        if s.has_shared and layer.sh_gate is not None:
            for name, field in (("sh_gate", "sh_gate"), ("sh_up", "sh_up"),
                                ("sh_down", "sh_down")):
                m = getattr(layer, name)
                hm = HostMat(m.packed, m.scales, m.scale2, s.expert_fmt)
                self._keep.append(hm)
                setattr(w, field, hm.c())
            self.sh_vec = _np(layer.sh_gate_vec)
            w.sh_gate_vec = _ptr(self.sh_vec)
        self.w = w

    def router_logits(self, x) -> np.ndarray:
        x = _np(x).astype(np.uint16, copy=False)
        rows = x.shape[0]
        out = np.zeros((rows, self.shape.num_experts), dtype=np.float64)
        lib().orc_router_logits(C.byref(self.cfg), C.byref(self.w), _ptr(x),
                                rows, _ptr(out))
        return out

    def topk_row(self, logits_row):
        lr = np.ascontiguousarray(np.asarray(logits_row, dtype=np.float64))
        k = self.shape.top_k
        ids = np.zeros(k, dtype=np.int32)
        wts = np.zeros(k, dtype=np.float64)
        lib().orc_topk_row(C.byref(self.cfg), C.byref(self.w), _ptr(lr),
                           _ptr(ids), _ptr(wts))
        return ids, wts

    def route(self, x):
        x = _np(x).astype(np.uint16, copy=False)
        rows = x.shape[0]
        E, k = self.shape.num_experts, self.shape.top_k
        logits = np.zeros((rows, E), dtype=np.float64)
        ids = np.zeros((rows, k), dtype=np.int32)
        wts = np.zeros((rows, k), dtype=np.float64)
        lib().orc_route(C.byref(self.cfg), C.byref(self.w), _ptr(x), rows,
                        _ptr(logits), _ptr(ids), _ptr(wts))
        return logits, ids, wts

    def forward(self, x, nthreads: int = 1) -> dict:
        x = _np(x).astype(np.uint16, copy=False)
        rows = x.shape[0]
        if self._subset is not None:
            _, sel, _ = self.route(x)
            missing = set(int(e) for e in sel.ravel()) - self._subset
            if missing:
                raise ValueError("oracle selects experts %s that were not "
                                 "copied to the host" % sorted(missing))
        H, E, k = self.shape.hidden, self.shape.num_experts, self.shape.top_k
        out = np.zeros((rows, H), dtype=np.float64)
        outb = np.zeros((rows, H), dtype=np.uint16)
        ids = np.zeros((rows, k), dtype=np.int32)
        wts = np.zeros((rows, k), dtype=np.float64)
        logits = np.zeros((rows, E), dtype=np.float64)
        lib().orc_forward(C.byref(self.cfg), C.byref(self.w), _ptr(x), rows,
                          int(nthreads), _ptr(out), _ptr(outb), _ptr(ids),
                          _ptr(wts), _ptr(logits))
        return {"out": out, "out_bf16": outb, "ids": ids, "wts": wts,
                "logits": logits}

    def weights_for_ids(self, logits_row, sel):
        """Routing weights of the given experts of one row (slot order)."""
        lr = np.ascontiguousarray(np.asarray(logits_row, dtype=np.float64))
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
        assert sel.shape == (self.shape.top_k,)
        w = np.zeros(self.shape.top_k, dtype=np.float64)
        lib().orc_weights_for_ids(C.byref(self.cfg), _ptr(lr), _ptr(sel),
                                  _ptr(w))
        return w

    def forward_ids(self, x, sel, nthreads: int = 1) -> dict:
        """The layer with every row's experts given (sel [rows, k], slot
        order, distinct ids per row) instead of chosen by the top-k."""
        x = _np(x).astype(np.uint16, copy=False)
        rows = x.shape[0]
        H, E, k = self.shape.hidden, self.shape.num_experts, self.shape.top_k
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
        assert sel.shape == (rows, k)
        for r in range(rows):
            if len(set(int(v) for v in sel[r])) != k or sel[r].min() < 0 \
                    or sel[r].max() >= E:
                raise ValueError("row %d: ids must be %d distinct experts" % (r, k))
        if self._subset is not None:
            missing = set(int(e) for e in sel.ravel()) - self._subset
            if missing:
                raise ValueError("experts %s were not copied to the host"
                                 % sorted(missing))
        out = np.zeros((rows, H), dtype=np.float64)
        outb = np.zeros((rows, H), dtype=np.uint16)
        wts = np.zeros((rows, k), dtype=np.float64)
        logits = np.zeros((rows, E), dtype=np.float64)
        lib().orc_forward_ids(C.byref(self.cfg), C.byref(self.w), _ptr(x), rows,
                              _ptr(sel), int(nthreads), _ptr(out), _ptr(outb),
                              _ptr(wts), _ptr(logits))
        return {"out": out, "out_bf16": outb, "ids": sel.copy(), "wts": wts,
                "logits": logits}
