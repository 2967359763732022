"""ctypes binding of the C ABI in include/moe_router.h (argument marshalling
only: every step of the layer runs in the CUDA library).

The library is loaded from the package's in-tree build folder
(_build/libmoe_router.so).  If it has not been built, every call raises
RuntimeError; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

MOE_MAX_ROWS = 32
MOE_MAX_IDS = 256
MOE_CHUNK_ROWS = 8
MOE_CHUNK_IDS = 64
MOE_STATIC_WORKSPACE_BYTES = 10 << 20
MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID = 0, 1
MOE_ROUTER_BF16, MOE_ROUTER_NVFP4 = 0, 1
MOE_EXPERT_NVFP4, MOE_EXPERT_FP8, MOE_EXPERT_BF16 = 0, 1, 2

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_STATUS"}
DEV_STATUS = {0: "MOE_DEV_OK", 1: "MOE_DEV_BAD_EXPERT_ID",
              2: "MOE_DEV_MISALIGNED_PTR", 3: "MOE_DEV_WAIT_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


class Nvfp4Desc(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("scales", C.c_void_p),
                ("scale2", C.c_float)]


class MoeConfig(C.Structure):
    _fields_ = [("hidden", C.c_int), ("num_experts", C.c_int),
                ("router_width", C.c_int), ("top_k", C.c_int),
                ("moe_inter", C.c_int), ("shared_inter", C.c_int),
                ("scoring", C.c_int), ("norm_topk_prob", C.c_int),
                ("routed_scaling_factor", C.c_float), ("router_fmt", C.c_int),
                ("has_shared", C.c_int), ("shared_gate", C.c_int),
                ("per_row_mode", C.c_int), ("gemv_lever", C.c_int),
                ("t_layout", C.c_int), ("expert_fmt", C.c_int)]


class ExpertTable(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("scales", C.c_void_p),
                ("scale2", C.c_void_p)]


class MoeWeights(C.Structure):
    _fields_ = [("router_bf16", C.c_void_p), ("router_nvfp4", Nvfp4Desc),
                ("correction_bias", C.c_void_p), ("gate", ExpertTable),
                ("up", ExpertTable), ("down", ExpertTable),
                ("shared_gate_proj", Nvfp4Desc), ("shared_up_proj", Nvfp4Desc),
                ("shared_down_proj", Nvfp4Desc),
                ("shared_expert_gate", C.c_void_p)]


class UnionTable(C.Structure):
    _fields_ = [("num_union", C.c_int32), ("rows", C.c_int32),
                ("top_k", C.c_int32), ("per_row_mode", C.c_int32),
                ("expert", C.c_int32 * MOE_MAX_IDS),
                ("rowmask", C.c_uint32 * MOE_MAX_IDS),
                ("slot2u", C.c_uint8 * MOE_MAX_IDS),
                ("uslot", (C.c_uint8 * MOE_MAX_ROWS) * MOE_MAX_IDS)]


EXPORTS = ("moe_abi_version", "moe_last_error", "moe_check_config",
           "moe_workspace_size", "moe_workspace_init", "moe_route", "moe_union",
           "moe_forward", "moe_forward_timed", "moe_read_routing",
           "moe_read_device_status", "moe_forward_static", "moe_nvfp4_to_t_layout")

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the in-tree CUDA library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                "CUDA library %s is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')" % path)
        L = C.CDLL(path)
        vp, sz, i = C.c_void_p, C.c_size_t, C.c_int
        L.moe_abi_version.restype = i
        L.moe_last_error.restype = C.c_char_p
        L.moe_check_config.argtypes = [C.POINTER(MoeConfig)]
        L.moe_workspace_size.restype = sz
        L.moe_workspace_size.argtypes = [C.POINTER(MoeConfig)]
        L.moe_workspace_init.argtypes = [vp, sz, vp]
        L.moe_route.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), vp, i,
                                vp, vp, vp, vp, sz, vp]
        L.moe_union.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), vp, i,
                                vp, vp, sz, vp]
        L.moe_forward.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), vp,
                                  vp, i, vp, sz, vp]
        L.moe_forward_timed.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights),
                                        vp, vp, i, vp, sz, vp, C.POINTER(vp)]
        L.moe_read_routing.argtypes = [C.POINTER(MoeConfig), vp, sz, i, vp, vp,
                                       vp, vp]
        L.moe_read_device_status.argtypes = [vp, sz, C.POINTER(C.c_int), vp]
        L.moe_forward_static.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights),
                                         vp, vp, i, vp]
        L.moe_nvfp4_to_t_layout.argtypes = [vp, vp, i, i, i, vp, vp, vp]
        for name in EXPORTS[2:]:
            if name != "moe_workspace_size":
                getattr(L, name).restype = i
        _lib = L
        return L


def _check(status: int):
    if status != 0:
        raise MoeError(status, lib().moe_last_error().decode())


# ---------------------------------------------------------------------------
# The C entry points, one-to-one
# ---------------------------------------------------------------------------

def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_check_config(cfg: MoeConfig):
    _check(lib().moe_check_config(C.byref(cfg)))


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = lib().moe_workspace_size(C.byref(cfg))
    if n == 0:
        moe_check_config(cfg)
    return n


def moe_workspace_init(ws: int, ws_bytes: int, stream: int = 0):
    _check(lib().moe_workspace_init(ws, ws_bytes, stream))


def moe_route(cfg, w, x: int, rows: int, ids: int, wts: int, logits: int,
              ws: int, ws_bytes: int, stream: int = 0):
    _check(lib().moe_route(C.byref(cfg), C.byref(w), x, rows, ids, wts,
                           logits, ws, ws_bytes, stream))


def moe_union(cfg, w, ids: int, rows: int, out: int, ws: int, ws_bytes: int,
              stream: int = 0):
    _check(lib().moe_union(C.byref(cfg), C.byref(w) if w is not None else None,
                           ids, rows, out, ws, ws_bytes, stream))


def moe_forward(cfg, w, x: int, out: int, rows: int, ws: int, ws_bytes: int,
                stream: int = 0):
    _check(lib().moe_forward(C.byref(cfg), C.byref(w), x, out, rows, ws,
                             ws_bytes, stream))


def moe_forward_timed(cfg, w, x: int, out: int, rows: int, ws: int,
                      ws_bytes: int, stream: int, events):
    """events: two cudaEvent_t handles (ints), recorded before and after the
    layer kernel."""
    arr = (C.c_void_p * 2)(*events)
    _check(lib().moe_forward_timed(C.byref(cfg), C.byref(w), x, out, rows, ws,
                                   ws_bytes, stream, arr))


def moe_read_routing(cfg, ws: int, ws_bytes: int, rows: int, ids: int,
                     wts: int, uni: int, stream: int = 0):
    _check(lib().moe_read_routing(C.byref(cfg), ws, ws_bytes, rows, ids, wts,
                                  uni, stream))


def moe_forward_static(cfg, w, x: int, out: int, rows: int, stream: int = 0):
    """moe_forward with the library's own static device workspace (for
    callers that cannot allocate device memory; see the header)."""
    _check(lib().moe_forward_static(C.byref(cfg), C.byref(w), x, out, rows, stream))


def moe_nvfp4_to_t_layout(packed: int, scales: int, count: int, n_out: int, k_in: int,
                          packed_t: int, scales_t: int, stream: int = 0):
    """Convert `count` stacked NVFP4 [n_out][k_in] matrices to the t layout
    (see the header)."""
    _check(lib().moe_nvfp4_to_t_layout(packed, scales, count, n_out, k_in, packed_t,
                                       scales_t, stream))


def moe_read_device_status(ws: int, ws_bytes: int, stream: int = 0) -> int:
    code = C.c_int(0)
    st = lib().moe_read_device_status(ws, ws_bytes, C.byref(code), stream)
    if st not in (0, 5):
        _check(st)
    return code.value
