"""Independent decoders used by the tests to pin the oracle.

They decode with library routines (torch's float8_e4m3fn and bfloat16 views)
and the published E2M1 value table in tests/golden/e2m1_values.txt; nothing
here is shared with the oracle or with the CUDA path.
"""
import os

import numpy as np
import torch

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def e2m1_table() -> np.ndarray:
    vals = np.zeros(16, dtype=np.float64)
    seen = set()
    with open(os.path.join(_GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            vals[int(code)] = float(val)
            seen.add(int(code))
    assert seen == set(range(16))
    return vals


def e4m3_decode(codes) -> np.ndarray:
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def bf16_decode(bits) -> np.ndarray:
    t = torch.as_tensor(np.asarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).float().numpy().astype(np.float64)


def to_np(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16).numpy().view(np.uint16)
        else:
            t = t.numpy()
    return np.asarray(t)


def nvfp4_dense(packed, scales, scale2) -> np.ndarray:
    """Dequantise one NVFP4 matrix [N][K] to float64 via float32 products:
    w = (e2m1 * e4m3) * scale2 with the last multiply rounded to float32
    (the storage reading: low nibble = even input, one scale per 16 inputs)."""
    packed = to_np(packed).astype(np.uint8)
    scales = to_np(scales).astype(np.uint8)
    s2 = np.float32(np.asarray(to_np(scale2)).reshape(()))
    N, half = packed.shape
    K = half * 2
    tab = e2m1_table().astype(np.float32)
    codes = np.empty((N, K), dtype=np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    q = tab[codes]
    s = e4m3_decode(scales).astype(np.float32)
    s = np.repeat(s, 16, axis=1)
    w = (q * s).astype(np.float32) * s2
    return w.astype(np.float32).astype(np.float64)


def fp8_dense(packed, scale2) -> np.ndarray:
    """One FP8 matrix [N][K] (E4M3 codes, one fp32 scale2): w = e4m3 * scale2
    with the multiply rounded to float32."""
    codes = to_np(packed).astype(np.uint8)
    s2 = np.float32(np.asarray(to_np(scale2)).reshape(()))
    q = e4m3_decode(codes).astype(np.float32)
    return (q * s2).astype(np.float32).astype(np.float64)


def bf16_dense(packed, scale2) -> np.ndarray:
    """One BF16 matrix [N][K] stored as [N][2K] little-endian bytes, times
    scale2 (float32 multiply)."""
    b = to_np(packed).astype(np.uint8)
    bits = np.ascontiguousarray(b).view("<u2")
    s2 = np.float32(np.asarray(to_np(scale2)).reshape(()))
    q = bf16_decode(bits).astype(np.float32)
    return (q * s2).astype(np.float32).astype(np.float64)


def expert_dense(fmt, packed, scales, scale2) -> np.ndarray:
    if fmt == "fp8":
        return fp8_dense(packed, scale2)
    if fmt == "bf16":
        return bf16_dense(packed, scale2)
    return nvfp4_dense(packed, scales, scale2)
