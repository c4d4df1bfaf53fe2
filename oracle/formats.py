"""Decoding of the 4-bit block-scaled weight format (oracle; test infrastructure only).

Sources:
  * Qwen3.8-Flash-Next DGX Spark deployment notes, section "NVFP4 code 和 scale
    如何反量化": a byte carries two codes (low and high nibble); the low three
    bits of a code select a magnitude from {0, 0.5, 1, 1.5, 2, 3, 4, 6}; the
    top bit is the sign; the value is the FP4 value times the FP8 block scale
    (one per 16 values) times the FP32 global scale.
  * Same page, section "一个 160 维向量在 packed 文件中占 90 字节" and the
    packed-file build step: a row stores its codes first, then its block
    scales (columns concatenated per row).
  * FP8 E4M3 (OCP 8-bit floating point specification): 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
    (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
"""
from __future__ import annotations

import numpy as np

# The eight magnitudes a code's low three bits select, in code order.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_value(code: np.ndarray) -> np.ndarray:
    """FP4 (E2M1) code (0..15) -> value; bit 3 is the sign."""
    code = np.asarray(code, dtype=np.uint8)
    mag = E2M1_MAGNITUDES[code & 7]
    return np.where((code >> 3) & 1, -mag, mag)


def e4m3_value(byte: np.ndarray) -> np.ndarray:
    """FP8 E4M3 byte -> value (fp64, exact), per the OCP definition."""
    b = np.asarray(byte, dtype=np.uint8).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, subnormal, normal) * sign
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> fp64 value (exact): the top half of an fp32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def unpack_codes(code_bytes: np.ndarray) -> np.ndarray:
    """``[rows, n]`` bytes -> ``[rows, 2n]`` codes; element 2j is the low nibble of byte j."""
    b = np.asarray(code_bytes, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def dequantize(packed: np.ndarray, cols: int, global_scale: float = 1.0) -> np.ndarray:
    """Canonical packed rows ``[rows, cols/2 + cols/16]`` -> fp64 matrix ``[rows, cols]``.

    value = FP4 code value * FP8 block scale (per 16 columns) * FP32 global scale.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    assert packed.shape[-1] == cols // 2 + cols // 16, (packed.shape, cols)
    codes = unpack_codes(packed[..., : cols // 2])
    scales = e4m3_value(packed[..., cols // 2:])
    blocks = e2m1_value(codes).reshape(packed.shape[:-1] + (cols // 16, 16))
    return (blocks * scales[..., None]).reshape(packed.shape[:-1] + (cols,)) * float(np.float32(global_scale))
