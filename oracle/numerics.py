"""Operand decoders and block-scale dequantisation (oracle; test infrastructure).

Encodings, from their published definitions:

* bf16: the upper 16 bits of an IEEE binary32; widening to float64 is exact.
* FP8 E4M3 (the "fn" variant used for MoE GEMMs): 1 sign bit, 4 exponent bits
  with bias 7, 3 mantissa bits.  Exponent field 0 is subnormal
  (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
* UE8M0: an unsigned 8-bit exponent, value 2^(s-127); 0xFF is NaN.

Block scales ("flops/deepgemm-grouped-masked-moe-gemm", "Workarounds": FP8
with per-group scaling; on SM100 the scales are UE8M0 power-of-two bytes).
The pages give no group sizes; these follow the workload description: one
scale per (token row, 128 K) for activations and one per (128 N, 128 K) block
for weights.
"""

import numpy as np


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes -> float64, from the bit-field definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where((exp == 0xF) & (man == 0x7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    """uint8 UE8M0 scale bytes -> float64 2^(s-127); 0xFF -> NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    v = np.exp2(c - 127.0)
    return np.where(c == 255.0, np.nan, v)


def dequant_rows(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Activation rows with one scale per (row, 128-wide K block).

    codes: uint8 [R, K] E4M3; sf: uint8 [K/128, R] (K-block major, one byte
    per row).  Returns float64 [R, K] with
    out[r, k] = e4m3(codes[r, k]) * 2^(sf[k // 128, r] - 127).
    """
    R, K = codes.shape
    assert K % 128 == 0 and sf.shape == (K // 128, R)
    scale = decode_ue8m0(sf).T                      # [R, K/128]
    return decode_e4m3(codes) * np.repeat(scale, 128, axis=1)


def dequant_weight(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """One expert's weight [N, K] with one scale per 128 x 128 block.

    codes: uint8 [N, K] E4M3; sf: uint8 [K/128, N/128].  Returns float64 with
    out[n, k] = e4m3(codes[n, k]) * 2^(sf[k // 128, n // 128] - 127).
    """
    N, K = codes.shape
    assert N % 128 == 0 and K % 128 == 0 and sf.shape == (K // 128, N // 128)
    scale = decode_ue8m0(sf).T                      # [N/128, K/128]
    full = np.repeat(np.repeat(scale, 128, axis=0), 128, axis=1)
    return decode_e4m3(codes) * full
