"""Operand decoders and block-scale dequantisation (oracle; test infrastructure).

Encodings, from their published definitions:

* bf16: the upper 16 bits of an IEEE binary32; widening to float64 is exact.
* FP8 E4M3 (the "fn" variant used for MoE GEMMs): 1 sign bit, 4 exponent bits
  with bias 7, 3 mantissa bits.  Exponent field 0 is subnormal
  (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
* UE8M0: an unsigned 8-bit exponent, value 2^(s-127); 0xFF is NaN.
* FP4 E2M1 (OCP Microscaling formats): 1 sign bit, 2 exponent bits with
  bias 1, 1 mantissa bit; exponent field 0 is subnormal (m/2); no infinity
  and no NaN.  Two codes per byte, element 2i in the low nibble of byte i.

Block scales ("flops/deepgemm-grouped-masked-moe-gemm", "Workarounds": FP8
with per-group scaling; on SM100 the scales are UE8M0 power-of-two bytes).
The pages give no group sizes; these follow the workload description: one
scale per (token row, 128 K) for activations and one per (128 N, 128 K) block
for weights.  FP4 weights ("flops/deepgemm-grouped-masked-moe-gemm",
"Workarounds": FP8xFP4 linear layers; the pages give no format) follow the
OCP MX convention: one UE8M0 scale per (weight row, 32 consecutive K).
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


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """4-bit E2M1 codes (values 0..15 in any integer array) -> float64, from
    the bit-field definition."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    exp = (c >> 1) & 0x3
    man = c & 0x1
    normal = (1.0 + man / 2.0) * np.exp2(exp.astype(np.float64) - 1.0)
    subnormal = man / 2.0
    mag = np.where(exp == 0, subnormal, normal)
    return np.where(sign == 1, -mag, mag)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [R, K/2] with two codes per byte -> codes [R, K] (element 2i =
    low nibble of byte i, element 2i+1 = high nibble)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant_weight_mx4(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """One expert's E2M1 weight [N, K] with one scale per (row, 32 K).

    packed: uint8 [N, K/2] (unpack_e2m1 order); sf: uint8 [N, K/32].
    Returns float64 with out[n, k] = e2m1(code[n, k]) * 2^(sf[n, k // 32] - 127).
    """
    codes = unpack_e2m1(packed)
    N, K = codes.shape
    assert K % 32 == 0 and sf.shape == (N, K // 32)
    return decode_e2m1(codes) * np.repeat(decode_ue8m0(sf), 32, axis=1)
