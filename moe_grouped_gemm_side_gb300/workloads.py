"""Seeded synthetic inputs shaped like the pages' MoE workloads.

This module draws inputs only: token-count histograms, dense operands and
their FP8 encoding.  It holds none of the grouped GEMM's own arithmetic (no
offsets, padding, tiles or products), so both the CUDA path and the CPU oracle
can consume what it makes without sharing any of the method's code.

Histograms (numpy ``default_rng(seed)``):

* ``counts_uniformish``  -- the near-uniform 8-expert example of "MoE GroupGEMM
  padding under expert skew", "Work a near-uniform routing example".
* ``counts_issue32``     -- the 32-expert histogram printed in "Query on
  performance-modeling of MoE Grouped GEMM", "Background".
* ``counts_zipf_decode`` -- masked decode: valid_m[e] from a Zipf(s) law
  truncated to 0..M_max, with at least ``min_zeros`` empty experts.
* ``counts_zipf_prefill``-- skewed prefill: Zipf(s) over expert ranks placed
  on experts by a seeded permutation, then a multinomial of all assignments.
* ``counts_dirichlet``   -- weight-gradient: Dirichlet(alpha) shares of a
  token total, rounded by the largest-remainder rule.

Dense operands come from ``torch.Generator`` seeded per tensor, drawn in
float32 on the requested device and rounded to bf16 (round-to-nearest-even).
FP8 operands are E4M3 codes with one UE8M0 exponent byte per block: per
(row, 128 K) for activations, per (128 N, 128 K) for weights.  The scale byte
of a block with absolute maximum a is s = clamp(ceil(log2(a / 448)) + 127,
1, 254) (s = 127 for an all-zero block) and each element is encoded as
e4m3(x / 2^(s - 127)) rounded to nearest even, which never exceeds 448.
FP4 weights (dtype "fp8xfp4") are E2M1 codes, two per byte (element 2i in
the low nibble of byte i), with one UE8M0 byte per (row, 32 K) chosen the
same way against the largest E2M1 magnitude 6; each element takes the
nearest E2M1 magnitude (the lower one on a tie).
"""

from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np
import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F
UE8M0_NAN_CODE = 0xFF

ISSUE32_COUNTS = [4, 1026, 1799, 166, 694, 753, 0, 16, 0, 240, 1119, 19, 6, 0, 46,
                  659, 10, 0, 112, 808, 181, 0, 28, 22, 90, 0, 176, 0, 37, 5, 10, 22]
UNIFORMISH_COUNTS = [17, 17, 17, 17, 16, 16, 16, 16]
CONCENTRATED_COUNTS = [100, 32, 0, 0, 0, 0, 0, 0]


# --------------------------------------------------------------------------
# histograms
# --------------------------------------------------------------------------

def counts_uniformish() -> List[int]:
    return list(UNIFORMISH_COUNTS)


def counts_issue32() -> List[int]:
    return list(ISSUE32_COUNTS)


def counts_zipf_decode(seed: int = 1003, E: int = 16, M_max: int = 256,
                       s: float = 1.1, min_zeros: int = 3) -> List[int]:
    """valid_m[e] ~ p(v) proportional to (v+1)^-s over v = 0..M_max.  If fewer
    than ``min_zeros`` draws are 0, the smallest non-zero draws (ties to the
    lower expert index) are set to 0 until there are."""
    rng = np.random.default_rng(seed)
    v = np.arange(M_max + 1)
    p = (v + 1.0) ** -s
    p /= p.sum()
    out = [int(x) for x in rng.choice(M_max + 1, size=E, p=p)]
    while sum(1 for x in out if x == 0) < min_zeros:
        nz = [(x, i) for i, x in enumerate(out) if x > 0]
        _, i = min(nz)
        out[i] = 0
    return out


def counts_zipf_prefill(seed: int = 1004, E: int = 64, total: int = 32768,
                        s: float = 1.2) -> List[int]:
    """Rank r = 1..E gets probability proportional to r^-s; a seeded
    permutation decides which expert holds which rank; counts are a
    multinomial draw of ``total`` assignments."""
    rng = np.random.default_rng(seed)
    r = np.arange(1, E + 1)
    p = r ** -s
    p = p / p.sum()
    perm = rng.permutation(E)
    pe = np.empty(E)
    pe[perm] = p
    return [int(x) for x in rng.multinomial(total, pe)]


def counts_dirichlet(seed: int = 1005, E: int = 32, total: int = 65536,
                     alpha: float = 0.3) -> List[int]:
    """Shares w ~ Dirichlet(alpha * 1_E); counts floor(w * total), the
    remainder handed out one by one by largest fractional part (ties to the
    lower index)."""
    rng = np.random.default_rng(seed)
    w = rng.dirichlet(np.full(E, alpha))
    x = w * total
    c = np.floor(x).astype(np.int64)
    rem = int(total - c.sum())
    frac = x - c
    order = sorted(range(E), key=lambda i: (-frac[i], i))
    for i in order[:rem]:
        c[i] += 1
    return [int(v) for v in c]


def counts_random(seed: int, E: int, max_count: int, zero_frac: float = 0.25) -> List[int]:
    """Uniform random histogram with a share of empty experts (test inputs)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, max_count + 1, size=E)
    c[rng.random(E) < zero_frac] = 0
    return [int(v) for v in c]


# --------------------------------------------------------------------------
# dense operands
# --------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal_f32(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def normal_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    return normal_f32(shape, seed, device, std).to(torch.bfloat16)


def integer_bf16(shape, seed: int, device="cpu", lo: int = -2, hi: int = 2) -> torch.Tensor:
    """Small integers as bf16: with K <= 256 every fp32 partial sum is exact."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device).to(torch.bfloat16)


def _ceil_log2(v: torch.Tensor) -> torch.Tensor:
    """ceil(log2(v)) for positive float32 v, exact (frexp based)."""
    m, e = torch.frexp(v)
    return torch.where(m == 0.5, e - 1, e)


def _scale_bytes(amax: torch.Tensor, fmax: float = E4M3_MAX) -> torch.Tensor:
    s = _ceil_log2(torch.clamp(amax, min=torch.finfo(torch.float32).tiny) / fmax) + 127
    s = torch.clamp(s, 1, 254)
    s = torch.where(amax == 0, torch.full_like(s, 127), s)
    return s.to(torch.uint8)


def _encode_e4m3(x: torch.Tensor, exp_bytes: torch.Tensor) -> torch.Tensor:
    scale = torch.pow(2.0, exp_bytes.to(torch.float32) - 127.0)
    y = x / scale
    assert bool((y.abs() <= E4M3_MAX).all()), "block scale too small"
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def quantize_rows_fp8(x: torch.Tensor):
    """x float32 [R, K] -> (codes uint8 [R, K], sf uint8 [K/128, R])."""
    R, K = x.shape
    assert K % 128 == 0
    xb = x.reshape(R, K // 128, 128)
    sf = _scale_bytes(xb.abs().amax(dim=2))                    # [R, K/128]
    codes = _encode_e4m3(xb, sf[:, :, None]).reshape(R, K)
    return codes, sf.t().contiguous()


def quantize_weight_fp8(w: torch.Tensor):
    """w float32 [N, K] -> (codes uint8 [N, K], sf uint8 [K/128, N/128])."""
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    wb = w.reshape(N // 128, 128, K // 128, 128)
    sf = _scale_bytes(wb.abs().amax(dim=(1, 3)))               # [N/128, K/128]
    codes = _encode_e4m3(wb, sf[:, None, :, None]).reshape(N, K)
    return codes, sf.t().contiguous()


def quantize_weight_mx4(w: torch.Tensor):
    """w float32 [N, K] -> (packed uint8 [N, K/2], sf uint8 [N, K/32])."""
    N, K = w.shape
    assert K % 32 == 0
    wb = w.reshape(N, K // 32, 32)
    sf = _scale_bytes(wb.abs().amax(dim=2), E2M1_MAX)            # [N, K/32]
    y = wb / torch.pow(2.0, sf.to(torch.float32) - 127.0)[:, :, None]
    mags = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float32, device=w.device)
    code = (y.abs()[..., None] - mags).abs().argmin(dim=-1)      # lowest index on a tie
    code = (code | torch.where(y < 0, 8, 0)).to(torch.uint8).reshape(N, K)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), sf.contiguous()


def integer_e2m1_packed(shape, seed: int, device="cpu"):
    """Packed E2M1 codes [..., K/2] of the values -2..2 (exact in E2M1)."""
    *lead, K = shape
    lut = torch.tensor([0xC, 0xA, 0x0, 0x2, 0x4], dtype=torch.uint8)   # -2, -1, 0, 1, 2
    g = torch.Generator().manual_seed(int(seed))
    codes = lut[torch.randint(0, 5, tuple(lead) + (K,), generator=g)]
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).contiguous().to(device)


@dataclass
class Operands:
    """A grouped-GEMM operand set.  ``A``/``B`` are bf16 tensors for the bf16
    path and uint8 E4M3 codes for the FP8 path, in which case ``SFA``/``SFB``
    hold the UE8M0 bytes (``None`` for bf16)."""
    A: torch.Tensor
    B: torch.Tensor
    SFA: Optional[torch.Tensor] = None
    SFB: Optional[torch.Tensor] = None


def expert_weight(e: int, N: int, K: int, dtype: str, seed: int, device="cpu",
                  std: float = 1.0):
    """The weights of expert e alone, exactly as make_weights draws them on
    the same device: (bf16 values, None) or (codes, scales)."""
    if dtype == "bf16":
        return normal_bf16((N, K), seed * 1000 + e, device, std), None
    w = normal_f32((N, K), seed * 1000 + e, device, std)
    return quantize_weight_mx4(w) if dtype == "fp8xfp4" else quantize_weight_fp8(w)


def make_weights(E: int, N: int, K: int, dtype: str, seed: int, device="cpu",
                 std: float = 1.0):
    """Expert weights [E, N, K] (+ SFB [E, K/128, N/128] for fp8), one seeded
    draw per expert."""
    if dtype == "bf16":
        B = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
        for e in range(E):
            B[e] = expert_weight(e, N, K, dtype, seed, device, std)[0]
        return B, None
    if dtype == "fp8xfp4":
        B = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
        SFB = torch.empty((E, N, K // 32), dtype=torch.uint8, device=device)
    else:
        B = torch.empty((E, N, K), dtype=torch.uint8, device=device)
        SFB = torch.empty((E, K // 128, N // 128), dtype=torch.uint8, device=device)
    for e in range(E):
        B[e], SFB[e] = expert_weight(e, N, K, dtype, seed, device, std)
    return B, SFB


def make_rows(R: int, K: int, dtype: str, seed: int, device="cpu", std: float = 1.0):
    """Activation rows [R, K] (+ SFA [K/128, R] for fp8)."""
    if dtype == "bf16":
        return normal_bf16((R, K), seed, device, std), None
    codes = torch.empty((R, K), dtype=torch.uint8, device=device)
    sf = torch.empty((K // 128, R), dtype=torch.uint8, device=device)
    chunk = max(1, (1 << 26) // max(K, 1))
    for r0 in range(0, R, chunk):
        r1 = min(R, r0 + chunk)
        x = normal_f32((r1 - r0, K), seed * 1000 + r0 // chunk, device, std)
        codes[r0:r1], sf[:, r0:r1] = quantize_rows_fp8(x)
    return codes, sf


def make_contiguous(E: int, rows_cap: int, N: int, K: int, dtype: str, seed: int,
                    device="cpu", a_std: float = 1.0, b_std: float = 1.0) -> Operands:
    """Operands of the M-grouped contiguous form: A [rows_cap, K] (every row
    drawn; the caller decides which rows hold which expert), B [E, N, K]."""
    A, SFA = make_rows(rows_cap, K, dtype, seed, device, a_std)
    B, SFB = make_weights(E, N, K, dtype, seed + 1, device, b_std)
    return Operands(A, B, SFA, SFB)


def make_masked(E: int, M_max: int, N: int, K: int, dtype: str, seed: int,
                device="cpu", a_std: float = 1.0, b_std: float = 1.0) -> Operands:
    """Operands of the masked form: A [E, M_max, K], SFA [E, K/128, M_max]."""
    A2, SFA2 = make_rows(E * M_max, K, dtype, seed, device, a_std)
    A = A2.reshape(E, M_max, K)
    SFA = None
    if SFA2 is not None:
        SFA = SFA2.reshape(K // 128, E, M_max).permute(1, 0, 2).contiguous()
    B, SFB = make_weights(E, N, K, dtype, seed + 1, device, b_std)
    return Operands(A, B, SFA, SFB)


def make_kgrouped(T_cap: int, N: int, K: int, seed: int, device="cpu"):
    """Operands of the K-grouped form: dY [T_cap, N], X [T_cap, K] bf16."""
    return normal_bf16((T_cap, N), seed, device), normal_bf16((T_cap, K), seed + 1, device)


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------

WORKLOADS: Dict[str, dict] = {
    "contig_bf16_e8_n256_k256": dict(
        form="contiguous", dtype="bf16", E=8, N=256, K=256, align_q=32, seed=1001,
        a_std=1.0, b_std=1.0, counts=counts_uniformish),
    "contig_bf16_e32_n4096_k2048": dict(
        form="contiguous", dtype="bf16", E=32, N=4096, K=2048, align_q=128, seed=1002,
        a_std=2048 ** -0.5, b_std=2048 ** -0.5, counts=counts_issue32),
    "masked_fp8_e16_m256_n4096_k7168": dict(
        form="masked", dtype="fp8", E=16, M_max=256, N=4096, K=7168, seed=1003,
        a_std=1.0, b_std=1.0, counts=counts_zipf_decode),
    # the decode case with FP4 weights (half the weight bytes)
    "masked_fp8xfp4_e16_m256_n4096_k7168": dict(
        form="masked", dtype="fp8xfp4", E=16, M_max=256, N=4096, K=7168, seed=1003,
        a_std=1.0, b_std=1.0, counts=counts_zipf_decode),
    "prefill_fp8_e64_t32768_n4096_k7168": dict(
        form="contiguous", dtype="fp8", E=64, N=4096, K=7168, align_q=128, seed=1004,
        a_std=1.0, b_std=1.0, counts=counts_zipf_prefill,
        second=dict(N=7168, K=2048)),
    # the same two GEMMs as one expert FFN: GEMM1's SwiGLU epilogue writes the
    # E4M3 activations (and scales) that GEMM2 reads
    "prefill_ffn_fp8_e64_t32768_n4096_k7168": dict(
        form="contiguous", dtype="fp8", E=64, N=4096, K=7168, align_q=128, seed=1004,
        a_std=1.0, b_std=7168 ** -0.5, counts=counts_zipf_prefill,
        second=dict(N=7168, K=2048), swiglu=True),
    "prefill_ffn_fp8_e16_t8192_n4096_k7168": dict(
        form="contiguous", dtype="fp8", E=16, N=4096, K=7168, align_q=128, seed=1006,
        a_std=1.0, b_std=7168 ** -0.5, counts=lambda: counts_zipf_prefill(seed=1006, E=16, total=8192),
        second=dict(N=7168, K=2048), swiglu=True),
    "prefill_fp8xfp4_e64_t32768_n4096_k7168": dict(
        form="contiguous", dtype="fp8xfp4", E=64, N=4096, K=7168, align_q=128, seed=1004,
        a_std=1.0, b_std=1.0, counts=counts_zipf_prefill,
        second=dict(N=7168, K=2048)),
    "prefill_bf16_e64_t32768_n4096_k7168": dict(
        form="contiguous", dtype="bf16", E=64, N=4096, K=7168, align_q=128, seed=1004,
        a_std=7168 ** -0.5, b_std=7168 ** -0.5, counts=counts_zipf_prefill,
        second=dict(N=7168, K=2048)),
    "prefill_fp8_e16_t8192_n4096_k7168": dict(
        form="contiguous", dtype="fp8", E=16, N=4096, K=7168, align_q=128, seed=1006,
        a_std=1.0, b_std=1.0, counts=lambda: counts_zipf_prefill(seed=1006, E=16, total=8192)),
    "kgrouped_bf16_e32_t65536_n4096_k2048": dict(
        form="kgrouped", dtype="bf16", E=32, N=4096, K=2048, T=65536, seed=1005,
        counts=counts_dirichlet),
}
