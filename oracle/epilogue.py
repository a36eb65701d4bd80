"""SwiGLU and FP8 re-quantisation of a GEMM1 output (oracle; test
infrastructure: only tests/, smoke() and bench.py's CPU legs use it).

"flops/deepgemm-grouped-masked-moe-gemm", "Workarounds": the fused MoE
kernel (Mega MoE) runs the expert's SwiGLU between the two grouped GEMMs,
and the FP8 path feeds the second GEMM per-group-scaled E4M3 activations
with UE8M0 scales.  The pages name SwiGLU but do not write it out; this is
the standard definition (Shazeer, "GLU Variants Improve Transformer"):

    h = SiLU(g) * u,   SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x)),

with g and u the two halves of GEMM1's output for the same feature.  The
re-quantisation follows the activation format of the first GEMM: one UE8M0
byte per (token row, 128 features), the smallest power of two 2^(s-127) with
max|h| <= 448 * 2^(s-127) (448 = largest finite E4M3), blocks of zeros get
s = 127; each element is rounded to the nearest E4M3 value of h / 2^(s-127)
(ties to the even code), magnitudes beyond 448 saturating to 448.  All in
float64.
"""

import numpy as np

E4M3_MAX = 448.0


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) in float64, written so that exp never overflows."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))                       # in (0, 1]
    sig = np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return x * sig


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    return silu(g) * np.asarray(u, dtype=np.float64)


def _e4m3_magnitudes() -> np.ndarray:
    """The 127 non-negative finite E4M3 values, ascending; index = code."""
    codes = np.arange(127)
    exp, man = codes >> 3, codes & 7
    return np.where(exp == 0, man / 8.0 * 2.0 ** -6, (1.0 + man / 8.0) * np.exp2(exp - 7.0))


_MAG = _e4m3_magnitudes()


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> E4M3 codes (uint8): nearest value, ties to the even code,
    magnitudes above 448 saturate to 448 (code 0x7E); the sign goes in bit 7
    (negative zero keeps it)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_MAG, a, side="left"), 0, 126)   # first value >= a
    lo = np.clip(hi - 1, 0, 126)
    d_hi, d_lo = _MAG[hi] - a, a - _MAG[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def ue8m0_for_amax(amax: np.ndarray) -> np.ndarray:
    """Smallest s with amax <= 448 * 2^(s-127), clamped to [1, 254]; 127 for
    amax == 0.  Exact: amax = m * 2^e with m in [0.5, 1) and 448 = 0.875 * 2^9,
    so the bound holds at s = e + 118 when m <= 0.875 and needs s = e + 119
    otherwise."""
    amax = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(amax)
    s = e.astype(np.int64) + 118 + (m > 0.875)
    s = np.clip(s, 1, 254)
    return np.where(amax == 0, 127, s).astype(np.uint8)


def quantize_blocks(h: np.ndarray):
    """h float64 [R, F] -> (codes uint8 [R, F], sf uint8 [F/128, R])."""
    h = np.asarray(h, dtype=np.float64)
    R, F = h.shape
    assert F % 128 == 0
    hb = h.reshape(R, F // 128, 128)
    sf = ue8m0_for_amax(np.abs(hb).max(axis=2))                    # [R, F/128]
    scale = np.exp2(sf.astype(np.float64) - 127.0)[:, :, None]
    codes = encode_e4m3(hb / scale).reshape(R, F)
    return codes, np.ascontiguousarray(sf.T)


def gate_up_halves(H: np.ndarray):
    """GEMM1 output H [R, 2F] whose weight rows are interleaved in 128-row
    blocks (gate rows of features 128j..128j+127, then their up rows) ->
    (g, u), each [R, F]."""
    R, N2 = H.shape
    assert N2 % 256 == 0
    Hb = H.reshape(R, N2 // 256, 2, 128)
    return Hb[:, :, 0, :].reshape(R, N2 // 2), Hb[:, :, 1, :].reshape(R, N2 // 2)
