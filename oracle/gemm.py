"""The three MoE grouped GEMM forms in float64 (oracle; test infrastructure).

N and K are the same for every expert; only the token dimension varies
("flops/deepgemm-grouped-masked-moe-gemm", "Arithmetic intensity": grouped
GEMM groups only the M axis and needs N and K fixed).  Conventions: tokens are
rows; expert weights are B[e] of shape [N, K] (K contiguous, the nn.Linear
layout); each expert computes D_e = A_e @ B[e]^T.  The forms differ only in
where each expert's token rows live and which rows are computed.

Inputs are already dequantised to float64 (see ``numerics``); numpy's float64
matmul is the only library primitive used.  Rows the form does not compute
come back as NaN with ``written == False``: the GPU must leave them untouched.
"""

import numpy as np

from .plan import plan, token_offsets


def expert_product(a_rows: np.ndarray, b_e: np.ndarray) -> np.ndarray:
    """D_e = A_e @ B_e^T for one expert: a_rows [t, K], b_e [N, K]."""
    return np.asarray(a_rows, np.float64) @ np.asarray(b_e, np.float64).T


def contiguous_segment(counts, align_q: int, e: int):
    """Row range of expert e in the M-grouped contiguous layout: segments are
    concatenated in expert order and each starts on a multiple of the token
    block align_q ("flops/deepgemm-grouped-masked-moe-gemm", "Arithmetic
    intensity")."""
    p = plan(counts, align_q)
    return p.offsets[e], p.offsets[e] + int(counts[e])


def contiguous(A: np.ndarray, B: np.ndarray, counts, align_q: int):
    """M-grouped contiguous form ("Workarounds": contiguous layout for
    prefill/training, where counts are known).

    A: float64 [rows_cap, K]; B: float64 [E, N, K].  For each expert with
    t_e > 0 and each row r < t_e: R[off_e + r] = A[off_e + r] @ B[e]^T.
    Padding rows between segments and rows past P are not computed
    ("Grouped execution does not require padded experts": zero-sized experts
    are skipped and tail rows are excluded).
    """
    rows_cap, K = A.shape
    E, N, K2 = B.shape
    assert K == K2 and len(counts) == E
    p = plan(counts, align_q)
    if p.P > rows_cap:
        raise ValueError("aligned segments do not fit in rows_cap")
    R = np.full((rows_cap, N), np.nan)
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        t = int(t)
        if t == 0:
            continue
        o = p.offsets[e]
        R[o:o + t] = expert_product(A[o:o + t], B[e])
        written[o:o + t] = True
    return R, written


def masked(A: np.ndarray, B: np.ndarray, valid_m):
    """Masked form ("Workarounds": masked grouped GEMM for decode under CUDA
    graphs; "Arithmetic intensity": fixed per-expert buffers, of which only
    the first valid_m[e] rows of expert e are computed).

    A: float64 [E, M_max, K]; B: float64 [E, N, K]; valid_m [E].
    R[e, r] = A[e, r] @ B[e]^T for r < valid_m[e]; other rows are untouched.
    """
    E, M_max, K = A.shape
    E2, N, K2 = B.shape
    assert E == E2 and K == K2 and len(valid_m) == E
    R = np.full((E, M_max, N), np.nan)
    written = np.zeros((E, M_max), dtype=bool)
    for e, v in enumerate(valid_m):
        v = int(v)
        if not 0 <= v <= M_max:
            raise ValueError("valid_m outside [0, M_max]")
        if v == 0:
            continue
        R[e, :v] = expert_product(A[e, :v], B[e])
        written[e, :v] = True
    return R, written


def kgrouped(dY: np.ndarray, X: np.ndarray, counts) -> np.ndarray:
    """K-grouped weight-gradient form ("Workarounds": K-grouped GEMM for MoE
    weight backward, M and N fixed and the contraction length varying).

    dY: float64 [T_cap, N]; X: float64 [T_cap, K]; tokens are packed by
    expert with no alignment.  dW[e] = sum over expert e's tokens t of
    dY[t]^T X[t] (an [N, K] outer-product sum); an expert with no tokens gets
    dW[e] = 0.  The result overwrites dW (no accumulation into prior values).
    """
    T_cap, N = dY.shape
    T2, K = X.shape
    assert T_cap == T2
    off = token_offsets(counts)
    if off[-1] > T_cap:
        raise ValueError("token counts exceed T_cap")
    dW = np.zeros((len(counts), N, K))
    for e in range(len(counts)):
        a, b = off[e], off[e + 1]
        if b > a:
            dW[e] = np.asarray(dY[a:b], np.float64).T @ np.asarray(X[a:b], np.float64)
    return dW
