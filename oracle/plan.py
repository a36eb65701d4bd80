"""Token-tile padding accounting (oracle; test infrastructure only).

Pure Python integers throughout, so nothing overflows; the two ratios are
computed as IEEE doubles in one stated order so that a GPU implementation can
be held to them bit for bit.
"""

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class Plan:
    q: int
    offsets: List[int]                    # E+1 entries, offsets[E] == P
    tiles: List[Tuple[int, int, int]]     # (expert, first row, rows)
    P: int
    U: int
    sumsq: int
    active: int
    num_tiles: int
    pad_frac: float
    eff_experts: float
    rounded: List[int] = field(default_factory=list)   # q*ceil(t_i/q) per expert


def padded_rows(counts: Sequence[int], q: int) -> int:
    """P: each expert's count rounded up to a multiple of the token tile q,
    summed; an expert with no tokens adds nothing.

    "MoE GroupGEMM padding under expert skew", "Calculate padded token
    columns": the executed token columns of expert i are q*ceil(t_i/q), and P
    is their sum over experts.
    """
    return sum(q * ceil_div(int(t), q) for t in counts)


def padding_fraction(P: int, U: int) -> float:
    """(P-U)/P ("Calculate padded token columns"); 0.0 for an empty layer,
    which the page leaves undefined."""
    if P == 0:
        return 0.0
    return float(P - U) / float(P)


def effective_experts(counts: Sequence[int]) -> float:
    """U^2 / sum_i t_i^2 ("MoE GroupGEMM padding under expert skew",
    "Summarize skew without losing the histogram"); 0.0 when no expert has
    tokens, which the page leaves undefined.  Evaluated as
    (double(U) * double(U)) / double(sum t_i^2)."""
    U = sum(int(t) for t in counts)
    sumsq = sum(int(t) * int(t) for t in counts)
    if sumsq == 0:
        return 0.0
    return (float(U) * float(U)) / float(sumsq)


def m_occupancy(M: int, B_M: int) -> float:
    """Single-GEMM M-occupancy of "Query on performance-modeling of MoE
    Grouped GEMM", "Background": tiles needed to fit M (M / B_M as a real
    number) over the tiles actually used (ceil(M / B_M))."""
    used = ceil_div(M, B_M)
    return (M / float(B_M)) / used


def avg_assignments_per_expert(concurrency: int, top_k: int, num_experts: int) -> float:
    """Expected matrix height: global concurrency times top-k over the expert
    count ("MoE GroupGEMM padding under expert skew", "Summarize skew without
    losing the histogram", last paragraph)."""
    return concurrency * top_k / float(num_experts)


def plan(counts: Sequence[int], q: int) -> Plan:
    """Full accounting for one histogram and one token tile q.

    offsets: exclusive prefix sum of q*ceil(t_e/q); expert e's rows are
    [offsets[e], offsets[e] + t_e), so every segment starts on a multiple of
    q -- the M-block alignment of the contiguous layout
    ("flops/deepgemm-grouped-masked-moe-gemm", "Arithmetic intensity").

    tiles: for e ascending and j ascending over 0..ceil(t_e/q)-1, the triple
    (e, offsets[e] + j*q, min(q, t_e - j*q)).  Experts without tokens get no
    tiles ("Grouped execution does not require padded experts": zero-sized
    experts are skipped).  The pages fix no tile-list format; this one is the
    plainest that names every executed tile once.
    """
    if q <= 0:
        raise ValueError("token tile q must be positive")
    counts = [int(t) for t in counts]
    if any(t < 0 for t in counts):
        raise ValueError("token counts must be non-negative")
    offsets = [0]
    rounded = []
    tiles = []
    for e, t in enumerate(counts):
        r = q * ceil_div(t, q)
        rounded.append(r)
        for j in range(ceil_div(t, q)):
            tiles.append((e, offsets[-1] + j * q, min(q, t - j * q)))
        offsets.append(offsets[-1] + r)
    P = offsets[-1]
    U = sum(counts)
    sumsq = sum(t * t for t in counts)
    return Plan(
        q=q,
        offsets=offsets,
        tiles=tiles,
        P=P,
        U=U,
        sumsq=sumsq,
        active=sum(1 for t in counts if t > 0),
        num_tiles=len(tiles),
        pad_frac=padding_fraction(P, U),
        eff_experts=effective_experts(counts),
        rounded=rounded,
    )


def token_offsets(counts: Sequence[int]) -> List[int]:
    """Exclusive prefix sum of the raw counts: the packed (unaligned) token
    layout of the K-grouped weight-gradient form."""
    out = [0]
    for t in counts:
        out.append(out[-1] + int(t))
    return out
