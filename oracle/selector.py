"""Distribution-aware kernel choice by exemplar matching (oracle; test
infrastructure: only tests/, smoke() and bench.py's CPU legs use it).

"MoE GroupGEMM padding under expert skew", "Adapt kernels without adding a
CPU stall": the selector sorts and normalises the per-expert count vector,
matches it against exemplars tuned offline on the target GPU, and needs
guardrails so that neighbouring histograms do not switch kernels on every
layer.  The pages give the steps, not the formulas; the choices below are
this implementation's, kept in integers so that the GPU reproduces every
decision exactly:

* features of a histogram c[0..E) (negative counts read as 0), U = sum c:
  - sort c descending;
  - for k = 1..16, m_k = ceil(k E / 16) and share_k =
    floor(65536 * (sum of the m_k largest counts) / U)  (all 0 when U = 0):
    the cumulative top-share curve, comparable across expert counts;
  - lu = 16 e + floor(16 (U - 2^e) / 2^e) with e = floor(log2 U) (lu = 0 for
    U = 0): log2 U in 1/16 steps, linear between powers of two.
* distance to an exemplar x: sum_k |share_k - x.share_k| + 2048 |lu - x.lu|
  (a factor of two in U costs half of a whole share unit);
* choice: the exemplar with the smallest distance, the lowest index on ties;
* hysteresis (a per-call-site state holding the previous choice): keep the
  previous exemplar while its distance exceeds the best one by at most the
  margin; the state then holds the exemplar used.
"""

import numpy as np

NUM_SHARES = 16
SHARE_ONE = 65536
LU_WEIGHT = 2048


def features(counts):
    """(lu, shares[16]) as Python ints."""
    c = sorted((max(0, int(x)) for x in counts), reverse=True)
    E = len(c)
    U = sum(c)
    if U == 0:
        return 0, [0] * NUM_SHARES
    prefix = [0]
    for v in c:
        prefix.append(prefix[-1] + v)
    shares = []
    for k in range(1, NUM_SHARES + 1):
        m = -(-k * E // NUM_SHARES)
        shares.append(SHARE_ONE * prefix[m] // U)
    e = U.bit_length() - 1
    lu = 16 * e + (16 * (U - (1 << e))) // (1 << e)
    return lu, shares


def distance(feat, exemplar):
    lu, shares = feat
    return sum(abs(a - b) for a, b in zip(shares, exemplar["shares"])) + LU_WEIGHT * abs(lu - exemplar["lu"])


def choose(counts, table, prev=-1, margin=0):
    """Index of the exemplar used for `counts` (prev = -1: no history)."""
    feat = features(counts)
    d = [distance(feat, x) for x in table]
    best = int(np.argmin(d))           # numpy argmin returns the first minimum
    if 0 <= prev < len(table) and d[prev] - d[best] <= margin:
        return prev
    return best
