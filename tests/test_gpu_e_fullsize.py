"""Full-size workloads, in the launch configuration bench.py times (device
tile selection, the same seeded generators), checked against the oracle:
every valid row where the oracle finishes in seconds, sampled experts or
blocks where it would not, and sentinel bits everywhere else."""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import gemm as og
from oracle import numerics as on
from oracle import plan as op
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _contiguous_full(name, dev, gemm_index=0):
    spec = wl.WORKLOADS[name]
    counts = spec["counts"]()
    E, align = spec["E"], spec["align_q"]
    p = op.plan(counts, align)
    rows_cap = (p.P + 15) // 16 * 16
    N, K = (spec["N"], spec["K"]) if gemm_index == 0 else (spec["second"]["N"], spec["second"]["K"])
    seed = spec["seed"] + 100 * gemm_index
    ops = wl.make_contiguous(E, rows_cap, N, K, spec["dtype"], seed, dev,
                             spec["a_std"] if gemm_index == 0 else 1.0,
                             spec["b_std"] if gemm_index == 0 else 1.0)
    written = np.zeros(rows_cap, dtype=bool)
    for e, t in enumerate(counts):
        written[p.offsets[e]:p.offsets[e] + t] = True
    gu.poison_rows_(ops.A, written, spec["dtype"] == "fp8", ops.SFA)
    D = gu.sentinel_like((rows_cap, N), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.mgemm_contiguous(ops.A, ops.B, D, torch.tensor(counts, dtype=torch.int32, device=dev), align,
                        SFA=ops.SFA, SFB=ops.SFB, tile_q=0, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Dbits = gu.bf16_bits(D)
    assert (Dbits[~written] == gu.SENTINEL_BITS).all()
    return counts, p, ops, Dbits


def test_issue32_bf16_all_rows(lib, cuda):
    """The issue's 32-expert histogram, N=4096, K=2048, bf16: every valid row."""
    counts, p, ops, Dbits = _contiguous_full("contig_bf16_e32_n4096_k2048", cuda)
    A = gu.deq_bf16(ops.A).reshape(ops.A.shape)
    for e, t in enumerate(counts):
        if t == 0:
            continue
        o = p.offsets[e]
        Be = gu.deq_bf16(ops.B[e]).reshape(ops.B.shape[1:])
        gu.check_rows_bf16(Dbits[o:o + t], og.expert_product(A[o:o + t], Be))


@pytest.mark.parametrize("gemm_index", [0, 1])
def test_prefill_fp8_sampled_experts(lib, cuda, gemm_index):
    """Skewed FP8 prefill (64 experts, 32768 assignments): the largest,
    the smallest and four more experts, all their rows and columns."""
    counts, p, ops, Dbits = _contiguous_full("prefill_fp8_e64_t32768_n4096_k7168", cuda, gemm_index)
    order = np.argsort(counts)
    sample = sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2]), 5, 17, 40})
    for e in sample:
        t = counts[e]
        o = p.offsets[e]
        a = on.dequant_rows(ops.A[o:o + t].cpu().numpy(), ops.SFA[:, o:o + t].cpu().numpy())
        b = on.dequant_weight(ops.B[e].cpu().numpy(), ops.SFB[e].cpu().numpy())
        gu.check_frobenius(Dbits[o:o + t], og.expert_product(a, b))


def test_prefill_fp8_gemm2_every_expert_all_rows(lib, cuda):
    """Skewed FP8 prefill, GEMM2 (N=7168, K=2048): every expert, all of its
    rows and columns, per-expert Frobenius rule (the oracle's ~1 TFLOP of
    fp64 work takes seconds here)."""
    counts, p, ops, Dbits = _contiguous_full("prefill_fp8_e64_t32768_n4096_k7168", cuda, 1)
    A = ops.A.cpu().numpy()
    SFA = ops.SFA.cpu().numpy()
    checked = 0
    for e, t in enumerate(counts):
        if t == 0:
            continue
        o = p.offsets[e]
        a = on.dequant_rows(A[o:o + t], SFA[:, o:o + t])
        b = on.dequant_weight(ops.B[e].cpu().numpy(), ops.SFB[e].cpu().numpy())
        gu.check_frobenius(Dbits[o:o + t], og.expert_product(a, b))
        checked += t
    assert checked == sum(counts)


def _row_sample(t, q, rng, extra=8):
    """Rows of an expert to check: its first rows, the rows of its last
    token tile (capped at 48) and the rows on either side of every other
    tile boundary, and a few random rows.  The kernel splits an expert's
    ceil(t / q) token tiles evenly (widths rounded up to 16, the last tile
    trimmed)."""
    n = -(-t // q)
    w = -(-(-(-t // n)) // 16) * 16
    last0 = (n - 1) * w
    rows = set(range(min(t, 8))) | set(range(last0, min(t, last0 + 48)))
    for j in range(1, n):
        rows |= {j * w - 1, j * w}
    rows |= set(int(r) for r in rng.integers(0, t, size=min(extra, t)))
    return np.array(sorted(rows))


@pytest.mark.parametrize("gemm_index", [0, 1])
def test_prefill_fp8_every_expert_row_sample(lib, cuda, gemm_index):
    """Skewed FP8 prefill, both GEMMs: every expert, on a row sample that
    holds the rows of its last token tile at the tile the device chose (the
    one the kernel trims), the rows around its tile boundaries, the first
    rows and random rows; the per-expert
    Frobenius rule applies to the sampled rows, all columns."""
    name = "prefill_fp8_e64_t32768_n4096_k7168"
    counts, p, ops, Dbits = _contiguous_full(name, cuda, gemm_index)
    N, K = ops.B.shape[1], ops.B.shape[2]
    q = mb.select_tile_host(mb.MG_FP8_E4M3_UE8M0, counts, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    rng = np.random.default_rng(11 + gemm_index)
    partial = 0
    for e, t in enumerate(counts):
        if t == 0:
            continue
        partial += t % q != 0
        o = p.offsets[e]
        rows = _row_sample(t, q, rng)
        idx = torch.from_numpy(o + rows).to(ops.A.device)
        a = on.dequant_rows(ops.A[idx].cpu().numpy(), ops.SFA[:, idx].cpu().numpy())
        b = on.dequant_weight(ops.B[e].cpu().numpy(), ops.SFB[e].cpu().numpy())
        gu.check_frobenius(Dbits[o + rows], og.expert_product(a, b))
    assert partial > 0


def test_prefill_bf16_sampled_experts(lib, cuda):
    counts, p, ops, Dbits = _contiguous_full("prefill_bf16_e64_t32768_n4096_k7168", cuda)
    order = np.argsort(counts)
    A = ops.A
    for e in sorted({int(order[-1]), int(order[0]), 9}):
        t = counts[e]
        o = p.offsets[e]
        a = gu.deq_bf16(A[o:o + t]).reshape(t, A.shape[1])
        b = gu.deq_bf16(ops.B[e]).reshape(ops.B.shape[1:])
        gu.check_rows_bf16(Dbits[o:o + t], og.expert_product(a, b))


def test_masked_decode_fp8_all_experts(lib, cuda):
    """Masked FP8 decode: 16 experts x 256-row buffers, Zipf(1.1) valid_m."""
    spec = wl.WORKLOADS["masked_fp8_e16_m256_n4096_k7168"]
    v = spec["counts"]()
    E, M, N, K = spec["E"], spec["M_max"], spec["N"], spec["K"]
    ops = wl.make_masked(E, M, N, K, "fp8", spec["seed"], cuda)
    valid = np.zeros((E, M), dtype=bool)
    for e, x in enumerate(v):
        valid[e, :x] = True
    gu.poison_rows_(ops.A.view(E * M, K), valid.reshape(-1), True)
    D = gu.sentinel_like((E, M, N), cuda)
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.mgemm_masked(ops.A, ops.B, D, torch.tensor(v, dtype=torch.int32, device=cuda),
                    SFA=ops.SFA, SFB=ops.SFB, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Dbits = gu.bf16_bits(D).reshape(E, M, N)
    assert (Dbits[~valid] == gu.SENTINEL_BITS).all()
    for e, x in enumerate(v):
        if x == 0:
            continue
        a = on.dequant_rows(ops.A[e, :x].cpu().numpy(), ops.SFA[e][:, :x].cpu().numpy())
        b = on.dequant_weight(ops.B[e].cpu().numpy(), ops.SFB[e].cpu().numpy())
        gu.check_frobenius(Dbits[e, :x], og.expert_product(a, b))


def test_kgrouped_weight_grad_sampled_blocks(lib, cuda):
    """K-grouped bf16 weight gradient, 32 experts, 65536 Dirichlet(0.3)
    tokens: two 128 x 256 blocks per expert plus every row of the smallest
    non-empty expert; empty experts must be exactly zero."""
    spec = wl.WORKLOADS["kgrouped_bf16_e32_t65536_n4096_k2048"]
    counts = spec["counts"]()
    E, N, K, T = spec["E"], spec["N"], spec["K"], spec["T"]
    dY, X = wl.make_kgrouped(T, N, K, spec["seed"], cuda)
    dW = torch.full((E, N, K), -1.0, dtype=torch.float32, device=cuda)
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    mb.kgemm_grouped(dY, X, dW, torch.tensor(counts, dtype=torch.int32, device=cuda), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    off = op.token_offsets(counts)
    rng = np.random.default_rng(5)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            assert torch.count_nonzero(dW[e]).item() == 0
            continue
        dy = gu.deq_bf16(dY[a:b]).reshape(b - a, N)
        x = gu.deq_bf16(X[a:b]).reshape(b - a, K)
        for _ in range(2):
            n0 = int(rng.integers(0, N // 128)) * 128
            k0 = int(rng.integers(0, K // 256)) * 256
            ref = og.kgrouped(dy[:, n0:n0 + 128], x[:, k0:k0 + 256], [b - a])[0]
            got = dW[e, n0:n0 + 128, k0:k0 + 256].cpu().numpy().astype(np.float64)
            m = np.abs(ref).max(axis=1)
            assert np.all(np.abs(got - ref).max(axis=1) <= 1e-2 * m)
    small = min((c, e) for e, c in enumerate(counts) if c > 0)[1]
    a, b = off[small], off[small + 1]
    ref = og.kgrouped(gu.deq_bf16(dY[a:b]).reshape(b - a, N), gu.deq_bf16(X[a:b]).reshape(b - a, K), [b - a])[0]
    got = dW[small].cpu().numpy().astype(np.float64)
    m = np.abs(ref).max(axis=1)
    assert np.all(np.abs(got - ref).max(axis=1) <= 1e-2 * m)
