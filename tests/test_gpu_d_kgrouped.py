"""K-grouped weight-gradient form on the GPU against the oracle."""
import numpy as np
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb
from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import gemm as og
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

F32_SENTINEL = -12345.5


def run_kgrouped(counts, N, K, seed=1, integer=False, T_extra=29, dev="cuda"):
    E = len(counts)
    T = sum(max(0, c) for c in counts)
    T_cap = T + T_extra
    if integer:
        dY = wl.integer_bf16((T_cap, N), seed, dev)
        X = wl.integer_bf16((T_cap, K), seed + 1, dev)
    else:
        dY, X = wl.make_kgrouped(T_cap, N, K, seed, dev)
    # tokens past the last expert are poisoned
    if T_extra:
        dY.view(torch.int16)[T:] = wl.BF16_NAN_BITS
        X.view(torch.int16)[T:] = wl.BF16_NAN_BITS
    dW = torch.full((E, N, K), F32_SENTINEL, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.kgemm_grouped(dY, X, dW, torch.tensor(counts, dtype=torch.int32, device=dev), status=status)
    torch.cuda.synchronize()
    R = og.kgrouped(gu.deq_bf16(dY).reshape(T_cap, N), gu.deq_bf16(X).reshape(T_cap, K),
                    [max(0, c) for c in counts])
    return dW.cpu().numpy().astype(np.float64), R, int(status.item())


def check_dw(got, ref):
    """fp32 accumulation of bf16 products: per output row of each expert,
    max|err| <= 1e-2 * max|ref row|; exact zero rows stay zero."""
    for e in range(ref.shape[0]):
        m = np.abs(ref[e]).max(axis=1)
        err = np.abs(got[e] - ref[e]).max(axis=1)
        assert np.all(np.isfinite(err))
        zero = m == 0
        assert np.all(err[zero] == 0)
        assert np.all(err[~zero] <= 1e-2 * m[~zero]), f"expert {e}: worst {np.max(err[~zero] / m[~zero])}"


@pytest.mark.parametrize("N", [256, 384, 512])
def test_integer_exact(lib, cuda, N):
    """N=384 runs one 128-row block of dW per tile, 256 and 512 two."""
    counts = [5, 0, 64, 17, 100, 1]
    got, ref, status = run_kgrouped(counts, N, 256, integer=True)
    assert status == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("K", [128, 256, 384])
def test_random_tails(lib, cuda, K):
    counts = [3, 64, 65, 0, 127, 200, 16, 15]
    got, ref, status = run_kgrouped(counts, 256, K, seed=K)
    assert status == 0
    check_dw(got, ref)


def test_dirichlet_small(lib, cuda):
    counts = wl.counts_dirichlet(seed=11, E=16, total=4000)
    got, ref, status = run_kgrouped(counts, 384, 256, seed=4)
    assert status == 0
    check_dw(got, ref)


def test_empty_and_errors(lib, cuda):
    got, ref, status = run_kgrouped([0, 0], 128, 128)
    assert status == 0 and np.array_equal(got, np.zeros_like(got))
    # negative count: that expert is skipped and left untouched
    got, ref, status = run_kgrouped([4, -1, 6], 128, 128, seed=2)
    assert status == 6
    assert np.all(got[1] == F32_SENTINEL)
    check_dw(got[[0, 2]], ref[[0, 2]])
    # counts beyond T_cap: experts that fit are computed, the others untouched
    dev = cuda
    dY = wl.normal_bf16((40, 128), 3, dev)
    X = wl.normal_bf16((40, 128), 4, dev)
    dW = torch.full((2, 128, 128), F32_SENTINEL, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mb.kgemm_grouped(dY, X, dW, torch.tensor([30, 30], dtype=torch.int32, device=dev), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    r0 = gu.deq_bf16(dY).reshape(40, 128)[:30].T @ gu.deq_bf16(X).reshape(40, 128)[:30]
    check_dw(dW.cpu().numpy()[:1].astype(np.float64), r0[None])
    assert np.all(dW.cpu().numpy()[1] == F32_SENTINEL)


def test_max_experts(lib, cuda):
    """E = 1024 experts of a few tokens each (many empty): the descending-count
    order of 1024 experts and many partial token blocks."""
    rng = np.random.default_rng(3)
    counts = [int(c) for c in rng.integers(0, 9, size=1024)]
    got, ref, status = run_kgrouped(counts, 256, 128, integer=True, T_extra=5)
    assert status == 0
    assert np.array_equal(got, ref)


def test_long_experts_with_tails(lib, cuda):
    """Experts of 2^15+ tokens ending in a partial token block: hundreds of
    full stages go by before the one whose tail rows need zeroing, so the
    tail-zeroing warp must stay in step with the ring all the way.  Integer
    operands keep every fp32 sum exact (|sum| <= 4 * 40037 < 2^24)."""
    counts = [40037, 0, 3, 33005]
    got, ref, status = run_kgrouped(counts, 256, 256, integer=True, T_extra=7)
    assert status == 0
    assert np.array_equal(got, ref)
