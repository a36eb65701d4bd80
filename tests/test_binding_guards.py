"""The Python binding refuses tensors the library would misread or overrun
(the C ABI takes bare pointers and cannot see buffer sizes): host tensors,
strided views, wrong dtypes and buffers shorter than the call reaches.  Runs
on the CPU against a stand-in library that records the calls it receives."""
import pytest
import torch

from moe_grouped_gemm_side_gb300 import binding as mb

pytestmark = pytest.mark.cpu


class StandIn:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def f(*args):
            self.calls.append(name)
            return 0
        return f


@pytest.fixture
def fake(monkeypatch):
    lib = StandIn()
    monkeypatch.setattr(mb, "load", lambda path=None: lib)
    monkeypatch.setattr(mb, "_on_device", lambda t: True)   # host tensors stand in for device ones
    monkeypatch.setattr(mb, "_stream", lambda s: None)
    return lib


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_contiguous_accepts_exact_operands(fake):
    E, R, N, K = 4, 96, 256, 512
    mb.mgemm_contiguous(bf16(R, K), bf16(E, N, K), bf16(R, N), i32(E), 16, status=i32(1))
    mb.mgemm_contiguous(u8(R, K), u8(E, N, K), bf16(R, N), i32(E), 16, SFA=u8(K // 128, R),
                        SFB=u8(E, K // 128, N // 128))
    mb.mgemm_contiguous(u8(R, K), u8(E, N, K // 2), bf16(R, N), i32(E), 16, SFA=u8(K // 128, R),
                        SFB=u8(E, N, K // 32))                                  # E2M1 weights
    assert fake.calls == ["mgemm_contiguous"] * 3


@pytest.mark.parametrize("case", ["short_D", "D_dtype", "strided_A", "short_counts", "counts_dtype",
                                  "short_SFA", "short_SFB", "short_SFB_fp4", "status_dtype"])
def test_contiguous_refusals(fake, case):
    E, R, N, K = 4, 96, 256, 512
    a = dict(A=u8(R, K), B=u8(E, N, K), D=bf16(R, N), d_counts=i32(E), SFA=u8(K // 128, R),
             SFB=u8(E, K // 128, N // 128), status=None)
    if case == "short_D":
        a["D"] = bf16(R - 1, N)
    elif case == "D_dtype":
        a["D"] = torch.zeros((R, N), dtype=torch.float32)
    elif case == "strided_A":
        a["A"] = u8(K, R).t()
    elif case == "short_counts":
        a["d_counts"] = i32(E - 1)
    elif case == "counts_dtype":
        a["d_counts"] = torch.zeros(E, dtype=torch.int64)
    elif case == "short_SFA":
        a["SFA"] = u8(K // 128, R - 16)
    elif case == "short_SFB":
        a["SFB"] = u8(E - 1, K // 128, N // 128)
    elif case == "short_SFB_fp4":
        a["B"], a["SFB"] = u8(E, N, K // 2), u8(E, K // 128, N // 128)      # E4M3-sized scales
    elif case == "status_dtype":
        a["status"] = torch.zeros(1, dtype=torch.int64)
    with pytest.raises((ValueError, TypeError)):
        mb.mgemm_contiguous(a["A"], a["B"], a["D"], a["d_counts"], 16, SFA=a["SFA"], SFB=a["SFB"],
                            status=a["status"])
    assert fake.calls == []


def test_host_tensor_refused_without_stand_in(monkeypatch):
    monkeypatch.setattr(mb, "load", lambda path=None: StandIn())
    with pytest.raises(ValueError, match="CUDA tensor"):
        mb.mgemm_contiguous(bf16(32, 128), bf16(1, 128, 128), bf16(32, 128), i32(1), 16)


def test_masked_and_swiglu_sizes(fake):
    E, M, N, K = 3, 64, 512, 256
    A, B, v = u8(E, M, K), u8(E, N, K), i32(E)
    SFA, SFB = u8(E, K // 128, M), u8(E, K // 128, N // 128)
    mb.mgemm_masked(A, B, bf16(E, M, N), v, SFA=SFA, SFB=SFB)
    with pytest.raises(ValueError):
        mb.mgemm_masked(A, B, bf16(E, M - 1, N), v, SFA=SFA, SFB=SFB)
    with pytest.raises(ValueError):
        mb.mgemm_masked(A, B, bf16(E, M, N), v, SFA=u8(1, K // 128, M), SFB=SFB)
    # SwiGLU: Y holds N/2 columns; E4M3 output needs SFY [E, N/256, M]
    mb.mgemm_masked_swiglu(A, B, bf16(E, M, N // 2), v, SFA=SFA, SFB=SFB)
    mb.mgemm_masked_swiglu(A, B, u8(E, M, N // 2), v, SFA=SFA, SFB=SFB, SFY=u8(E, N // 256, M))
    with pytest.raises(ValueError):
        mb.mgemm_masked_swiglu(A, B, u8(E, M, N // 2), v, SFA=SFA, SFB=SFB, SFY=u8(E, N // 256, M - 1))
    with pytest.raises(ValueError):
        mb.mgemm_masked_swiglu(A, B, bf16(E, M, N // 2 - 1), v, SFA=SFA, SFB=SFB)
    R = 128
    mb.mgemm_contiguous_swiglu(u8(R, K), B, u8(R, N // 2), v, 16, SFA=u8(K // 128, R), SFB=SFB,
                               SFY=u8(N // 256, R))
    with pytest.raises(ValueError):
        mb.mgemm_contiguous_swiglu(u8(R, K), B, u8(R, N // 2), v, 16, SFA=u8(K // 128, R), SFB=SFB,
                                   SFY=u8(N // 256 - 1, R))
    assert fake.calls == ["mgemm_masked", "mgemm_masked_swiglu", "mgemm_masked_swiglu",
                          "mgemm_contiguous_swiglu"]


def test_kgrouped_sizes(fake):
    T, N, K, E = 100, 256, 128, 3
    dY, X = bf16(T, N), bf16(T, K)
    mb.kgemm_grouped(dY, X, torch.zeros((E, N, K)), i32(E))
    with pytest.raises(ValueError):
        mb.kgemm_grouped(dY, bf16(T - 1, K), torch.zeros((E, N, K)), i32(E))     # X shorter than dY
    with pytest.raises(ValueError):
        mb.kgemm_grouped(dY, X, torch.zeros((E, N - 128, K)), i32(E))           # dW not [E, N, K]
    with pytest.raises(TypeError):
        mb.kgemm_grouped(dY, X, torch.zeros((E, N, K), dtype=torch.float64), i32(E))
    assert fake.calls == ["kgemm_grouped"]


def test_selector_and_tactic_sizes(fake):
    table = mb.exemplar_table([{"lu": 0, "shares": [0] * 16, "tile_q": 32, "blocks": 1}] * 2)
    d_table = torch.from_numpy(table.view("u1").copy())
    mb.select_exemplar(i32(8), d_table, 2, i32(3), d_state=i32(1))
    with pytest.raises(ValueError):
        mb.select_exemplar(i32(8), d_table, 3, i32(3))                          # table holds 2 entries
    with pytest.raises(ValueError):
        mb.select_exemplar(i32(8), d_table, 2, i32(2))                          # tactic needs 3 words
    E, R, N, K = 2, 64, 256, 256
    mb.mgemm_contiguous_tactic(bf16(R, K), bf16(E, N, K), bf16(R, N), i32(E), 16, i32(3))
    with pytest.raises(ValueError):
        mb.mgemm_contiguous_tactic(bf16(R, K), bf16(E, N, K), bf16(R, N), i32(E), 16, i32(1))
    mb.mgemm_masked_tactic(bf16(E, R, K), bf16(E, N, K), bf16(E, R, N), i32(E), i32(2))
    assert fake.calls == ["moe_select_exemplar", "mgemm_contiguous_tactic", "mgemm_masked_tactic"]


def test_plan_and_wait_arguments(fake):
    mb.plan(i32(5), 8, 0)
    with pytest.raises(TypeError):
        mb.plan(torch.zeros(5, dtype=torch.int64), 8, 0)
    with pytest.raises(ValueError):
        mb.wait_selftest(None, 1000)
    with pytest.raises(TypeError):
        mb.select_tile(mb.MG_BF16, i32(4), 256, 256, status=torch.zeros(1))
