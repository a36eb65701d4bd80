"""Thin ctypes binding of libmoegemm.so (C ABI in include/moegemm.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Torch tensors supply device memory and the current stream; nothing
here computes the method, and every call raises if the library is missing or
returns an error.  Because the C ABI receives bare pointers, each device call
first checks its tensors (on the GPU, contiguous, expected dtype, at least as
many bytes as the call reaches) and raises ValueError / TypeError before any
launch.
"""
import ctypes
import os

import numpy as np

from . import build as _build

MG_OK = 0
STATUS_NAMES = {
    0: "MG_OK", 1: "MG_ERR_INVALID_ARG", 2: "MG_ERR_UNSUPPORTED", 3: "MG_ERR_CUDA",
    4: "MG_ERR_CAPACITY", 5: "MG_ERR_TIMEOUT", 6: "MG_ERR_DEVICE_ARG",
}
MG_BF16, MG_FP8_E4M3_UE8M0, MG_FP8_X_FP4_E2M1 = 0, 1, 2
MG_SWIGLU_BF16, MG_SWIGLU_FP8_E4M3_UE8M0 = 1, 2

# Every function the header declares, with its ctypes signature.
_c_i32p = ctypes.POINTER(ctypes.c_int32)
_c_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class PlanStats(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int64), ("U", ctypes.c_int64), ("sumsq", ctypes.c_int64),
                ("active", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("pad_frac", ctypes.c_double), ("eff_experts", ctypes.c_double)]


SIGNATURES = {
    "mg_status_str": (ctypes.c_char_p, [_i32]),
    "moe_plan_host": (_i32, [_c_i32p, _i32, _i32, _c_i64p, _c_i32p, _i32, ctypes.POINTER(PlanStats)]),
    "moe_plan": (_i32, [_vp, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp]),
    "moe_select_tile": (_i32, [_i32, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_select_tile_host": (_i32, [_i32, _c_i32p, _i32, _i32, _i32, _i32, _c_i32p]),
    "mgemm_contiguous": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _vp, _vp]),
    "mgemm_masked": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "mgemm_contiguous_swiglu": (_i32, [_i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                       _i32, _i32, _vp, _vp]),
    "mgemm_masked_swiglu": (_i32, [_i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp,
                                   _vp]),
    "moe_exemplar_features_host": (_i32, [_c_i32p, _i32, _c_i32p, _c_i32p]),
    "moe_select_exemplar_host": (_i32, [_c_i32p, _i32, _vp, _i32, _i32, _i32, _c_i32p]),
    "moe_select_exemplar": (_i32, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp]),
    "mgemm_contiguous_tactic": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _vp,
                                       _vp, _vp]),
    "mgemm_masked_tactic": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "mgemm_masked_exemplar": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp,
                                     _vp, _vp]),
    "kgemm_grouped": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _vp, _vp]),
    "mg_set_wait_limit_ns": (_i32, [_i64]),
    "mg_get_wait_limit_ns": (_i64, []),
    "mg_wait_selftest": (_i32, [_vp, _i64, _vp]),
    "mg_set_kernel_policy": (_i32, [_i32]),
    "mg_get_kernel_policy": (_i32, []),
}

# Kernel families of the contiguous and masked forms (mg_set_kernel_policy).
POLICY_AUTO, POLICY_SINGLE, POLICY_DUAL, POLICY_PAIR, POLICY_PAIR_DUAL, POLICY_TOKM = 0, 1, 2, 3, 4, 5
POLICIES = {"auto": POLICY_AUTO, "single": POLICY_SINGLE, "dual": POLICY_DUAL,
            "pair": POLICY_PAIR, "pair_dual": POLICY_PAIR_DUAL, "tokm": POLICY_TOKM}

_LIB = None


class MoeGemmError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


def load(path: str = None) -> ctypes.CDLL:
    """Loads the library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _check(fn, code):
    if code != MG_OK:
        raise MoeGemmError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on_device(t) -> bool:
    return t.is_cuda


def _need(t, name: str, nbytes: int, dtypes=None):
    """Checks a tensor the library reaches through a bare pointer: on the GPU,
    dense row-major, of an accepted dtype and at least `nbytes` long (the C
    ABI cannot see buffer sizes, so a short buffer would be overrun)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if not _on_device(t):
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes; the call reaches {nbytes}")


def _opt(t, name: str, nbytes: int, dtypes=None):
    if t is not None:
        _need(t, name, nbytes, dtypes)


def _int32():
    import torch
    return (torch.int32,)


def _check_fwd(dt, A, B, D, d_counts, SFA, SFB, status, rows_total, rows_sf, sf_groups, N, K, E):
    """Operands of the contiguous and masked forms: D bf16 [rows_total, N];
    SFA [sf_groups, K/128, rows_sf]; SFB [E, K/128, N/128] (E4M3 weights) or
    [E, N, K/32] (E2M1 weights); counts int32 [E]."""
    import torch
    _need(A, "A", A.numel() * A.element_size())
    _need(B, "B", B.numel() * B.element_size())
    _need(D, "D", rows_total * N * 2, (torch.bfloat16,))
    _need(d_counts, "counts", E * 4, _int32())
    _opt(SFA, "SFA", sf_groups * (K // 128) * rows_sf)
    _opt(SFB, "SFB", E * N * (K // 32) if dt == MG_FP8_X_FP4_E2M1 else E * (K // 128) * (N // 128))
    _opt(status, "status", 4, _int32())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_of(A):
    import torch
    if A.dtype == torch.bfloat16:
        return MG_BF16
    if A.dtype in (torch.uint8, torch.float8_e4m3fn):
        return MG_FP8_E4M3_UE8M0
    raise TypeError(f"unsupported operand dtype {A.dtype}")


def _fwd_dtype(A, B, K):
    """E4M3 activations with packed E2M1 weights ([E, N, K/2]) are FP8 x FP4."""
    dt = _dtype_of(A)
    if dt == MG_FP8_E4M3_UE8M0 and 2 * B.shape[-1] == K:
        return MG_FP8_X_FP4_E2M1
    return dt


def status_str(code: int) -> str:
    return load().mg_status_str(code).decode()


# ------------------------------------------------------------------ host plan
def plan_host(counts, q: int, max_tiles: int = None):
    """moe_plan_host: returns (offsets int64 [E+1], tiles int32 [T,3], PlanStats, status).

    With max_tiles None the tile list is sized by the library: a first call
    without a list reports the tile count in its stats."""
    lib = load()
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    E = len(c)
    offsets = np.zeros(E + 1, dtype=np.int64)
    st = PlanStats()
    if max_tiles is None:
        code = lib.moe_plan_host(c.ctypes.data_as(_c_i32p), E, q, offsets.ctypes.data_as(_c_i64p),
                                 None, 0, ctypes.byref(st))
        if code != MG_OK:
            return offsets, np.zeros((0, 3), dtype=np.int32), st, code
        if st.num_tiles == 2 ** 31 - 1:
            # saturated count: rows of such a list would pass 2^31 - 1, which
            # an int32 tile list refuses anyway
            return offsets, np.zeros((0, 3), dtype=np.int32), st, 2
        max_tiles = st.num_tiles
    tiles = np.zeros((max(max_tiles, 1), 3), dtype=np.int32)
    code = lib.moe_plan_host(c.ctypes.data_as(_c_i32p), E, q, offsets.ctypes.data_as(_c_i64p),
                             tiles.ctypes.data_as(_c_i32p) if max_tiles > 0 else None,
                             max_tiles, ctypes.byref(st))
    return offsets, tiles[:max_tiles], st, code


def select_tile_host(dtype: int, counts, N: int, K: int, num_sms: int = 0) -> int:
    lib = load()
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    out = ctypes.c_int32(0)
    _check("moe_select_tile_host",
           lib.moe_select_tile_host(dtype, c.ctypes.data_as(_c_i32p), len(c), N, K, num_sms, ctypes.byref(out)))
    return out.value


# ---------------------------------------------------------------- device calls
STATS_DTYPE = np.dtype([("P", "<i8"), ("U", "<i8"), ("sumsq", "<i8"), ("active", "<i4"),
                        ("num_tiles", "<i4"), ("pad_frac", "<f8"), ("eff_experts", "<f8")])


def decode_stats(buf) -> dict:
    """48-byte mg_plan_stats (a uint8 tensor) -> dict."""
    a = np.frombuffer(buf.cpu().numpy().tobytes(), dtype=STATS_DTYPE)[0]
    return {k: a[k].item() for k in STATS_DTYPE.names}


def plan(d_counts, q: int, max_tiles: int, status=None, stream=None):
    """moe_plan on device tensors; returns (offsets, tiles, stats_bytes)."""
    import torch
    lib = load()
    _need(d_counts, "counts", 0, _int32())
    _opt(status, "status", 4, _int32())
    dev = d_counts.device
    E = d_counts.numel()
    offsets = torch.empty(E + 1, dtype=torch.int64, device=dev)
    tiles = torch.empty((max(max_tiles, 1), 3), dtype=torch.int32, device=dev)
    stats = torch.zeros(48, dtype=torch.uint8, device=dev)
    _check("moe_plan", lib.moe_plan(_ptr(d_counts), E, q, _ptr(offsets),
                                    _ptr(tiles) if max_tiles > 0 else None, max_tiles,
                                    _ptr(stats), _ptr(status), _stream(stream)))
    return offsets, tiles[:max_tiles], stats


def select_tile(dtype: int, d_counts, N: int, K: int, status=None, stream=None):
    import torch
    lib = load()
    _need(d_counts, "counts", 0, _int32())
    _opt(status, "status", 4, _int32())
    out = torch.zeros(1, dtype=torch.int32, device=d_counts.device)
    _check("moe_select_tile", lib.moe_select_tile(dtype, _ptr(d_counts), d_counts.numel(), N, K,
                                                  _ptr(out), _ptr(status), _stream(stream)))
    return out


def mgemm_contiguous(A, B, D, d_counts, align_q: int, SFA=None, SFB=None, tile_q: int = 0,
                     status=None, stream=None):
    lib = load()
    rows_cap, K = A.shape
    E, N, _ = B.shape
    dt = _fwd_dtype(A, B, K)
    _check_fwd(dt, A, B, D, d_counts, SFA, SFB, status, rows_cap, rows_cap, 1, N, K, E)
    _check("mgemm_contiguous", lib.mgemm_contiguous(
        dt, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(d_counts), E,
        rows_cap, N, K, align_q, tile_q, _ptr(status), _stream(stream)))


def mgemm_masked(A, B, D, d_valid_m, SFA=None, SFB=None, status=None, stream=None):
    lib = load()
    E, M_max, K = A.shape
    N = B.shape[1]
    dt = _fwd_dtype(A, B, K)
    _check_fwd(dt, A, B, D, d_valid_m, SFA, SFB, status, E * M_max, M_max, E, N, K, E)
    _check("mgemm_masked", lib.mgemm_masked(
        dt, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(d_valid_m), E,
        M_max, N, K, _ptr(status), _stream(stream)))


def _swiglu_out(Y):
    import torch
    if Y.dtype == torch.bfloat16:
        return MG_SWIGLU_BF16
    if Y.dtype in (torch.uint8, torch.float8_e4m3fn):
        return MG_SWIGLU_FP8_E4M3_UE8M0
    raise TypeError(f"unsupported SwiGLU output dtype {Y.dtype}")


def _check_swiglu(dt, out, A, B, Y, SFY, d_counts, SFA, SFB, status, rows_total, rows_sf, sf_groups, N, K, E):
    """As _check_fwd, with Y [rows_total, N/2] in place of D and, for E4M3
    output, SFY [sf_groups, N/256, rows_sf]."""
    _need(A, "A", A.numel() * A.element_size())
    _need(B, "B", B.numel() * B.element_size())
    _need(Y, "Y", rows_total * (N // 2) * Y.element_size())
    _need(d_counts, "counts", E * 4, _int32())
    _opt(SFA, "SFA", sf_groups * (K // 128) * rows_sf)
    _opt(SFB, "SFB", E * N * (K // 32) if dt == MG_FP8_X_FP4_E2M1 else E * (K // 128) * (N // 128))
    if out == MG_SWIGLU_FP8_E4M3_UE8M0:
        _opt(SFY, "SFY", sf_groups * (N // 256) * rows_sf)
    _opt(status, "status", 4, _int32())


def mgemm_contiguous_swiglu(A, B, Y, d_counts, align_q: int, SFA=None, SFB=None, SFY=None,
                            tile_q: int = 0, status=None, stream=None):
    """GEMM1 with SwiGLU fused into its epilogue; Y bf16 [rows_cap, N/2], or
    E4M3 bytes with UE8M0 scales SFY [N/256, rows_cap]."""
    lib = load()
    rows_cap, K = A.shape
    E, N, _ = B.shape
    dt, out = _fwd_dtype(A, B, K), _swiglu_out(Y)
    _check_swiglu(dt, out, A, B, Y, SFY, d_counts, SFA, SFB, status, rows_cap, rows_cap, 1, N, K, E)
    _check("mgemm_contiguous_swiglu", lib.mgemm_contiguous_swiglu(
        dt, out, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(Y), _ptr(SFY),
        _ptr(d_counts), E, rows_cap, N, K, align_q, tile_q, _ptr(status), _stream(stream)))


def mgemm_masked_swiglu(A, B, Y, d_valid_m, SFA=None, SFB=None, SFY=None, status=None, stream=None):
    """Masked GEMM1 with SwiGLU fused; Y [E, M_max, N/2], SFY [E, N/256, M_max]."""
    lib = load()
    E, M_max, K = A.shape
    N = B.shape[1]
    dt, out = _fwd_dtype(A, B, K), _swiglu_out(Y)
    _check_swiglu(dt, out, A, B, Y, SFY, d_valid_m, SFA, SFB, status, E * M_max, M_max, E, N, K, E)
    _check("mgemm_masked_swiglu", lib.mgemm_masked_swiglu(
        dt, out, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(Y), _ptr(SFY),
        _ptr(d_valid_m), E, M_max, N, K, _ptr(status), _stream(stream)))


# ------------------------------------------------------------ exemplar selector
EXEMPLAR_DTYPE = np.dtype([("lu", "<i4"), ("share", "<i4", (16,)), ("tile_q", "<i4"), ("blocks", "<i4"),
                           ("reserved", "<i4")])
assert EXEMPLAR_DTYPE.itemsize == 80


def exemplar_table(entries) -> np.ndarray:
    """List of {"lu", "shares", "tile_q", "blocks"} -> mg_exemplar array."""
    t = np.zeros(len(entries), dtype=EXEMPLAR_DTYPE)
    for i, x in enumerate(entries):
        t[i]["lu"] = x["lu"]
        t[i]["share"] = x["shares"]
        t[i]["tile_q"] = x["tile_q"]
        t[i]["blocks"] = x["blocks"]
    return t


def exemplar_table_device(table: np.ndarray, device="cuda"):
    """mg_exemplar array -> uint8 device tensor holding the same bytes."""
    import torch
    return torch.from_numpy(np.frombuffer(table.tobytes(), dtype=np.uint8).copy()).to(device)


def exemplar_features_host(counts):
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    lu = ctypes.c_int32(0)
    share = np.zeros(16, dtype=np.int32)
    _check("moe_exemplar_features_host", load().moe_exemplar_features_host(
        c.ctypes.data_as(_c_i32p), len(c), ctypes.byref(lu), share.ctypes.data_as(_c_i32p)))
    return lu.value, share.tolist()


def select_exemplar_host(counts, table: np.ndarray, margin: int = 0, prev: int = -1) -> int:
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    t = np.ascontiguousarray(table)
    out = ctypes.c_int32(0)
    _check("moe_select_exemplar_host", load().moe_select_exemplar_host(
        c.ctypes.data_as(_c_i32p), len(c), t.ctypes.data, len(t), margin, prev, ctypes.byref(out)))
    return out.value


def select_exemplar(d_counts, d_table, n: int, d_tactic, margin: int = 0, d_state=None, status=None,
                    stream=None):
    """moe_select_exemplar: writes {tile_q, blocks, index} to d_tactic (int32 [3])."""
    _need(d_counts, "counts", 0, _int32())
    _need(d_table, "table", n * EXEMPLAR_DTYPE.itemsize)
    _need(d_tactic, "tactic", 12, _int32())
    _opt(d_state, "state", 4, _int32())
    _opt(status, "status", 4, _int32())
    _check("moe_select_exemplar", load().moe_select_exemplar(
        _ptr(d_counts), d_counts.numel(), _ptr(d_table), n, margin, _ptr(d_state), _ptr(d_tactic),
        _ptr(status), _stream(stream)))


def mgemm_contiguous_tactic(A, B, D, d_counts, align_q: int, d_tactic, SFA=None, SFB=None, status=None,
                            stream=None):
    lib = load()
    rows_cap, K = A.shape
    E, N, _ = B.shape
    dt = _fwd_dtype(A, B, K)
    _check_fwd(dt, A, B, D, d_counts, SFA, SFB, status, rows_cap, rows_cap, 1, N, K, E)
    _need(d_tactic, "tactic", 8, _int32())
    _check("mgemm_contiguous_tactic", lib.mgemm_contiguous_tactic(
        dt, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(d_counts), E,
        rows_cap, N, K, align_q, _ptr(d_tactic), _ptr(status), _stream(stream)))


def mgemm_masked_tactic(A, B, D, d_valid_m, d_tactic, SFA=None, SFB=None, status=None, stream=None):
    lib = load()
    E, M_max, K = A.shape
    N = B.shape[1]
    dt = _fwd_dtype(A, B, K)
    _check_fwd(dt, A, B, D, d_valid_m, SFA, SFB, status, E * M_max, M_max, E, N, K, E)
    _need(d_tactic, "tactic", 8, _int32())
    _check("mgemm_masked_tactic", lib.mgemm_masked_tactic(
        dt, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(d_valid_m), E,
        M_max, N, K, _ptr(d_tactic), _ptr(status), _stream(stream)))


def mgemm_masked_exemplar(A, B, D, d_valid_m, d_table, n: int, SFA=None, SFB=None, tactic_out=None,
                          status=None, stream=None):
    """mgemm_masked with the exemplar matched inside the GEMM (E <= 32)."""
    lib = load()
    E, M_max, K = A.shape
    N = B.shape[1]
    dt = _fwd_dtype(A, B, K)
    _check_fwd(dt, A, B, D, d_valid_m, SFA, SFB, status, E * M_max, M_max, E, N, K, E)
    _need(d_table, "table", n * EXEMPLAR_DTYPE.itemsize)
    _opt(tactic_out, "tactic_out", 12, _int32())
    _check("mgemm_masked_exemplar", lib.mgemm_masked_exemplar(
        dt, _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(D), _ptr(d_valid_m), E,
        M_max, N, K, _ptr(d_table), n, _ptr(tactic_out), _ptr(status), _stream(stream)))


def kgemm_grouped(dY, X, dW, d_counts, status=None, stream=None):
    import torch
    lib = load()
    T_cap, N = dY.shape
    K = X.shape[1]
    E = dW.shape[0]
    _need(dY, "dY", T_cap * N * 2, (torch.bfloat16,))
    _need(X, "X", T_cap * K * 2, (torch.bfloat16,))
    _need(dW, "dW", E * N * K * 4, (torch.float32,))
    _need(d_counts, "counts", E * 4, _int32())
    _opt(status, "status", 4, _int32())
    _check("kgemm_grouped", lib.kgemm_grouped(_ptr(dY), _ptr(X), _ptr(dW), _ptr(d_counts), E,
                                              T_cap, N, K, _ptr(status), _stream(stream)))


def set_wait_limit_ns(ns: int):
    load().mg_set_wait_limit_ns(int(ns))


def get_wait_limit_ns() -> int:
    return load().mg_get_wait_limit_ns()


def wait_selftest(status, limit_ns: int, stream=None):
    _need(status, "status", 4, _int32())
    _check("mg_wait_selftest", load().mg_wait_selftest(_ptr(status), int(limit_ns), _stream(stream)))


def set_kernel_policy(policy: int):
    _check("mg_set_kernel_policy", load().mg_set_kernel_policy(int(policy)))


def get_kernel_policy() -> int:
    return load().mg_get_kernel_policy()
