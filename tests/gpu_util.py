"""Shared pieces of the GPU parity tests: operand set-up with poisoned
padding, sentinel-filled outputs, and the acceptance rules.

Acceptance (fixed for every form):
* bf16 inputs, fp32 accumulation, bf16 output: per output row,
  max|D - R| <= 1e-2 * max|R|; a row whose reference is all zero must be 0.
* fp8 inputs: per expert, ||D - R||_F <= 2e-3 * ||R||_F.
* rows the form does not compute keep the sentinel bit pattern exactly.
"""
import numpy as np
import torch

from moe_grouped_gemm_side_gb300 import workloads as wl
from oracle import numerics as on

SENTINEL_BITS = 0x7BAD          # a finite bf16 (~1.9e36) no kernel produces here
BF16_ROW_TOL = 1e-2
FP8_FROB_TOL = 2e-3


def sentinel_like(shape, device):
    return torch.full(shape, SENTINEL_BITS, dtype=torch.int16, device=device).view(torch.bfloat16)


def bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def deq_bf16(t):
    return on.decode_bf16(bf16_bits(t.contiguous()))


def deq_rows_fp8(codes, sf):
    return on.dequant_rows(codes.cpu().numpy(), sf.cpu().numpy())


def deq_weight_fp8(codes, sf):
    return on.dequant_weight(codes.cpu().numpy(), sf.cpu().numpy())


def check_rows_bf16(D_rows_bits, R_rows):
    """Per-row max-abs rule on written rows; returns the worst ratio."""
    D = on.decode_bf16(D_rows_bits).reshape(R_rows.shape)
    m = np.max(np.abs(R_rows), axis=-1)
    err = np.max(np.abs(D - R_rows), axis=-1)
    assert np.all(np.isfinite(err)), "non-finite output in a valid row"
    zero = m == 0.0
    assert np.all(err[zero] == 0.0), "a row whose reference is zero is not zero"
    ratio = err[~zero] / m[~zero]
    bad = np.nonzero(ratio > BF16_ROW_TOL)[0]
    assert bad.size == 0, f"{bad.size} rows over tolerance, worst {ratio.max()}"
    return float(ratio.max()) if ratio.size else 0.0


def check_frobenius(D_bits, R):
    D = on.decode_bf16(D_bits)
    num = np.linalg.norm(D - R)
    den = np.linalg.norm(R)
    assert np.isfinite(num)
    if den == 0.0:
        assert num == 0.0
        return 0.0
    rel = num / den
    assert rel <= FP8_FROB_TOL, f"relative Frobenius error {rel}"
    return rel


def poison_rows_(A, rows_mask_np, fp8: bool, SFA=None):
    """Fill rows outside `rows_mask` with NaN (and their scales with the UE8M0
    NaN byte) so that any leak into a valid output row shows up."""
    idx = torch.from_numpy(np.nonzero(~rows_mask_np)[0]).to(A.device)
    if idx.numel() == 0:
        return
    if fp8:
        A.index_fill_(0, idx, wl.E4M3_NAN_CODE)
        if SFA is not None:
            SFA.index_fill_(1, idx, wl.UE8M0_NAN_CODE)
    else:
        A.view(torch.int16).index_fill_(0, idx, wl.BF16_NAN_BITS)


def poison_experts_(B, dead, fp8: bool, SFB=None):
    """Fill the weights (and weight scales) of experts that have no rows to
    compute with NaN.  Such an expert loads no weights, and a tile that took
    its weights from the wrong expert would carry the NaN into a valid row."""
    idx = [e for e, d in enumerate(dead) if d]
    if not idx:
        return
    i = torch.tensor(idx, dtype=torch.int64, device=B.device)
    if fp8:
        B.index_fill_(0, i, wl.E4M3_NAN_CODE)
        if SFB is not None:
            SFB.index_fill_(0, i, wl.UE8M0_NAN_CODE)
    else:
        B.view(torch.int16).index_fill_(0, i, wl.BF16_NAN_BITS)


def integer_e4m3(shape, seed, device):
    """E4M3 codes of the integers -2..2 (exactly representable)."""
    lut = torch.tensor([0xC0, 0xB8, 0x00, 0x38, 0x40], dtype=torch.uint8)
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, 5, tuple(shape), generator=g)
    return lut[idx].to(device)


def rand_scales(shape, seed, device, lo=124, hi=130):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32).to(torch.uint8).to(device)


def round_bf16_bits(R):
    """Round-to-nearest-even of float64 values that are exact in fp32."""
    t = torch.from_numpy(np.ascontiguousarray(R)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)
