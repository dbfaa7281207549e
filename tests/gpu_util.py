"""Helpers for the GPU parity tests: device transfer and the comparison rules."""
from __future__ import annotations

import numpy as np
import torch

# Output tolerance of the layer (bf16 out vs the fp32 oracle):
#   max |gpu - ref| <= 2e-2 * max |ref|   and   sum |gpu - ref| / sum |ref| <= 5e-3
OUT_MAX_REL = 2e-2
OUT_MEAN_REL = 5e-3
# Routing weights: fp32 on both sides, the logits summed in different orders.
# A logit error d changes p by a relative ~d; with |logit error| of a few 1e-6
# for H <= 4096 (random-walk rounding of fp32 sums of bf16 products), 1e-4
# relative leaves a wide margin while still catching any wrong formula.
W_RTOL = 1e-4
W_ATOL = 1e-7
TIE_GAP = 1e-4  # k-th vs (k+1)-th logit gap below which either expert is correct
# RMSNorm rows: the oracle takes the exact mean of the squares (rounded once
# to float32), a kernel its own float32 sum. The two inverse norms then differ
# by a few float32 ulps, which moves y = bf16(x * inv) by one bf16 step where
# x * inv sits within that distance of a rounding boundary (a fraction of
# order 1e-4 of the elements), and weight * y by at most two steps after its
# own rounding. Anything beyond that is a wrong formula.
NORM_MAX_STEPS = 2
NORM_MAX_MISMATCH = 2e-3


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def f32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def i32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_steps(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in representable bf16 values between two arrays of bf16 bit
    patterns (sign-magnitude mapped to a monotone integer scale)."""
    def ordered(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        return np.where(b & 0x8000, 0x8000 - b, b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def assert_norm_rows_close(got_bits: np.ndarray, want_bits: np.ndarray, what="normed") -> None:
    d = bf16_steps(got_bits, want_bits)
    assert d.max() <= NORM_MAX_STEPS, f"{what}: {d.max()} bf16 steps from the oracle"
    frac = np.count_nonzero(d) / max(d.size, 1)
    assert frac <= NORM_MAX_MISMATCH, f"{what}: {frac:.2e} of elements differ"


def assert_out_close(got: np.ndarray, ref: np.ndarray, what: str = "out",
                     max_rel: float = OUT_MAX_REL, mean_rel: float = OUT_MEAN_REL) -> None:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    denom = np.abs(ref).sum()
    assert err.max() <= max_rel * scale + 1e-30, \
        f"{what}: max|err| {err.max():.3e} > {max_rel} * max|ref| {scale:.3e}"
    assert err.sum() <= mean_rel * denom + 1e-30, \
        f"{what}: sum|err|/sum|ref| {err.sum() / max(denom, 1e-30):.3e} > {mean_rel}"
