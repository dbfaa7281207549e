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


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def f32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def i32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


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
