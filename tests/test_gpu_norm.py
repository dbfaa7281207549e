"""GPU parity of the residual add + RMSNorm step (mm_add_rmsnorm) and of the
MoE layer behind it (mm_moe_forward_add_norm) against the CPU oracle.

The new residual is one correctly rounded bf16 add on both sides, so it must
be bit-exact. For the normalised rows the oracle takes the exact mean of the
squares, rounded once to float32, and the kernel its own float32 sum: they
must agree within NORM_MAX_STEPS bf16 steps, and differ at all only on a
small fraction of the elements (gpu_util states the bound and its reason).
Rows whose sum of squares is exact in float32 (the hand-worked case) must be
bit-exact. The layer's output is then compared as in test_gpu_forward: with
the oracle's expert step on the GPU's own normalised rows and routing, and
with the plain oracle on tokens whose rows match bit for bit and are not
near ties.
"""
import json
import os

import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import (DECODE, PREFILL, TINY, make_inputs,
                                                      make_norm_inputs)
from oracle import moe_oracle as O
from gpu_util import TIE_GAP, assert_norm_rows_close, assert_out_close, dev_bf16

pytestmark = pytest.mark.gpu
EPS = 1e-6
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "add_rmsnorm_worked.json")


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,H", [(1, 64), (37, 128), (5, 192), (64, 2048), (300, 4096),
                                 (4096, 2048)])
@pytest.mark.parametrize("with_residual", [True, False])
def test_add_rmsnorm(T, H, with_residual):
    d = make_norm_inputs(T + H, T, H)
    res = dev_bf16(d["residual"]) if with_residual else None
    normed = mm.mm_add_rmsnorm(dev_bf16(d["x"]), dev_bf16(d["norm_w"]), EPS, residual=res)
    torch.cuda.synchronize()
    want_n, want_r = O.fused_add_rmsnorm(d["x"], d["residual"] if with_residual else None,
                                         d["norm_w"], EPS)
    assert_norm_rows_close(_bits(normed), want_n)
    if with_residual:
        assert np.array_equal(_bits(res), want_r)


def test_add_rmsnorm_golden():
    g = json.load(open(GOLDEN))

    def row(spec):
        return np.concatenate([np.full(n, int(b, 16), dtype=np.uint16) for b, n in spec.items()])
    x = dev_bf16(row(g["x_bits"])[None, :])
    res = dev_bf16(row(g["residual_bits"])[None, :])
    w = dev_bf16(np.full(g["H"], int(g["weight_bits"], 16), dtype=np.uint16))
    normed = mm.mm_add_rmsnorm(x, w, g["eps"], residual=res)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(res)[0], row(g["residual_out_bits"]))
    assert np.array_equal(_bits(normed)[0], row(g["normed_bits"]))


def test_add_rmsnorm_large_values():
    # Rows far from unit scale (residual stream of a deep model): the sum of
    # squares grows to ~1e9 without leaving float32's exact-rounding regime.
    T, H = 33, 2048
    d = make_norm_inputs(5, T, H, residual_std=300.0)
    res = dev_bf16(d["residual"])
    normed = mm.mm_add_rmsnorm(dev_bf16(d["x"]), dev_bf16(d["norm_w"]), EPS, residual=res)
    torch.cuda.synchronize()
    want_n, want_r = O.fused_add_rmsnorm(d["x"], d["residual"], d["norm_w"], EPS)
    assert np.array_equal(_bits(res), want_r)
    assert_norm_rows_close(_bits(normed), want_n)


@pytest.mark.parametrize("shape", [TINY, DECODE.with_T(8), DECODE, PREFILL],
                         ids=lambda s: s.name)
def test_moe_forward_add_norm(shape):
    T, H, k = shape.T, shape.H, shape.top_k
    w = make_inputs(shape)
    n = make_norm_inputs(shape.seed + 17, T, H)
    dw = {name: dev_bf16(w[name]) for name in ("router_w", "w_gate_up", "w_down")}
    x, nw = dev_bf16(n["x"]), dev_bf16(n["norm_w"])
    res = dev_bf16(n["residual"])
    out = mm.mm_moe_forward_add_norm(x, nw, EPS, dw["router_w"], dw["w_gate_up"], dw["w_down"],
                                     k, shape.renorm, residual=res)
    # The GPU's routing of the same normalised rows (same kernels, deterministic).
    res2 = dev_bf16(n["residual"])
    normed_g = mm.mm_add_rmsnorm(x, nw, EPS, residual=res2)
    ids_g, _ = mm.mm_route(normed_g, dw["router_w"], k, shape.renorm)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    out = out.float().cpu().numpy()
    ids_g = ids_g.cpu().numpy()

    normed, r = O.fused_add_rmsnorm(n["x"], n["residual"], n["norm_w"], EPS)
    assert np.array_equal(_bits(res), r)
    normed_gb = _bits(normed_g)
    assert_norm_rows_close(normed_gb, normed)
    # The layer's routing: the oracle's on the GPU's own normalised rows.
    ids_c, _, logits_c = O.route(normed_gb, w["router_w"], k, shape.renorm)
    tie = O.near_tie_tokens(logits_c, k, TIE_GAP)
    assert np.array_equal(ids_g[~tie], ids_c[~tie])
    tok = np.arange(T)
    if T > 1024:
        rng = np.random.default_rng(0)
        tok = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 1024, replace=False)]))
    probs = O.softmax_over_experts(logits_c[tok])
    w_c = O.routing_weights(probs, ids_g[tok], shape.renorm)
    ref = O.experts_loop(normed_gb[tok], w["w_gate_up"], w["w_down"], ids_g[tok], w_c)
    assert_out_close(out[tok], ref, "out (conditional oracle)")
    # The plain oracle end to end, on tokens whose rows the two sides
    # normalised identically and whose routing is not a near tie.
    ids_r, w_r, logits = O.route(normed, w["router_w"], k, shape.renorm)
    same = (normed_gb == normed).all(axis=1)
    keep = tok[same[tok] & ~O.near_tie_tokens(logits, k, TIE_GAP)[tok]]
    assert keep.size >= 0.75 * tok.size
    ref_u = O.experts_loop(normed[keep], w["w_gate_up"], w["w_down"], ids_r[keep], w_r[keep])
    assert_out_close(out[keep], ref_u, "out (oracle, non-tie tokens)")


def test_moe_forward_add_norm_first_layer():
    # No residual yet: x is the residual and stays as it was.
    shape = TINY
    w = make_inputs(shape)
    n = make_norm_inputs(3, shape.T, shape.H)
    dw = {name: dev_bf16(w[name]) for name in ("router_w", "w_gate_up", "w_down")}
    x, nw = dev_bf16(n["x"]), dev_bf16(n["norm_w"])
    out = mm.mm_moe_forward_add_norm(x, nw, EPS, dw["router_w"], dw["w_gate_up"], dw["w_down"],
                                     shape.top_k, shape.renorm)
    normed_g = _bits(mm.mm_add_rmsnorm(x, nw, EPS))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(x), n["x"])
    normed, _ = O.fused_add_rmsnorm(n["x"], None, n["norm_w"], EPS)
    assert_norm_rows_close(normed_g, normed)
    ids_r, w_r, logits = O.route(normed_g, w["router_w"], shape.top_k, shape.renorm)
    keep = ~O.near_tie_tokens(logits, shape.top_k, TIE_GAP)
    ref = O.experts_loop(normed_g[keep], w["w_gate_up"], w["w_down"], ids_r[keep], w_r[keep])
    assert_out_close(out.float().cpu().numpy()[keep], ref, "out (first layer)")


def _bf16_add(a_bits, b_bits):
    """bf16(a + b) of two bf16 tensors (a correctly rounded float32 add of
    exact widenings, as a bf16 tensor add does)."""
    return O.round_bf16(O.widen_bf16(a_bits) + O.widen_bf16(b_bits))


@pytest.mark.parametrize("shape", [TINY, DECODE.with_T(8), DECODE, PREFILL],
                         ids=lambda s: s.name)
@pytest.mark.parametrize("in_place", [True, False])
def test_moe_forward_add_norm_residual(shape, in_place):
    # DecoderLayer.forward's order: residual' = x + residual, the MoE block on
    # rmsnorm(residual'), then the next add: residual'' = out + residual'.
    T, H, k = shape.T, shape.H, shape.top_k
    w = make_inputs(shape)
    n = make_norm_inputs(shape.seed + 29, T, H)
    dw = {name: dev_bf16(w[name]) for name in ("router_w", "w_gate_up", "w_down")}
    x, nw = dev_bf16(n["x"]), dev_bf16(n["norm_w"])
    res = dev_bf16(n["residual"])
    res_out = None if in_place else torch.empty_like(res)
    out, r2 = mm.mm_moe_forward_add_norm_residual(x, nw, EPS, dw["router_w"], dw["w_gate_up"],
                                                  dw["w_down"], k, shape.renorm, residual=res,
                                                  residual_out=res_out)
    normed_g = mm.mm_add_rmsnorm(x, nw, EPS, residual=dev_bf16(n["residual"]))
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    assert (r2.data_ptr() == res.data_ptr()) == in_place
    normed, r1 = O.fused_add_rmsnorm(n["x"], n["residual"], n["norm_w"], EPS)
    out_b = _bits(out)
    # the add after the layer: bit for bit on the layer's own output
    assert np.array_equal(_bits(r2), _bf16_add(out_b, r1))
    if not in_place:
        assert np.array_equal(_bits(res), r1)  # residual' left in residual
    # the layer's output against the oracle on the GPU's normalised rows
    normed_gb = _bits(normed_g)
    assert_norm_rows_close(normed_gb, normed)
    ids_c, _, logits_c = O.route(normed_gb, w["router_w"], k, shape.renorm)
    tok = np.arange(T)
    if T > 1024:
        rng = np.random.default_rng(1)
        tok = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 1024, replace=False)]))
    keep = tok[~O.near_tie_tokens(logits_c, k, TIE_GAP)[tok]]
    probs = O.softmax_over_experts(logits_c[keep])
    w_c = O.routing_weights(probs, ids_c[keep], shape.renorm)
    ref = O.experts_loop(normed_gb[keep], w["w_gate_up"], w["w_down"], ids_c[keep], w_c)
    assert_out_close(O.widen_bf16(out_b)[keep], ref, "out (oracle on the GPU's normed rows)")


def test_moe_forward_add_norm_residual_first_layer():
    # No residual yet: residual' = x, and residual_out = bf16(out + x).
    shape = TINY
    w = make_inputs(shape)
    n = make_norm_inputs(31, shape.T, shape.H)
    dw = {name: dev_bf16(w[name]) for name in ("router_w", "w_gate_up", "w_down")}
    x = dev_bf16(n["x"])
    out, r2 = mm.mm_moe_forward_add_norm_residual(x, dev_bf16(n["norm_w"]), EPS, dw["router_w"],
                                                  dw["w_gate_up"], dw["w_down"], shape.top_k,
                                                  shape.renorm)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(x), n["x"])
    assert np.array_equal(_bits(r2), _bf16_add(_bits(out), n["x"]))
