"""GPU parity of mm_route and mm_align against the CPU oracle, through the C ABI.

Route: topk_ids bit-exact on every token whose k-th and (k+1)-th oracle logits
differ by more than 1e-4; on near-tie tokens the GPU's set must still be a
valid top-k within that gap. Weights within W_RTOL.
Align: all three outputs bit-exact, on every input (integer work).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import (DECODE, LARGE, PREFILL, SWEEP, TINY,
                                                      MoEShape, make_hidden, make_router_bias,
                                                      make_weights, random_small_inputs)
from oracle import moe_oracle as O
from gpu_util import TIE_GAP, W_ATOL, W_RTOL, dev_bf16, f32_dev, i32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


def _check_route(hidden, router_w, bias, k, renorm):
    T = hidden.shape[0]
    ids_ref, w_ref, logits = O.route(hidden, router_w, k, renorm, bias)
    ids_g, w_g = mm.mm_route(dev_bf16(hidden), dev_bf16(router_w), k, renorm,
                             router_bias=None if bias is None else f32_dev(bias))
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    ids_g = ids_g.cpu().numpy()
    w_g = w_g.cpu().numpy()
    tie = O.near_tie_tokens(logits, k, TIE_GAP)
    ok = ~tie
    assert np.array_equal(ids_g[ok], ids_ref[ok]), "topk_ids differ on non-tie tokens"
    np.testing.assert_allclose(w_g[ok], w_ref[ok], rtol=W_RTOL, atol=W_ATOL)
    # Near ties: ascending, distinct, and a valid top-k up to the gap.
    for t in np.nonzero(tie)[0]:
        s = ids_g[t]
        assert list(s) == sorted(set(s.tolist())) and len(s) == k
        rest = np.setdiff1d(np.arange(logits.shape[1]), s)
        if rest.size:
            assert logits[t, s].min() >= logits[t, rest].max() - TIE_GAP
        probs = O.softmax_over_experts(logits[t:t + 1])
        w_c = O.routing_weights(probs, s[None, :], renorm)[0]
        np.testing.assert_allclose(w_g[t], w_c, rtol=W_RTOL, atol=W_ATOL)
    if renorm:
        np.testing.assert_allclose(w_g.sum(1), 1.0, atol=1e-5)
    return ids_g, int(tie.sum())


@pytest.mark.parametrize("shape", [TINY, DECODE, PREFILL, LARGE, SWEEP.with_T(16384)],
                         ids=lambda s: s.name)
def test_route_workloads(shape):
    hidden = make_hidden(shape)
    w = make_weights(shape, experts=False)
    _check_route(hidden, w["router_w"], make_router_bias(shape), shape.top_k, shape.renorm)


@pytest.mark.parametrize("T,H,E,k,renorm,bias", [
    (1, 64, 1, 1, True, False), (63, 64, 5, 2, False, True), (65, 192, 33, 7, True, False),
    (130, 128, 200, 8, False, True), (257, 64, 256, 32, True, False), (64, 64, 256, 1, True, True),
    (100, 320, 64, 32, True, False), (7, 64, 31, 31, False, False),
])
def test_route_shapes(T, H, E, k, renorm, bias):
    d = random_small_inputs(T * 7 + E, T, H, E, 64, bias=bias)
    _check_route(d["hidden"], d["router_w"], d["router_bias"], k, renorm)


# Batches above 2048 tokens with at most 128 experts take the tensor-core
# router, with 32-, 64- or 128-token tiles as T grows (up to 32 x SMs, 64 x
# SMs, beyond): odd expert counts (rows past E of its 128-row tile), bias, no
# renorm, k up to 32, ragged last tiles, and wider rows (H up to 768: up to
# 12 K steps per tile).
@pytest.mark.parametrize("T,H,E,k,renorm,bias", [
    (65, 128, 128, 8, True, False), (4097, 64, 33, 7, True, True),
    (4500, 128, 128, 8, False, False), (5000, 192, 97, 32, True, False),
    (12001, 64, 64, 1, False, True), (20000, 64, 120, 6, True, True),
    (4097, 256, 128, 8, True, True), (4864, 512, 97, 8, False, False),
    (2200, 768, 128, 32, True, True), (6000, 256, 64, 6, True, True),
    (9000, 384, 128, 8, True, False), (9728, 128, 100, 4, False, True),
])
def test_route_tensor_core_shapes(T, H, E, k, renorm, bias):
    d = random_small_inputs(T + E + k, T, H, E, 64, bias=bias)
    _check_route(d["hidden"], d["router_w"], d["router_bias"], k, renorm)


@pytest.mark.parametrize("T,H", [(4200, 64), (8000, 64), (20000, 64), (4200, 256), (8000, 256)])
def test_route_tensor_core_forced_ties(T, H):
    # As below, at batch sizes that take the tensor-core router with each
    # token-tile size (H = 256: four times the K steps per tile): exact ties
    # between experts held by different threads of the group that finishes a
    # token.
    E, k = 128, 8
    c = (np.arange(E) % 5 + 1).astype(np.float64)  # values 1..5, each ~26 times
    bias = np.log(c).astype(np.float32)
    hidden = random_small_inputs(7, T, H, E, 64)["hidden"]
    rw = np.zeros((E, H), dtype=np.uint16)
    ids_g, w_g = mm.mm_route(dev_bf16(hidden), dev_bf16(rw), k, False, router_bias=f32_dev(bias))
    ids_g = ids_g.cpu().numpy()
    ids_ref, w_ref, _ = O.route(hidden, rw, k, False, bias)
    assert np.array_equal(ids_g, ids_ref)
    assert (ids_g == np.array([4, 9, 14, 19, 24, 29, 34, 39])[None, :]).all()
    np.testing.assert_allclose(w_g.cpu().numpy(), w_ref, rtol=W_RTOL)


def test_route_forced_ties():
    # Router weights zero, bias ln(c) with repeated c: exact ties resolved to
    # the lower expert id, identically on both sides.
    T, H, E, k = 40, 64, 16, 4
    c = np.array([3, 1, 3, 2, 3, 1, 1, 2, 3, 2, 1, 1, 2, 3, 1, 1], dtype=np.float64)
    bias = np.log(c).astype(np.float32)
    hidden = random_small_inputs(5, T, H, E, 64)["hidden"]
    rw = np.zeros((E, H), dtype=np.uint16)
    ids_g, w_g = mm.mm_route(dev_bf16(hidden), dev_bf16(rw), k, True, router_bias=f32_dev(bias))
    ids_g = ids_g.cpu().numpy()
    ids_ref, w_ref, _ = O.route(hidden, rw, k, True, bias)
    assert np.array_equal(ids_g, ids_ref)
    assert (ids_g == np.array([0, 2, 4, 8])[None, :]).all()
    np.testing.assert_allclose(w_g.cpu().numpy(), w_ref, rtol=W_RTOL)


def test_route_rejects_bad_args():
    h = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    rw = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mm.MMError) as ei:
        mm.mm_route(h, rw, 9, True)           # k > E
    assert ei.value.code == mm.MM_ERR_UNSUPPORTED
    h2 = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    rw2 = torch.zeros((8, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mm.MMError) as ei:
        mm.mm_route(h2, rw2, 2, True)         # H % 64 != 0
    assert ei.value.code == mm.MM_ERR_UNSUPPORTED


# ------------------------------------------------------------------ align ---

def _random_ids(rng, T, E, k):
    keys = rng.random((T, E))
    return np.sort(np.argsort(keys, axis=1)[:, :k], axis=1).astype(np.int32)


def _check_align(ids, E, block_m):
    T, k = ids.shape
    s_ref, off_ref, cnt_ref = O.align(ids, E, block_m)
    s_g, off_g, cnt_g = mm.mm_align(i32_dev(ids.reshape(T, k)), E, block_m)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    assert np.array_equal(off_g.cpu().numpy(), off_ref)
    assert np.array_equal(cnt_g.cpu().numpy(), cnt_ref)
    assert np.array_equal(s_g.cpu().numpy(), s_ref)
    return s_g, off_g, cnt_g


@pytest.mark.parametrize("T,E,k,block_m", [
    (1, 8, 2, 16), (16, 8, 2, 16), (64, 128, 8, 16), (1000, 128, 8, 16), (1024, 128, 8, 16),
    (1025, 128, 8, 16), (4096, 128, 8, 16), (16384, 128, 8, 16), (5000, 256, 8, 1),
    (3000, 33, 5, 128), (2049, 1, 1, 7), (700, 256, 32, 64), (8192, 128, 8, 128),
])
def test_align_random(T, E, k, block_m):
    ids = _random_ids(np.random.default_rng(T + E + k), T, E, k)
    s1 = _check_align(ids, E, block_m)
    s2 = mm.mm_align(i32_dev(ids), E, block_m)  # deterministic: bit-identical on a re-run
    assert torch.equal(s1[0], s2[0]) and torch.equal(s1[1], s2[1])


def test_align_edge_cases():
    bm = 16
    for c in (bm - 1, bm, bm + 1, 1):   # one expert with a count around the block size
        _check_align(np.full((c, 1), 3, dtype=np.int32), 8, bm)
    # every token on the same k experts: one expert holds T rows; others none
    _check_align(np.tile(np.array([[2, 5, 6]], dtype=np.int32), (3000, 1)), 8, bm)
    _check_align(np.tile(np.array([[0, 127]], dtype=np.int32), (777, 1)), 128, 128)
    # T = 0: empty segments, all sentinels
    s, off, cnt = mm.mm_align(torch.zeros((0, 2), dtype=torch.int32, device="cuda"), 8, bm)
    assert (off.cpu().numpy() == 0).all() and (s.cpu().numpy() == 0).all()
    # Zipf-skewed real routing, T = 16384
    shape = SWEEP.with_T(16384)
    ids, _, _ = O.route(make_hidden(shape), make_weights(shape, experts=False)["router_w"],
                        shape.top_k, shape.renorm, make_router_bias(shape))
    _check_align(ids, shape.E, bm)


def test_align_flags_bad_ids():
    ids = np.array([[0, 3], [1, 9], [2, 2], [-1, 4]], dtype=np.int32)
    s, off, cnt = mm.mm_align(i32_dev(ids), 8, 4)
    assert mm.mm_poll_device_status() == mm.MM_ERR_DEVICE
    assert mm.mm_poll_device_status() == mm.MM_OK   # cleared by the read
    # The valid, first-occurrence assignments are still grouped correctly.
    flat = ids.reshape(-1)
    s = s.cpu().numpy()
    off = off.cpu().numpy()
    for e in range(8):
        want = [f for f in range(flat.size) if flat[f] == e and
                f not in (5,)]  # f = 5 is the repeated '2' of token 2
        got = [f for f in s[off[e]:off[e + 1]] if f < flat.size]
        assert got == want, (e, got, want)
