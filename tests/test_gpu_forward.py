"""End-to-end parity of mm_moe_forward against the CPU oracle.

Every workload shape is run at its full size. Where the oracle's expert loop
is too slow for the whole batch (T*I*H large), it is evaluated on a sample of
tokens (routing is per token, so a token's output depends only on its own
row); the routing and grouping are still compared on the whole batch.

The forward runs with a caller workspace, and the routing and grouping
compared here are the ones the forward itself computed and used (read from
that workspace at the offsets mm_moe_workspace_layout gives), whichever
kernels it chose for the batch size: the single launch (T <= 16 where its
shape limits allow, and mm_moe_forward_single_launch up to T = 64, which
routes and groups inside every CTA), the grouping fused into the router
(T <= 64), the one-block grouping (T <= 1024), count + place (up to 2048
tokens, or more than 128 experts), and the grouping from the tensor-core
router's per-tile counts (above 2048 tokens), with the token-row copy in the
same launch (E % 4 == 0) or after it. Expert ids must equal the oracle's on
every token whose k-th and (k+1)-th logits differ by more than 1e-4; the
grouping must equal the oracle's grouping of the forward's ids bit for bit;
the routing weights must match the oracle's weights of those ids within
W_RTOL.

The output is compared with the oracle's expert step taken on the GPU's own
routing (the conditional oracle) and, where no token is a near tie, with the
unconditional oracle, within max|err| <= 2e-2 max|ref| and mean relative
error <= 5e-3.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import (DECODE, LARGE, PREFILL, SWEEP, SWEEP_T,
                                                      TINY, MoEShape, make_inputs,
                                                      random_small_inputs)
from oracle import moe_oracle as O
from gpu_util import TIE_GAP, W_ATOL, W_RTOL, assert_out_close, dev_bf16, f32_dev

pytestmark = pytest.mark.gpu

_WEIGHTS = {}


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    yield mmlib
    _WEIGHTS.clear()


def _inputs(shape: MoEShape):
    key = (shape.H, shape.E, shape.I, shape.w_std, shape.router_std, shape.seed)
    d = make_inputs(shape, weights=key not in _WEIGHTS)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()  # one model shape at a time keeps host memory bounded
        _WEIGHTS[key] = {n: d[n] for n in ("router_w", "w_gate_up", "w_down")}
        _WEIGHTS[key]["dev"] = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    d.update({n: v for n, v in _WEIGHTS[key].items() if n != "dev"})
    return d, _WEIGHTS[key]["dev"]


def _run(d, dev_w, k, renorm, fn=None):
    """One forward (mm_moe_forward, or fn with the same arguments) with a
    caller workspace; returns out and the routing and grouping the forward
    left in that workspace."""
    fn = fn or mm.mm_moe_forward
    hidden = dev_bf16(d["hidden"])
    T, H = hidden.shape
    E, I = dev_w["router_w"].shape[0], dev_w["w_down"].shape[2]
    bias = None if d["router_bias"] is None else f32_dev(d["router_bias"])
    ws = torch.empty(mm.mm_moe_workspace_size(T, H, E, I, k), dtype=torch.uint8, device="cuda")
    out = fn(hidden, dev_w["router_w"], dev_w["w_gate_up"], dev_w["w_down"], k, renorm,
             router_bias=bias, workspace=ws)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    r = mm.forward_routing(ws, T, H, E, I, k)
    got = {n: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for n, v in r.items()}
    return out.float().cpu().numpy(), got


def _check(d, k, renorm, out_g, r_g, sample=None):
    T = d["hidden"].shape[0]
    E = d["router_w"].shape[0]
    ids_g, w_g = r_g["topk_ids"], r_g["topk_w"]
    ids_r, w_r, logits = O.route(d["hidden"], d["router_w"], k, renorm, d["router_bias"])
    tie = O.near_tie_tokens(logits, k, TIE_GAP)
    # ids: equal to the oracle's wherever the choice is unique, and valid everywhere
    assert np.array_equal(ids_g[~tie], ids_r[~tie])
    assert ids_g.min() >= 0 and ids_g.max() < E
    assert (np.diff(ids_g, axis=1) > 0).all(), "ids of a token must be distinct and ascending"
    # weights: the oracle's formula applied to the forward's ids
    probs_all = O.softmax_over_experts(logits)
    w_ids_g = O.routing_weights(probs_all, ids_g, renorm)
    np.testing.assert_allclose(w_g, w_ids_g, rtol=W_RTOL, atol=W_ATOL)
    # grouping: bit for bit the oracle's grouping of the forward's ids (the
    # oracle's own ids when no token is a near tie)
    s_r, off_r, cnt_r = O.align(ids_r if not tie.any() else ids_g, E, r_g["block_m"])
    assert np.array_equal(r_g["expert_counts"], cnt_r), "expert_counts"
    assert np.array_equal(r_g["expert_offsets"], off_r), "expert_offsets"
    assert np.array_equal(r_g["sorted_token_ids"], s_r), "sorted_token_ids"
    tok = np.arange(T) if sample is None else sample
    ref = O.experts_loop(d["hidden"][tok], d["w_gate_up"], d["w_down"], ids_g[tok], w_ids_g[tok])
    assert_out_close(out_g[tok], ref, "out (conditional oracle)")
    if not tie[tok].any():
        ref_u = O.experts_loop(d["hidden"][tok], d["w_gate_up"], d["w_down"], ids_r[tok], w_r[tok])
        assert_out_close(out_g[tok], ref_u, "out (oracle)")


def _sample(T, n, seed=0):
    if T <= n:
        return None
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], rng.choice(T, n, replace=False)]))


@pytest.mark.parametrize("shape", [TINY, DECODE, PREFILL], ids=lambda s: s.name)
def test_forward_workloads(shape):
    d, w = _inputs(shape)
    out, r = _run(d, w, shape.top_k, shape.renorm)
    _check(d, shape.top_k, shape.renorm, out, r, _sample(shape.T, 4096))


def test_forward_large_sampled():
    d, w = _inputs(LARGE)
    out, r = _run(d, w, LARGE.top_k, LARGE.renorm)
    _check(d, LARGE.top_k, LARGE.renorm, out, r, _sample(LARGE.T, 192))


@pytest.mark.parametrize("T", SWEEP_T)
def test_forward_zipf_sweep(T):
    shape = SWEEP.with_T(T)
    d, w = _inputs(shape)
    out, r = _run(d, w, shape.top_k, shape.renorm)
    _check(d, shape.top_k, shape.renorm, out, r, _sample(T, 1024))
    load = np.bincount(r["topk_ids"].reshape(-1), minlength=shape.E)
    if T >= 512:  # the bias skews the load: the busiest expert gets far more than the mean
        assert load.max() >= 3 * load.mean()


@pytest.mark.parametrize("T,H,E,k,I,renorm", [
    (1, 64, 1, 1, 64, True),      # one expert: the dense SwiGLU MLP
    (37, 128, 6, 1, 128, True),   # k = 1
    (50, 192, 8, 8, 64, False),   # every expert on every token
    (129, 256, 40, 5, 192, True), # E not a power of two, partial m-tiles
    (1000, 128, 64, 8, 64, True), # the one-block grouping at its largest token count
    (300, 64, 256, 32, 64, False),
    (2000, 128, 16, 4, 320, True),
    # above 2048 tokens the tensor-core router also writes per-tile expert
    # counts for the grouping: 32-, 64- and 128-token tiles; with E % 4 == 0
    # the grouping also copies the token rows (one launch), else a separate
    # row copy follows it
    (3000, 64, 100, 8, 64, False), (5000, 128, 40, 5, 192, True),
    (12000, 64, 128, 8, 64, True), (2500, 64, 30, 4, 64, True),
    # 32-token router tiles with a ragged last tile, wider rows
    (4100, 256, 64, 6, 128, True),
    # more than 128 experts above 2048 tokens: the cluster router, the
    # two-launch grouping and a separate row copy
    (2600, 64, 160, 4, 64, True),
])
def test_forward_shapes(T, H, E, k, I, renorm):
    d = random_small_inputs(T + 3 * E, T, H, E, I, w_std=0.08, bias=(E % 2 == 0))
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    out, r = _run(d, dw, k, renorm)
    _check(d, k, renorm, out, r)


# Shapes that mm_moe_forward_single_launch takes (T <= 64, T*k <= 512,
# H % 256 == 0 and H <= 2048, I % 128 == 0 and I <= 1024): one expert and one
# token; k = 1 with E not a power of two; every expert on every token (50
# tokens per expert: two passes of token groups over each weight slot); 256
# experts (the widest router finish) with T*k = 512; the largest I; K slices
# of three 32-column steps with E = 40; three experts holding up to 64 tokens;
# the decode workload itself (T = 64, its full size).
@pytest.mark.parametrize("T,H,E,k,I,renorm", [
    (1, 256, 1, 1, 128, True),
    (7, 256, 6, 1, 128, True),
    (50, 512, 8, 8, 256, False),
    (64, 256, 256, 8, 128, True),
    (16, 512, 4, 2, 1024, True),
    (33, 768, 40, 5, 384, True),
    (64, 256, 3, 2, 128, False),
])
def test_forward_single_launch_shapes(T, H, E, k, I, renorm):
    d = random_small_inputs(T + 5 * E, T, H, E, I, w_std=0.08, bias=(E % 2 == 0))
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    out, r = _run(d, dw, k, renorm, fn=mm.mm_moe_forward_single_launch)
    _check(d, k, renorm, out, r)


def test_forward_single_launch_decode_workload():
    d, dw = _inputs(DECODE)
    out, r = _run(d, dw, DECODE.top_k, DECODE.renorm, fn=mm.mm_moe_forward_single_launch)
    _check(d, DECODE.top_k, DECODE.renorm, out, r)


def test_forward_single_launch_rejects_other_shapes():
    T, H, E, k, I = 8, 192, 8, 2, 128  # H % 256 != 0
    d = random_small_inputs(3, T, H, E, I, w_std=0.08)
    dw = {n: dev_bf16(d[n]) for n in ("hidden", "router_w", "w_gate_up", "w_down")}
    with pytest.raises(mm.MMError) as ei:
        mm.mm_moe_forward_single_launch(dw["hidden"], dw["router_w"], dw["w_gate_up"],
                                        dw["w_down"], k, True)
    assert ei.value.code == mm.MM_ERR_UNSUPPORTED
    empty = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    d = random_small_inputs(3, 1, 256, E, I, w_std=0.08)
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    out0 = mm.mm_moe_forward_single_launch(empty, dw["router_w"], dw["w_gate_up"], dw["w_down"],
                                           k, True)
    assert out0.shape == (0, 256)


def test_forward_single_launch_forced_routing():
    # every token to experts {1, 6}: 64 tokens per expert, all in the same
    # two experts' units
    T, H, E, k, I = 64, 256, 8, 2, 128
    d = random_small_inputs(19, T, H, E, I, w_std=0.08)
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    bias = np.full(E, -30.0, dtype=np.float32)
    bias[[1, 6]] = 30.0
    out = mm.mm_moe_forward_single_launch(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"],
                                          dw["w_down"], k, True, router_bias=f32_dev(bias))
    ids, w, _ = O.route(d["hidden"], d["router_w"], k, True, bias)
    assert (ids == np.array([1, 6])).all()
    ref = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
    assert_out_close(out.float().cpu().numpy(), ref, "forced routing, single launch")


def test_forward_closed_forms():
    T, H, E, k, I = 200, 128, 8, 2, 128
    d = random_small_inputs(9, T, H, E, I, w_std=0.08)
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    # gate rows zero -> silu(0) = 0 -> out exactly zero
    wgu = d["w_gate_up"].copy()
    wgu[:, :I, :] = 0
    out0 = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dev_bf16(wgu), dw["w_down"],
                             k, True)
    assert (out0.float() == 0).all()
    # forced routing: every token to experts {1, 6} through the bias, renorm
    bias = np.full(E, -30.0, dtype=np.float32)
    bias[[1, 6]] = 30.0
    out_f = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"],
                              dw["w_down"], k, True, router_bias=f32_dev(bias))
    ids, w, _ = O.route(d["hidden"], d["router_w"], k, True, bias)
    assert (ids == np.array([1, 6])).all()
    ref = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
    assert_out_close(out_f.float().cpu().numpy(), ref, "forced routing")
    # repeat calls give the same routing and outputs within rounding of the
    # atomic accumulation order
    a = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"], dw["w_down"],
                          k, True).float()
    b = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"], dw["w_down"],
                          k, True).float()
    assert (a - b).abs().max().item() <= 1e-2 * a.abs().max().item()


def test_forward_caller_workspace_and_t0():
    T, H, E, k, I = 96, 128, 8, 2, 64
    d = random_small_inputs(4, T, H, E, I, w_std=0.08)
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    nbytes = mm.mm_moe_workspace_size(T, H, E, I, k)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"], dw["w_down"],
                            k, True, workspace=ws)
    ref = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"], dw["w_down"],
                            k, True)
    torch.cuda.synchronize()
    assert (out.float() - ref.float()).abs().max().item() <= 1e-2 * ref.float().abs().max().item()
    small = torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mm.MMError) as ei:
        mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"], dw["w_down"],
                          k, True, workspace=small)
    assert ei.value.code == mm.MM_ERR_NO_MEMORY
    empty = torch.zeros((0, H), dtype=torch.bfloat16, device="cuda")
    out0 = mm.mm_moe_forward(empty, dw["router_w"], dw["w_gate_up"], dw["w_down"], k, True)
    assert out0.shape == (0, H)
