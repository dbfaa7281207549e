"""Checks that pin the CPU oracle to facts fixed outside it.

Each ``check_*`` raises AssertionError when the oracle disagrees with a closed
form, an invariant, a brute-force formulation or a textbook routine. They are
run as plain tests (test_oracle_pins.py) and again against oracles with a
planted mistake (test_oracle_mutations.py), which must each fail at least one.
Functions are looked up on the module at call time so that a mutation planted
with monkeypatch is seen.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

from oracle import moe_oracle as O
from mixture_experts_layer_mm_gb300.synthetic import f32_to_bf16_bits, random_small_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------- widening ---

def check_widen_bf16():
    # IEEE binary32 layout: sign | 8-bit exponent | mantissa; bf16 = top half.
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x4049],
                    dtype=np.uint16)
    want = [1.0, -2.0, 0.5, 0.0, -0.0, 3.3895313892515355e38, 2.0 ** -133, 3.140625]
    got = O.widen_bf16(bits)
    assert got.dtype == np.float32
    for g, w in zip(got.tolist(), want):
        assert g == w, (g, w)
    assert math.copysign(1.0, float(got[4])) < 0


# -------------------------------------------------------------- routing ---

# ------------------------------------------------------ bf16 rounding ---

def check_round_bf16():
    # Worked values: exact, ties to even (1 + 2^-8 sits halfway between 1 and
    # 1 + 2^-7), a tie that rounds up to the even neighbour, sign, inf, NaN.
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, np.inf, -0.0],
                 dtype=np.float32)
    want = [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F80, 0x8000]
    assert O.round_bf16(x).tolist() == want
    assert np.isnan(O.widen_bf16(O.round_bf16(np.array([np.nan], dtype=np.float32))))[0]
    # Library routine: torch's float32 -> bfloat16 cast (round to nearest even),
    # on random values and on random bit patterns (NaNs excluded).
    import torch
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 3,
                           rng.integers(0, 2 ** 32, 20000, dtype=np.uint64)
                           .astype(np.uint32).view(np.float32)])
    vals = vals[~np.isnan(vals)]
    lib = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(O.round_bf16(vals), lib.view(np.uint16))


# ------------------------------------------------------ add + RMSNorm ---

def check_mean_of_squares():
    rng = np.random.default_rng(12)
    # Small integers and H a power of two: the exact mean is a short binary
    # fraction, representable in float32, so the result must equal it.
    for H in (64, 2048, 4096):
        x = rng.integers(-3, 4, size=(5, H)).astype(np.float32)
        exact = (x.astype(np.int64) ** 2).sum(1) / H
        assert np.array_equal(O.mean_of_squares(x), exact.astype(np.float32))
    # Random rows (H not a power of two too): the exactly rounded float32 of
    # math.fsum's correctly rounded sum / H, to within one float32 rounding.
    for H in (192, 4096):
        x = rng.standard_normal((7, H)).astype(np.float32) * 30
        got = O.mean_of_squares(x).astype(np.float64)
        exact = np.array([math.fsum((r.astype(np.float64) ** 2).tolist()) / H for r in x])
        assert (np.abs(got - exact) <= 2.0 ** -24 * exact).all()
    # One element carries the whole sum: mean = v^2 / H exactly (H = 2^k).
    x = np.zeros((1, 1024), np.float32)
    x[0, 777] = 3.0
    assert O.mean_of_squares(x)[0] == np.float32(9.0 / 1024)


def _textbook_rmsnorm(r_bits, w_bits, eps):
    """float64 weight * x / sqrt(mean(x^2) + eps) via torch's rms_norm."""
    import torch
    xf = torch.from_numpy(O.widen_bf16(r_bits).astype(np.float64))
    wf = torch.from_numpy(O.widen_bf16(w_bits).astype(np.float64))
    return torch.nn.functional.rms_norm(xf, (xf.shape[-1],), wf, eps).numpy()


def check_rmsnorm_golden():
    g = json.load(open(os.path.join(GOLDEN, "add_rmsnorm_worked.json")))
    def row(d):
        return np.concatenate([np.full(n, int(b, 16), dtype=np.uint16) for b, n in d.items()])
    x, res = row(g["x_bits"])[None, :], row(g["residual_bits"])[None, :]
    w = np.full(g["H"], int(g["weight_bits"], 16), dtype=np.uint16)
    normed, r = O.fused_add_rmsnorm(x, res, w, g["eps"])
    assert np.array_equal(r[0], row(g["residual_out_bits"]))
    assert np.array_equal(normed[0], row(g["normed_bits"]))
    assert np.array_equal(O.rmsnorm(r, w, g["eps"]), normed)


def check_rmsnorm_closed_forms():
    rng = np.random.default_rng(13)
    H = 256
    w = _bf16(rng.uniform(0.5, 1.5, H))
    # Constant rows c * 1 with c a power of two, eps = 0: the row normalises
    # to sign(c) exactly, so the output is the weight with c's sign.
    for c in (0.25, -4.0, 1.0):
        out = O.rmsnorm(_bf16(np.full((1, H), c)), w, 0.0)
        assert np.array_equal(O.widen_bf16(out)[0], np.sign(c) * O.widen_bf16(w))
    # Scale invariance: with eps = 0 scaling a row by a power of two scales
    # every intermediate exactly, so the output is bit-identical.
    x = _bf16(rng.standard_normal((4, H)))
    for a in (2.0 ** -3, 2.0 ** 5):
        xs = _bf16(O.widen_bf16(x) * np.float32(a))
        assert np.array_equal(O.rmsnorm(xs, w, 0.0), O.rmsnorm(x, w, 0.0))
    # A zero row with eps > 0 gives zeros (no 0/0).
    assert not O.widen_bf16(O.rmsnorm(np.zeros((1, H), np.uint16), w, 1e-6)).any()
    # The textbook float64 RMSNorm (torch's rms_norm), within the two bf16
    # roundings; eps = 1 on small rows makes eps carry weight.
    for eps, scale in ((1e-6, 1.0), (1.0, 0.3)):
        x = _bf16(rng.standard_normal((6, H)) * scale)
        ref = _textbook_rmsnorm(x, w, eps)
        got = O.widen_bf16(O.rmsnorm(x, w, eps)).astype(np.float64)
        assert (np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30).all()


def check_fused_add_rmsnorm():
    rng = np.random.default_rng(14)
    T, H = 5, 192
    x = _bf16(rng.standard_normal((T, H)))
    res = _bf16(rng.standard_normal((T, H)) * 4)
    w = _bf16(rng.uniform(0.5, 1.5, H))
    normed, r = O.fused_add_rmsnorm(x, res, w, 1e-6)
    # The residual add is torch's bf16 add (one rounding of the exact sum).
    import torch
    tb = lambda b: torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    lib = (tb(x) + tb(res)).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r, lib)
    assert np.array_equal(normed, O.rmsnorm(r, w, 1e-6))
    n2, r2 = O.fused_add_rmsnorm(res, x, w, 1e-6)  # the add is symmetric
    assert np.array_equal(n2, normed) and np.array_equal(r2, r)
    # First layer: no residual yet, x is the residual.
    n0, r0 = O.fused_add_rmsnorm(x, None, w, 1e-6)
    assert np.array_equal(r0, x) and np.array_equal(n0, O.rmsnorm(x, w, 1e-6))


def check_router_logits_one_hot():
    # x[t] = e_{h_t}: logit[t, e] must be Wr[e, h_t] (+ bias[e]) exactly.
    rng = np.random.default_rng(1)
    T, H, E = 6, 16, 5
    hpos = rng.integers(0, H, size=T)
    x = np.zeros((T, H), dtype=np.float32)
    x[np.arange(T), hpos] = 1.0
    wr = O.widen_bf16(_bf16(rng.standard_normal((E, H))))
    bias = rng.standard_normal(E).astype(np.float32)
    got = O.router_logits(x, wr)
    assert np.array_equal(got, wr[:, hpos].T)
    got_b = O.router_logits(x, wr, bias)
    assert np.array_equal(got_b, (wr[:, hpos].T + bias[None, :]).astype(np.float32))


def check_softmax_closed_form():
    # softmax(ln c) = c / sum(c); invariant under a common shift of the logits.
    c = np.array([1.0, 2.0, 3.0, 4.0, 10.0])
    l = np.log(c).astype(np.float32)[None, :]
    p = O.softmax_over_experts(l)[0].astype(np.float64)
    assert np.allclose(p, c / c.sum(), rtol=2e-6, atol=0)
    p2 = O.softmax_over_experts(l + np.float32(300.0))[0]
    assert np.allclose(p2, c / c.sum(), rtol=2e-5, atol=0)
    big = np.array([[1000.0, 999.0, -1000.0]], dtype=np.float32)
    pb = O.softmax_over_experts(big)[0].astype(np.float64)
    e = math.e
    assert np.allclose(pb, [e / (e + 1), 1 / (e + 1), 0.0], rtol=1e-6, atol=1e-30)


def _topk_bruteforce(row: np.ndarray, k: int):
    """The k-subset with the largest logit sum (unique for distinct logits)."""
    best, best_s = None, -np.inf
    for s in itertools.combinations(range(row.size), k):
        v = float(np.sum(row[list(s)].astype(np.float64)))
        if v > best_s:
            best, best_s = s, v
    return list(best)


def check_topk_bruteforce():
    rng = np.random.default_rng(2)
    for E in (1, 2, 5, 8):
        for k in range(1, E + 1):
            logits = rng.standard_normal((7, E)).astype(np.float32)
            ids = O.select_topk(logits, k)
            assert ids.shape == (7, k) and ids.dtype == np.int32
            for t in range(7):
                assert list(ids[t]) == sorted(_topk_bruteforce(logits[t], k)), (E, k, t)


def check_topk_ties():
    # With ties the selected set S must satisfy, for s in S and u not in S:
    # l_s > l_u, or l_s == l_u and s < u (lower id wins); ids ascending.
    rng = np.random.default_rng(3)
    for _ in range(50):
        E = int(rng.integers(2, 10))
        k = int(rng.integers(1, E + 1))
        row = rng.integers(-2, 3, size=E).astype(np.float32)
        ids = list(O.select_topk(row[None, :], k)[0])
        assert ids == sorted(set(ids)) and len(ids) == k
        rest = [u for u in range(E) if u not in ids]
        for s in ids:
            for u in rest:
                assert row[s] > row[u] or (row[s] == row[u] and s < u), (row, ids)


def check_forced_routing_golden():
    g = json.load(open(os.path.join(GOLDEN, "forced_routing.json")))
    E = g["E"]
    H = 8
    x = _bf16(np.random.default_rng(4).standard_normal((3, H)))
    wr = np.zeros((E, H), dtype=np.uint16)          # router weights all zero
    bias = np.log(np.array(g["c"], dtype=np.float64)).astype(np.float32)
    ids, w, logits = O.route(x, wr, g["top_k"], False, bias)
    p = O.softmax_over_experts(logits)
    for t in range(3):
        assert np.allclose(p[t], g["probs"], rtol=2e-6, atol=0)
        assert list(ids[t]) == g["topk_ids_ascending"]
        assert np.allclose(w[t], g["topk_w_no_renorm"], rtol=2e-6, atol=0)
    ids, w, _ = O.route(x, wr, g["top_k"], True, bias)
    assert np.allclose(w, np.array(g["topk_w_renorm"])[None, :], rtol=2e-6, atol=0)
    ids, w, _ = O.route(x, wr, g["top_k3"], True, bias)
    assert (ids == np.array(g["topk3_ids_ascending"])[None, :]).all()
    assert np.allclose(w, np.array(g["topk3_w_renorm"])[None, :], rtol=2e-6, atol=0)


def check_forced_one_hot_ties():
    # H >= E, x_t = c * e_{pi(t)}, Wr = [I_E | 0]: token t's logits are c at
    # expert pi(t) and 0 elsewhere, so its top-1 is pi(t) and the remaining
    # k-1 slots go to the lowest ids among the tied zeros.
    E, H, T, k = 6, 8, 6, 3
    pi = np.array([3, 0, 5, 1, 4, 2])
    x = np.zeros((T, H), dtype=np.float32)
    x[np.arange(T), pi] = 2.0
    wr = np.zeros((E, H), dtype=np.float32)
    wr[np.arange(E), np.arange(E)] = 1.0
    ids, w, _ = O.route(_bf16(x), _bf16(wr), k, True)
    for t in range(T):
        rest = [e for e in range(E) if e != pi[t]][: k - 1]
        assert list(ids[t]) == sorted([pi[t]] + rest), (t, ids[t])
        e2 = math.exp(2.0)
        wt = {int(i): float(v) for i, v in zip(ids[t], w[t])}
        assert abs(wt[int(pi[t])] - e2 / (e2 + k - 1)) < 1e-6


def check_routing_weights():
    rng = np.random.default_rng(5)
    T, E, k = 9, 12, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    p = O.softmax_over_experts(logits)
    assert np.allclose(p.sum(1), 1.0, atol=1e-6) and (p > 0).all()
    ids = O.select_topk(logits, k)
    w0 = O.routing_weights(p, ids, False)
    w1 = O.routing_weights(p, ids, True)
    for t in range(T):
        for j in range(k):
            assert w0[t, j] == p[t, ids[t, j]]
    assert np.allclose(w1.sum(1), 1.0, atol=1e-6)
    assert np.allclose(w1 * w0.sum(1, keepdims=True), w0, rtol=1e-6)
    assert (w0.sum(1) < 1.0 + 1e-6).all() and (w1 <= 1.0 + 1e-6).all()


# ---------------------------------------------------------------- align ---

def _align_bruteforce(ids: np.ndarray, E: int, block_m: int):
    T, k = ids.shape
    flat = ids.reshape(-1)
    segs = []
    for e in range(E):
        fs = [f for f in range(T * k) if flat[f] == e]
        if fs:
            pad = (-len(fs)) % block_m
            segs.append((e, fs + [T * k] * pad))
        else:
            segs.append((e, []))
    return segs


def check_align_bruteforce():
    rng = np.random.default_rng(6)
    cases = []
    for _ in range(20):
        E = int(rng.integers(1, 12)); k = int(rng.integers(1, E + 1)); T = int(rng.integers(1, 40))
        ids = np.stack([np.sort(rng.choice(E, size=k, replace=False)) for _ in range(T)])
        cases.append((ids.astype(np.int32), E))
    # Edge cases: counts of block_m-1, block_m, block_m+1, zero-count experts,
    # one expert holding every token, a single token.
    bm = 4
    for c in (bm - 1, bm, bm + 1):
        cases.append((np.zeros((c, 1), dtype=np.int32) + 2, 5))
    cases.append((np.tile(np.array([[1, 3]], dtype=np.int32), (9, 1)), 6))
    cases.append((np.array([[0, 4, 7]], dtype=np.int32), 8))
    for ids, E in cases:
        T, k = ids.shape
        for block_m in (1, 4, 16, 128):
            s, off, cnt = O.align(ids, E, block_m)
            cap = O.align_capacity(T, k, E, block_m)
            assert s.shape == (cap,) and off.shape == (E + 1,) and cnt.shape == (E,)
            assert off[0] == 0 and off[E] <= cap
            for e, seg in _align_bruteforce(ids, E, block_m):
                assert list(s[off[e]:off[e + 1]]) == seg, (e, block_m)
                assert cnt[e] == sum(1 for f in seg if f < T * k)
                assert (off[e + 1] - off[e]) % block_m == 0
            assert (s[off[E]:] == T * k).all()
            real = s[s < T * k]
            assert np.array_equal(np.sort(real), np.arange(T * k))  # each f once


def check_align_rejects_bad_ids():
    try:
        O.align(np.array([[0, 9]], dtype=np.int32), 4, 4)
    except ValueError:
        return
    raise AssertionError("out-of-range expert id accepted")


# -------------------------------------------------------------- experts ---

def check_silu_identities():
    x = np.linspace(-30, 30, 121)
    one = np.ones_like(x)
    s = O.silu_and_mul(x, one)
    assert O.silu_and_mul(np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert np.allclose(s - O.silu_and_mul(-x, one), x, atol=1e-12)   # silu(x)-silu(-x)=x
    assert np.allclose(O.silu_and_mul(x, 3 * one), 3 * s, rtol=1e-15)
    assert abs(O.silu_and_mul(np.array([30.0]), np.array([1.0]))[0] - 30.0) < 1e-9
    assert abs(O.silu_and_mul(np.array([1.0]), np.array([1.0]))[0] - 1 / (1 + math.exp(-1))) < 1e-15


def _route_small(d, k, renorm):
    ids, w, _ = O.route(d["hidden"], d["router_w"], k, renorm, d["router_bias"])
    return ids, w


def check_loop_vs_dense():
    rng = np.random.default_rng(7)
    for trial in range(12):
        E = int(rng.integers(1, 9)); k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 40)); H = int(rng.choice([8, 16, 32])); I = int(rng.choice([4, 8, 16]))
        d = random_small_inputs(100 + trial, T, H, E, I, bias=bool(trial % 2))
        ids, w = _route_small(d, k, bool(trial % 3))
        ref = O.experts_dense_bruteforce(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
        got64 = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w, dtype=np.float64)
        got32 = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
        scale = np.abs(ref).max() + 1e-30
        assert np.abs(got64 - ref).max() <= 1e-12 * scale
        assert np.abs(got32 - ref).max() <= 1e-5 * scale


def check_k1_is_dense_gated_mlp():
    # k = 1 with renorm: the weight is 1 and the layer is the dense SwiGLU MLP
    # (GatedMLP) of the chosen expert; the same holds for E = 1.
    import torch
    import torch.nn.functional as F
    for E, k in ((6, 1), (1, 1)):
        T, H, I = 11, 16, 8
        d = random_small_inputs(11 + E, T, H, E, I)
        ids, w = _route_small(d, k, True)
        assert np.allclose(w, 1.0, atol=1e-7)
        got = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w, dtype=np.float64)
        x = torch.from_numpy(O.widen_bf16(d["hidden"]).astype(np.float64))
        for t in range(T):
            e = int(ids[t, 0])
            wgu = torch.from_numpy(O.widen_bf16(d["w_gate_up"][e]).astype(np.float64))
            wd = torch.from_numpy(O.widen_bf16(d["w_down"][e]).astype(np.float64))
            gate = F.linear(x[t:t + 1], wgu[:I])
            up = F.linear(x[t:t + 1], wgu[I:])
            want = F.linear(F.silu(gate) * up, wd)[0].numpy()
            assert np.allclose(got[t], want, rtol=1e-12, atol=1e-14), t


def check_closed_forms():
    T, H, E, I, k = 13, 16, 5, 8, 2
    d = random_small_inputs(21, T, H, E, I)
    ids, w = _route_small(d, k, True)
    base = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
    # gate rows zero -> silu(0) = 0 -> out is exactly zero
    wgu0 = d["w_gate_up"].copy(); wgu0[:, :I, :] = 0
    assert (O.experts_loop(d["hidden"], wgu0, d["w_down"], ids, w) == 0).all()
    # up rows zero -> out is exactly zero as well
    wgu1 = d["w_gate_up"].copy(); wgu1[:, I:, :] = 0
    assert (O.experts_loop(d["hidden"], wgu1, d["w_down"], ids, w) == 0).all()
    # doubling w_down (exact in bf16: exponent + 1) doubles out bit for bit
    wd2 = _bf16(O.widen_bf16(d["w_down"]) * 2)
    assert np.array_equal(O.experts_loop(d["hidden"], d["w_gate_up"], wd2, ids, w), 2 * base)
    # permuting tokens permutes out
    perm = np.random.default_rng(0).permutation(T)
    dp = dict(d); dp["hidden"] = d["hidden"][perm]
    ids_p, w_p = _route_small(dp, k, True)
    assert np.array_equal(ids_p, ids[perm])
    outp = O.experts_loop(dp["hidden"], d["w_gate_up"], d["w_down"], ids_p, w_p)
    assert np.allclose(outp, base[perm], rtol=1e-5, atol=1e-6 * np.abs(base).max())
    # relabelling experts jointly (router rows and both weight stacks) leaves out unchanged
    q = np.random.default_rng(1).permutation(E)
    dq = dict(d); dq["router_w"] = d["router_w"][q]
    dq["w_gate_up"] = d["w_gate_up"][q]; dq["w_down"] = d["w_down"][q]
    ids_q, w_q = _route_small(dq, k, True)
    outq = O.experts_loop(dq["hidden"], dq["w_gate_up"], dq["w_down"], ids_q, w_q)
    assert np.allclose(outq, base, rtol=1e-5, atol=1e-6 * np.abs(base).max())
    # a token whose weights are all on one expert equals that expert's MLP
    # (checked in check_k1_is_dense_gated_mlp); weights scale the output linearly
    w3 = (w * 3).astype(np.float32)
    assert np.allclose(O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w3),
                       3 * base, rtol=1e-6, atol=1e-7 * np.abs(base).max())


def check_moe_layer_invariants():
    from mixture_experts_layer_mm_gb300.synthetic import TINY, make_inputs
    d = make_inputs(TINY)
    r = O.moe_layer(d, TINY.top_k, TINY.renorm, block_m=4)
    T, k, E = TINY.T, TINY.top_k, TINY.E
    assert np.allclose(r["topk_w"].sum(1), 1.0, atol=1e-6)
    s, off = r["sorted_token_ids"], r["expert_offsets"]
    real = s[s < T * k]
    assert np.array_equal(np.sort(real), np.arange(T * k))
    tok = real // k
    assert np.array_equal(np.bincount(tok, minlength=T), np.full(T, k))  # k times each
    for e in range(E):
        seg = s[off[e]:off[e + 1]]
        seg = seg[seg < T * k]
        assert (r["topk_ids"].reshape(-1)[seg] == e).all()
    ref = O.experts_dense_bruteforce(d["hidden"], d["w_gate_up"], d["w_down"],
                                     r["topk_ids"], r["topk_w"])
    assert np.abs(r["out"] - ref).max() <= 1e-5 * np.abs(ref).max()


ALL_CHECKS = [v for n, v in sorted(globals().items()) if n.startswith("check_")]
