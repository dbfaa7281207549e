"""The seeded input recipe, on CPU: what the GPU path and the oracle both read.

Checks that the generators give exactly representable bf16 values with the
stated spreads, that the streams are independent of T and of one another, and
that the per-expert logit bias of the skewed sweep has the Zipf(1.1) ratios
and skews the realised routing.
"""
import dataclasses

import numpy as np
import pytest
import torch

from mixture_experts_layer_mm_gb300 import synthetic as S
from oracle import moe_oracle as O


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(7).standard_normal(100_000, dtype=np.float32) * 3
    ours = S.f32_to_bf16_bits(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_spreads_and_determinism():
    sh = dataclasses.replace(S.DECODE, T=256, E=4)      # the decode recipe with 4 experts
    h = S.make_hidden(sh)
    w = S.make_weights(sh)
    assert h.dtype == np.uint16 and h.shape == (256, 2048)
    assert np.std(_f32(h)) == pytest.approx(1.0, rel=0.02)
    assert np.std(_f32(w["router_w"])) == pytest.approx(0.02, rel=0.05)
    assert np.std(_f32(w["w_gate_up"])) == pytest.approx(0.02, rel=0.01)
    assert w["w_gate_up"].shape == (4, 1536, 2048) and w["w_down"].shape == (4, 2048, 768)
    assert np.array_equal(S.make_hidden(sh), h)           # same seed, same bits


def test_weights_do_not_depend_on_T():
    a = S.make_weights(dataclasses.replace(S.TINY, T=1))
    b = S.make_weights(dataclasses.replace(S.TINY, T=999))
    for name in ("router_w", "w_gate_up", "w_down"):
        assert np.array_equal(a[name], b[name])
    # the first rows of hidden do not depend on T either (one stream, drawn in order)
    h1 = S.make_hidden(dataclasses.replace(S.TINY, T=4))
    h2 = S.make_hidden(dataclasses.replace(S.TINY, T=16))
    assert np.array_equal(h1, h2[:4])


def test_zipf_bias_ratios():
    perm = np.random.default_rng(0).permutation(128)
    b = S.zipf_logit_bias(128, 1.1, perm).astype(np.float64)
    q = np.exp(b)
    assert q.sum() == pytest.approx(1.0, rel=1e-6)
    by_rank = q[np.argsort(perm)]                        # expert holding rank 1, 2, ...
    assert np.all(np.diff(by_rank) < 0)
    assert by_rank[0] / by_rank[1] == pytest.approx(2 ** 1.1, rel=1e-5)
    assert by_rank[0] / by_rank[9] == pytest.approx(10 ** 1.1, rel=1e-5)


def test_zipf_bias_skews_the_routing():
    sh = S.SWEEP.with_T(512)
    d = S.make_inputs(sh, weights=False)                # hidden, router_w and the bias
    ids, _, _ = O.route(d["hidden"], d["router_w"], sh.top_k, sh.renorm, d["router_bias"])
    load = np.bincount(ids.reshape(-1), minlength=sh.E)
    assert load.max() >= 3 * load.mean()
    assert load.max() <= sh.T                            # one row per token at most
    ids_u, _, _ = O.route(d["hidden"], d["router_w"], sh.top_k, sh.renorm)
    load_u = np.bincount(ids_u.reshape(-1), minlength=sh.E)
    assert load_u.max() < 2 * load_u.mean()              # without the bias: near uniform
