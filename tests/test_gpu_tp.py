"""The tensor-parallel split of the layer on one GPU: W slices of the
experts' intermediates ("The op layer: BaseOP and the layers", "Linear
layers"), each run by mm_moe_forward_partial, summed in fp32 (the all-reduce
of W ranks) and rounded once by mm_round_bf16, must give the layer: checked
against the oracle with the layer's tolerance, and against the unsliced
forward. mm_round_bf16 itself must round exactly as the oracle's round_bf16.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import DECODE, PREFILL, TINY, make_inputs
from oracle import moe_oracle as O
from gpu_util import TIE_GAP, assert_out_close, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


def test_round_bf16_matches_the_oracle():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(1 << 16).astype(np.float32) * 3,
                        # exact ties between two bf16 values, both parities
                        (np.arange(1 << 12, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, 1e-40, -3e38, np.inf, -np.inf], np.float32)])
    x = x[: len(x) // 4 * 4]
    got = mm.mm_round_bf16(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16), O.round_bf16(x))


# T=8 takes the single-launch layer for the whole layer and for 2-way
# slices (I/2 = 384), the kernel chain for 4-way slices (I/4 = 192 is not a
# multiple of 128).
@pytest.mark.parametrize("shape", [DECODE.with_T(8), DECODE, PREFILL], ids=lambda s: s.name)
@pytest.mark.parametrize("world", [2, 4])
def test_slices_sum_to_the_layer(shape, world):
    d = make_inputs(shape)
    k = shape.top_k
    hidden, rw = dev_bf16(d["hidden"]), dev_bf16(d["router_w"])
    wgu, wdn = dev_bf16(d["w_gate_up"]), dev_bf16(d["w_down"])
    total = torch.zeros((shape.T, shape.H), dtype=torch.float32, device="cuda")
    for r in range(world):
        gu, dn = mm.tp_slice(wgu, wdn, r, world)
        total += mm.mm_moe_forward_partial(hidden, rw, gu, dn, k, shape.renorm)
    out = mm.mm_round_bf16(total)
    full = mm.mm_moe_forward(hidden, rw, wgu, wdn, k, shape.renorm)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    got = out.float().cpu().numpy()
    # the sliced layer against the unsliced one (the same routing, other
    # summation orders and roundings of act)
    assert_out_close(got, full.float().cpu().numpy(), "sliced vs unsliced")
    # and against the oracle, on tokens whose routing is unique
    ids_r, w_r, logits = O.route(d["hidden"], d["router_w"], k, shape.renorm)
    tok = np.arange(shape.T)
    if shape.T > 512:
        tok = np.unique(np.random.default_rng(2).choice(shape.T, 512, replace=False))
    tok = tok[~O.near_tie_tokens(logits[tok], k, TIE_GAP)]
    ref = O.experts_loop(d["hidden"][tok], d["w_gate_up"], d["w_down"], ids_r[tok], w_r[tok])
    assert_out_close(got[tok], ref, "sliced layer vs oracle")


def test_partial_of_one_slice_is_the_unrounded_layer():
    shape = TINY
    d = make_inputs(shape)
    hidden, rw = dev_bf16(d["hidden"]), dev_bf16(d["router_w"])
    wgu, wdn = dev_bf16(d["w_gate_up"]), dev_bf16(d["w_down"])
    part = mm.mm_moe_forward_partial(hidden, rw, wgu, wdn, shape.top_k, shape.renorm)
    torch.cuda.synchronize()
    ref = O.moe_layer(d, shape.top_k, shape.renorm)["out"]
    assert_out_close(part.cpu().numpy(), ref, "fp32 partial of the whole layer")
