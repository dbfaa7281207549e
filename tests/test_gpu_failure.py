"""The device-side failure path: a bounded wait that runs out.

Every kernel waits on mbarriers with a time limit (about a second of
%globaltimer); when it runs out the kernel records a timeout in the
per-device status word, unwinds and returns. mm_selftest_wait_timeout runs
one kernel whose wait can never complete (a barrier nothing arrives on),
which is the only way to make the limit run out without breaking a real
kernel. mm_selftest_layer_barrier_timeout runs the single-launch small-batch
layer with a host-set flag that keeps CTA 0 from arriving at one of its
grid-wide barriers, so every CTA's wait there runs out. The tests check the
reported status, the time it took, and that the library works normally
afterwards.
"""
import time

import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import TINY, make_inputs, random_small_inputs
from oracle import moe_oracle as O
from gpu_util import assert_out_close, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


def test_wait_times_out_and_context_survives():
    assert mm.mm_poll_device_status() == mm.MM_OK  # nothing pending
    t0 = time.perf_counter()
    mm.mm_selftest_wait_timeout()
    rc = mm.mm_poll_device_status()
    dt = time.perf_counter() - t0
    assert rc == mm.MM_ERR_TIMEOUT
    assert 0.9 <= dt < 30.0, dt                     # the limit is about a second
    assert mm.mm_poll_device_status() == mm.MM_OK  # the word was cleared

    d = make_inputs(TINY)
    dw = {n: dev_bf16(d[n]) for n in ("router_w", "w_gate_up", "w_down")}
    out = mm.mm_moe_forward(dev_bf16(d["hidden"]), dw["router_w"], dw["w_gate_up"],
                            dw["w_down"], TINY.top_k, TINY.renorm)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    ref = O.moe_layer(d, TINY.top_k, TINY.renorm)
    assert_out_close(out.float().cpu().numpy(), ref["out"], "out after the timeout")


def _small_layer(seed=11, T=8, H=256, E=8, I=128):
    d = random_small_inputs(seed, T, H, E, I, w_std=0.08)
    return d, {n: dev_bf16(d[n]) for n in ("hidden", "router_w", "w_gate_up", "w_down")}


@pytest.mark.parametrize("barrier", [0, 1, 2])
def test_layer_grid_wait_times_out_and_context_survives(barrier):
    k = 2
    d, dw = _small_layer()
    assert mm.mm_poll_device_status() == mm.MM_OK
    t0 = time.perf_counter()
    mm.mm_selftest_layer_barrier_timeout(dw["hidden"], dw["router_w"], dw["w_gate_up"],
                                         dw["w_down"], k, True, barrier)
    rc = mm.mm_poll_device_status()
    dt = time.perf_counter() - t0
    assert rc == mm.MM_ERR_TIMEOUT
    assert 0.9 <= dt < 30.0, dt
    assert mm.mm_poll_device_status() == mm.MM_OK

    out = mm.mm_moe_forward(dw["hidden"], dw["router_w"], dw["w_gate_up"], dw["w_down"], k, True)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    ids, w, _ = O.route(d["hidden"], d["router_w"], k, True, None)
    ref = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
    assert_out_close(out.float().cpu().numpy(), ref, "out after the grid-wide timeout")


def test_layer_grid_wait_selftest_rejects():
    d, dw = _small_layer(H=128)  # H % 256 != 0: not the single-launch path
    with pytest.raises(mm.MMError) as ei:
        mm.mm_selftest_layer_barrier_timeout(dw["hidden"], dw["router_w"], dw["w_gate_up"],
                                             dw["w_down"], 2, True, 0)
    assert ei.value.code == mm.MM_ERR_UNSUPPORTED
    d, dw = _small_layer()
    with pytest.raises(mm.MMError) as ei:
        mm.mm_selftest_layer_barrier_timeout(dw["hidden"], dw["router_w"], dw["w_gate_up"],
                                             dw["w_down"], 2, True, 3)
    assert ei.value.code == mm.MM_ERR_INVALID_ARG
    assert mm.mm_poll_device_status() == mm.MM_OK
