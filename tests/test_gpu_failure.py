"""The device-side failure path: a bounded wait that runs out.

Every kernel waits on mbarriers with a time limit (about a second of
%globaltimer); when it runs out the kernel records a timeout in the
per-device status word, unwinds and returns. mm_selftest_wait_timeout runs
one kernel whose wait can never complete (a barrier nothing arrives on),
which is the only way to make the limit run out without breaking a real
kernel. The test checks the reported status, the time it took, and that the
library works normally afterwards.
"""
import time

import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import TINY, make_inputs
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
