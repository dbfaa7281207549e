"""mm_gated_mlp: the dense SwiGLU MLP ("模型与权重加载", GatedMLP) through the
grouped-GEMM kernels, against the oracle's expert loop with one expert,
top_k = 1 and weight 1 (which the oracle's pins tie to the textbook dense
MLP). When the down GEMM splits K (few tiles for the SMs), its partial sums
reach the fp32 accumulator in no fixed order, so each call is checked
against the oracle on its own."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import random_small_inputs
from oracle import moe_oracle as O
from gpu_util import assert_out_close, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


@pytest.mark.parametrize("T,H,I", [(1, 64, 64), (17, 128, 64), (300, 256, 192), (129, 512, 320),
                                   (1024, 1024, 1536)])
def test_gated_mlp(T, H, I):
    d = random_small_inputs(T + H + I, T, H, 1, I, w_std=0.05)
    wgu, wd = d["w_gate_up"][0], d["w_down"][0]
    out = mm.mm_gated_mlp(dev_bf16(d["hidden"]), dev_bf16(wgu), dev_bf16(wd))
    out2 = mm.mm_gated_mlp(dev_bf16(d["hidden"]), dev_bf16(wgu), dev_bf16(wd))
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    ref = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w)
    assert_out_close(out.float().cpu().numpy(), ref, "dense GatedMLP")
    assert_out_close(out2.float().cpu().numpy(), ref, "dense GatedMLP, second call")


def test_gated_mlp_args():
    z = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    assert mm.mm_gated_mlp(z, w, w.view(64, 128)[:, :64].contiguous()).shape == (0, 64)
    assert mm.mm_gated_mlp_workspace_size(4, 100, 64) == -1
    assert mm.mm_gated_mlp_workspace_size(4, 128, 64) > 0
