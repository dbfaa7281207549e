"""The arithmetic behind bench.py's roofline object, on CPU.

The achieved bandwidth and flop rates divide algorithmic bytes and flops by
measured times, so the counts themselves are checked here against values
worked out by hand for the Qwen3-30B-A3B-shaped layer (H=2048, E=128, k=8,
I=768): 6.29 MB of gate/up weights and 3.15 MB of down weights per selected
expert, 76.0 MFLOP per token for the whole layer.
"""
import dataclasses
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_layer_mm_gb300 import synthetic as S  # noqa: E402


def _all_experts_ids(T, k, E):
    # token t takes experts t*k .. t*k+k-1 (mod E): with T*k >= E every expert appears
    return (np.arange(T * k) % E).reshape(T, k).astype(np.int32)


def test_decode_counts_by_hand():
    sh = S.DECODE                              # T=64, H=2048, E=128, k=8, I=768
    w = bench.algorithmic_work(sh, _all_experts_ids(sh.T, sh.top_k, sh.E))
    assert w["D"] == 128
    gate_up_weights = 128 * (2 * 768) * 2048 * 2          # 805,306,368 B
    # weights of the selected experts + the token rows read once (x) or the
    # output written once (out); the act round trip and the fp32 accumulator
    # are not algorithmic
    assert w["gate_up"]["bytes"] == gate_up_weights + 64 * 2048 * 2
    assert w["gate_up"]["flops"] == 2 * 512 * 2048 * 1536  # 3.22 GFLOP
    down_weights = 128 * 2048 * 768 * 2                   # 402,653,184 B
    assert w["down"]["bytes"] == down_weights + 64 * 2048 * 2
    assert w["down"]["flops"] == 2 * 512 * 768 * 2048
    # per expert: 6.29 MB of gate/up rows, 3.15 MB of down rows
    assert gate_up_weights / 128 == pytest.approx(6.29e6, rel=1e-3)
    assert down_weights / 128 == pytest.approx(3.15e6, rel=2e-3)
    # 76.0 MFLOP per token: router 2*E*H plus three expert projections per slot
    assert w["layer"]["flops"] / sh.T == pytest.approx(76.02e6, rel=1e-4)
    # the layer's bytes: every selected expert's three matrices, the router, x and out
    assert w["layer"]["bytes"] == 128 * 3 * 2048 * 768 * 2 + 128 * 2048 * 2 + 2 * 64 * 2048 * 2


def test_distinct_experts_follow_the_routing():
    sh = S.DECODE
    ids = np.tile(np.array([3, 9, 77, 3, 9, 77, 3, 9], dtype=np.int32), (sh.T, 1))
    w = bench.algorithmic_work(sh, ids)
    assert w["D"] == 3
    assert w["gate_up"]["bytes"] == 3 * 1536 * 2048 * 2 + 64 * 2048 * 2


def test_roofline_axis_follows_the_regime():
    # Decode streams the selected experts' weights: bytes / time against the
    # HBM peak. Prefill (T*k > 64*E rows) is measured as flops / time against
    # the bf16 peak, although its gate_up intensity (251 flop per
    # algorithmic byte) is just under the measured ridge (~283 flop/B).
    assert not bench.tensor_regime(S.DECODE)
    assert bench.tensor_regime(S.PREFILL) and bench.tensor_regime(S.LARGE)
    assert not bench.tensor_regime(S.SWEEP.with_T(512))
    assert bench.tensor_regime(S.SWEEP.with_T(2048))
    sh = S.PREFILL
    w = bench.algorithmic_work(sh, _all_experts_ids(sh.T, sh.top_k, sh.E))
    intensity = w["gate_up"]["flops"] / w["gate_up"]["bytes"]
    assert intensity == pytest.approx(206.16e9 / (805.31e6 + 16.78e6), rel=1e-3)
    pk = {"hbm_gbs": 6793.4, "bf16_tflops": 1924.4}
    stage = {"gate_up": 0.2, "down": 0.1}
    roof = bench.roofline(sh, w, stage, 0.4, pk, "measured")
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["achieved"] == pytest.approx(w["gate_up"]["flops"] / 0.2e-3 / 1e12)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1924.4)
    assert roof["layer"]["flops_frac_bf16"] == pytest.approx(
        w["layer"]["flops"] / 0.4e-3 / 1e12 / 1924.4)
    roof_d = bench.roofline(S.DECODE, bench.algorithmic_work(S.DECODE, _all_experts_ids(64, 8, 128)),
                            stage, 0.2, pk, "measured")
    assert roof_d["bound"] == "hbm" and roof_d["unit"] == "GB/s"


def test_kernel_launches_follow_the_launch_sequence():
    # decode (T=64): route with the grouping fused, gate_up, down, finalize;
    # up to 16 tokens: the single-launch layer; prefill (T=4096): tensor-core
    # route, grouping + row copy, gate_up, down, finalize (the kernels an ncu
    # launch list shows per pass)
    assert bench.kernel_launches(S.DECODE) == 4
    assert bench.kernel_launches(S.SWEEP.with_T(1)) == 1
    assert bench.kernel_launches(S.SWEEP.with_T(8)) == 1
    assert bench.kernel_launches(S.SWEEP.with_T(32)) == 4
    assert bench.kernel_launches(S.PREFILL) == 5
    assert bench.kernel_launches(S.LARGE) == 5
    assert bench.kernel_launches(S.DECODE, add_norm=True) == 5
    assert bench.kernel_launches(S.SWEEP.with_T(8), add_norm=True) == 2
    # shapes the single launch does not take (H % 256 != 0) use the chain
    assert bench.kernel_launches(dataclasses.replace(S.SWEEP, T=8, H=192)) == 4
    # one-block grouping; count + place + a separate row copy; E % 4 != 0
    assert bench.kernel_launches(S.SWEEP.with_T(512)) == 5
    assert bench.kernel_launches(S.SWEEP.with_T(2048)) == 7
    odd_e = dataclasses.replace(S.PREFILL, E=30, top_k=4)
    assert bench.kernel_launches(odd_e) == 6


def test_flush_overwrites_the_scratch_buffer():
    # The flush between small steps writes the whole buffer and reads it back
    # (here on a CPU tensor: the same torch calls the GPU run makes).
    torch = pytest.importorskip("torch")
    scratch = torch.full((1024,), 7.0)
    bench.flush_l2(scratch)
    assert torch.count_nonzero(scratch).item() == 0
