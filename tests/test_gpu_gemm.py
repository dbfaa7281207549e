"""GPU parity of the two grouped GEMMs (mm_grouped_gemm) against oracle
arithmetic, on shapes that span several tiles with ragged tails: token chunks
of 1..128 rows, partial weight m-tiles, several K blocks, empty experts."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import f32_to_bf16_bits, random_small_inputs
from oracle import moe_oracle as O
from gpu_util import assert_out_close, dev_bf16, f32_dev, i32_dev

pytestmark = pytest.mark.gpu

BM = mm.FORWARD_BLOCK_M


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


def _routing(T, E, k, seed, skew=False):
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E))
    if skew:
        keys += np.linspace(0, 2, E)[None, :]   # uneven load, some experts empty
    ids = np.sort(np.argsort(-keys, axis=1)[:, :k], axis=1).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return ids, w


CASES = [  # T, H, E, k, I, skew
    (16, 128, 8, 2, 64, False),
    (300, 256, 8, 2, 192, False),
    (1000, 320, 4, 2, 128, False),
    (64, 2048, 128, 8, 768, False),
    (700, 512, 16, 3, 320, True),
    (1, 64, 3, 1, 64, False),
]


@pytest.mark.parametrize("T,H,E,k,I,skew", CASES)
def test_gate_up(T, H, E, k, I, skew):
    d = random_small_inputs(T + H, T, H, E, I)
    ids, _ = _routing(T, E, k, T, skew)
    s, off, cnt = O.align(ids, E, BM)
    cap = s.size
    act = torch.full((cap, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    mm.mm_grouped_gemm(mm.MM_GEMM_GATE_UP, dev_bf16(d["hidden"]), dev_bf16(d["w_gate_up"]), act,
                       i32_dev(s), i32_dev(off), None, T, k, BM)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    act = act.float().cpu().numpy()
    x = O.widen_bf16(d["hidden"])
    rows, ref = [], []
    for e in range(E):
        seg = s[off[e]:off[e + 1]]
        real = np.nonzero(seg < T * k)[0]
        if real.size == 0:
            continue
        wg = O.widen_bf16(d["w_gate_up"][e])
        xe = x[seg[real] // k]
        rows.extend((off[e] + real).tolist())
        ref.append(O.silu_and_mul(xe @ wg[:I].T, xe @ wg[I:].T))
    ref = np.concatenate(ref)
    rows = np.array(rows)
    assert_out_close(act[rows], ref, "act")


@pytest.mark.parametrize("T,H,E,k,I,skew", CASES)
def test_down(T, H, E, k, I, skew):
    d = random_small_inputs(T + 2 * H, T, H, E, I)
    ids, w = _routing(T, E, k, T + 1, skew)
    s, off, cnt = O.align(ids, E, BM)
    cap = s.size
    rng = np.random.default_rng(3)
    act_bits = f32_to_bf16_bits(rng.standard_normal((cap, I)).astype(np.float32))
    acc = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    mm.mm_grouped_gemm(mm.MM_GEMM_DOWN, dev_bf16(act_bits), dev_bf16(d["w_down"]), acc,
                       i32_dev(s), i32_dev(off), f32_dev(w.reshape(-1)), T, k, BM)
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    a = O.widen_bf16(act_bits)
    ref = np.zeros((T, H), dtype=np.float64)
    wf = w.reshape(-1)
    for e in range(E):
        wd = O.widen_bf16(d["w_down"][e]).astype(np.float64)
        for r in range(off[e], off[e + 1]):
            f = s[r]
            if f < T * k:
                ref[f // k] += wf[f] * (a[r].astype(np.float64) @ wd.T)
    assert_out_close(acc.cpu().numpy(), ref, "acc", max_rel=1e-4, mean_rel=1e-5)

