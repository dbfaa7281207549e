"""Guard regions around every buffer a call reads or writes.

A memory checker is not available here, so each buffer handed to the
library is the middle of a larger allocation whose head and tail hold a
fixed byte pattern. After the call and a device synchronisation the pattern
must be intact: no kernel may write outside the outputs (or the caller
workspace) it is given, nor into its inputs' neighbourhood. The shapes take
the different launch sequences of the layer: the router with the fused
grouping (T <= 64), the one-block grouping, and the tensor-core router whose
grouping also copies the token rows (T > 2048), plus the dense MLP and the
add + RMSNorm step.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_mm_gb300 as mm
from mixture_experts_layer_mm_gb300.synthetic import random_small_inputs

pytestmark = pytest.mark.gpu
GUARD = 4096    # bytes on each side; keeps the middle 16-byte (and 256-byte) aligned
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib(mmlib):
    return mmlib


class Guarded:
    """A tensor of `shape` and `dtype` inside guard bytes."""

    def __init__(self, shape, dtype, fill=None):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        self.n = int(np.prod(shape)) * itemsize
        self.raw = torch.full((GUARD + self.n + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw[GUARD:GUARD + self.n].view(dtype).view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self) -> bool:
        return bool((self.raw[:GUARD] == PATTERN).all()) and \
            bool((self.raw[GUARD + self.n:] == PATTERN).all())


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _check_all(*bufs):
    torch.cuda.synchronize()
    assert mm.mm_poll_device_status() == mm.MM_OK
    for name, g in bufs:
        assert g.intact(), f"guard bytes around {name} were overwritten"


@pytest.mark.parametrize("T,H,E,k,I", [
    (16, 128, 8, 2, 64),       # router + fused grouping, gathered token rows
    (129, 256, 40, 5, 192),    # one-block grouping, ragged m-tiles
    (64, 256, 32, 8, 128),     # 64-token GEMM tiles, gather4
    (3000, 64, 100, 8, 64),    # tensor-core router, grouping + row copy, 128-token tiles
])
def test_forward_writes_only_its_outputs(T, H, E, k, I):
    d = random_small_inputs(T + E, T, H, E, I, w_std=0.08)
    hid = Guarded((T, H), torch.bfloat16, _bf16(d["hidden"]))
    rw = Guarded((E, H), torch.bfloat16, _bf16(d["router_w"]))
    wgu = Guarded((E, 2 * I, H), torch.bfloat16, _bf16(d["w_gate_up"]))
    wdn = Guarded((E, H, I), torch.bfloat16, _bf16(d["w_down"]))
    out = Guarded((T, H), torch.bfloat16)
    ws = Guarded((mm.mm_moe_workspace_size(T, H, E, I, k),), torch.uint8)
    mm.mm_moe_forward(hid.t, rw.t, wgu.t, wdn.t, k, True, out=out.t, workspace=ws.t)
    _check_all(("hidden", hid), ("router_w", rw), ("w_gate_up", wgu), ("w_down", wdn),
               ("out", out), ("workspace", ws))
    assert torch.isfinite(out.t.float()).all()


@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (3000, 100, 8)])
def test_route_and_align_write_only_their_outputs(T, E, k):
    H = 128
    d = random_small_inputs(7, T, H, E, 64, w_std=0.08)
    hid = Guarded((T, H), torch.bfloat16, _bf16(d["hidden"]))
    rw = Guarded((E, H), torch.bfloat16, _bf16(d["router_w"]))
    ids = Guarded((T, k), torch.int32)
    w = Guarded((T, k), torch.float32)
    mm.mm_route(hid.t, rw.t, k, True, topk_ids=ids.t, topk_w=w.t)
    block_m = 16
    cap = mm.mm_align_capacity(T, k, E, block_m)
    srt = Guarded((cap,), torch.int32)
    off = Guarded((E + 1,), torch.int32)
    cnt = Guarded((E,), torch.int32)
    mm.mm_align(ids.t, E, block_m, sorted_token_ids=srt.t, expert_offsets=off.t,
                expert_counts=cnt.t)
    _check_all(("hidden", hid), ("router_w", rw), ("topk_ids", ids), ("topk_w", w),
               ("sorted_token_ids", srt), ("expert_offsets", off), ("expert_counts", cnt))
    assert int(cnt.t.sum()) == T * k


def test_dense_mlp_and_norm_write_only_their_outputs():
    T, H, I = 64, 128, 256
    rng = np.random.default_rng(3)
    x = Guarded((T, H), torch.bfloat16,
                torch.from_numpy(rng.standard_normal((T, H), dtype=np.float32)).to(torch.bfloat16))
    wgu = Guarded((2 * I, H), torch.bfloat16,
                  (0.05 * torch.from_numpy(rng.standard_normal((2 * I, H), dtype=np.float32)))
                  .to(torch.bfloat16))
    wdn = Guarded((H, I), torch.bfloat16,
                  (0.05 * torch.from_numpy(rng.standard_normal((H, I), dtype=np.float32)))
                  .to(torch.bfloat16))
    out = Guarded((T, H), torch.bfloat16)
    mm.mm_gated_mlp(x.t, wgu.t, wdn.t, out=out.t)
    nw = Guarded((H,), torch.bfloat16, torch.ones(H, dtype=torch.bfloat16))
    res = Guarded((T, H), torch.bfloat16, torch.zeros(T, H, dtype=torch.bfloat16))
    normed = Guarded((T, H), torch.bfloat16)
    mm.mm_add_rmsnorm(x.t, nw.t, 1e-6, residual=res.t, normed=normed.t)
    _check_all(("x", x), ("w_gate_up", wgu), ("w_down", wdn), ("out", out), ("norm_w", nw),
               ("residual", res), ("normed", normed))
    assert torch.equal(res.t, x.t)  # residual' = x + 0


@pytest.mark.parametrize("T,H,E,k,I", [(64, 256, 32, 8, 128), (3000, 64, 100, 8, 64)])
def test_moe_block_with_residual_adds_writes_only_its_outputs(T, H, E, k, I):
    # The add + RMSNorm step, the layer (SM-pair GEMMs for the 3000-token
    # batch) and the add after it, which the down GEMM performs.
    d = random_small_inputs(T + 3 * E, T, H, E, I, w_std=0.08)
    x = Guarded((T, H), torch.bfloat16, _bf16(d["hidden"]))
    res = Guarded((T, H), torch.bfloat16, 0.5 * _bf16(d["hidden"]).flip(0))
    nw = Guarded((H,), torch.bfloat16, torch.ones(H, dtype=torch.bfloat16))
    rw = Guarded((E, H), torch.bfloat16, _bf16(d["router_w"]))
    wgu = Guarded((E, 2 * I, H), torch.bfloat16, _bf16(d["w_gate_up"]))
    wdn = Guarded((E, H, I), torch.bfloat16, _bf16(d["w_down"]))
    out = Guarded((T, H), torch.bfloat16)
    r2 = Guarded((T, H), torch.bfloat16)
    mm.mm_moe_forward_add_norm_residual(x.t, nw.t, 1e-6, rw.t, wgu.t, wdn.t, k, True,
                                        residual=res.t, residual_out=r2.t, out=out.t)
    _check_all(("x", x), ("residual", res), ("norm_w", nw), ("router_w", rw),
               ("w_gate_up", wgu), ("w_down", wdn), ("out", out), ("residual_out", r2))
    assert torch.isfinite(out.t.float()).all() and torch.isfinite(r2.t.float()).all()
