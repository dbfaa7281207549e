"""Tensor-parallel split of the layer, on CPU ("The op layer: BaseOP and the
layers", "Linear layers": gate_up a merged column-parallel linear, down a
row-parallel linear followed by an all-reduce, the router replicated).

Each rank holds the intermediate slice tp_slice gives it; the layer on a
slice is the same loop over experts with I/W intermediates, and the ranks'
unrounded partial outputs summed by one all-reduce equal the whole layer.
Checked with the oracle in float64 on two gloo ranks (the collective bench.py
issues over NCCL on GPUs), and the slicing itself by hand.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mixture_experts_layer_mm_gb300 import tp_slice  # noqa: E402
from mixture_experts_layer_mm_gb300.synthetic import random_small_inputs  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402

T, H, E, K, I = 24, 64, 6, 2, 64


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slices_hold_the_gate_and_up_rows_and_down_columns():
    d = random_small_inputs(3, T, H, E, I)
    for world in (1, 2, 4):
        il = I // world
        for r in range(world):
            gu, dn = tp_slice(d["w_gate_up"], d["w_down"], r, world)
            assert gu.shape == (E, 2 * il, H) and dn.shape == (E, H, il)
            assert np.array_equal(gu[:, :il], d["w_gate_up"][:, r * il:(r + 1) * il])
            assert np.array_equal(gu[:, il:], d["w_gate_up"][:, I + r * il:I + (r + 1) * il])
            assert np.array_equal(dn, d["w_down"][:, :, r * il:(r + 1) * il])
    with pytest.raises(ValueError):
        tp_slice(d["w_gate_up"], d["w_down"], 0, 5)  # 64 does not split into 5


def _rank_main(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    d = random_small_inputs(11, T, H, E, I)  # the same inputs on every rank
    ids, w, _ = O.route(d["hidden"], d["router_w"], K, True)  # the replicated router
    gu, dn = tp_slice(d["w_gate_up"], d["w_down"], rank, ws)
    part = torch.from_numpy(O.experts_loop(d["hidden"], gu, dn, ids, w, dtype=np.float64))
    total = bench.tp_combine(part.clone(), ws)  # the one exchange: a sum over the ranks
    q.put((rank, part.numpy().tobytes(), total.numpy().tobytes()))
    dist.destroy_process_group()


def test_two_gloo_ranks_sum_to_the_whole_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, part, total = q.get(timeout=120)
        got[rank] = (np.frombuffer(part).reshape(T, H), np.frombuffer(total).reshape(T, H))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    d = random_small_inputs(11, T, H, E, I)
    ids, w, _ = O.route(d["hidden"], d["router_w"], K, True)
    whole = O.experts_loop(d["hidden"], d["w_gate_up"], d["w_down"], ids, w, dtype=np.float64)
    for r in (0, 1):
        np.testing.assert_allclose(got[r][1], whole, rtol=1e-12, atol=1e-15)
    # each rank's part is a real share of the output, not all of it
    assert np.abs(got[0][0] - whole).max() > 1e-3 * np.abs(whole).max()
