"""The multi-rank path of bench.py on CPU: two gloo ranks.

The layer shards by tokens with no exchange step, so N GPUs run N replicas
(each its own seeded batch, the same weights); the ranks meet only at the
barrier around the timed region and in the maximum of their times. These
tests run that logic with the gloo backend (no GPU), and launch the
reference arm under torchrun with two ranks, where rank 0 alone works and
prints one line.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    from mixture_experts_layer_mm_gb300 import synthetic as S
    slowest = bench.max_over_ranks(10.0 + rank, ws)  # rank r took 10 + r ms
    bench.barrier(ws)
    # what bench.py hands each replica: its own batch, the layer of the base shape
    q.put((rank, slowest, S.make_hidden(bench.replica_batch(S.TINY, rank)).tobytes(),
           S.make_weights(S.TINY)["w_gate_up"].tobytes()))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict()
    for _ in procs:
        rank, slowest, hid, wgu = q.get(timeout=120)
        got[rank] = (slowest, hid, wgu)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 11.0          # both ranks see the slowest time
    assert got[0][1] != got[1][1]                  # each replica has its own batch
    assert got[0][2] == got[1][2]                  # and the same layer weights


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_tokens_per_s(64, 1, 0.2) == pytest.approx(320000.0)
    assert bench.job_tokens_per_s(64, 4, 0.25) == pytest.approx(4 * 64 / 0.25e-3)


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--workload", "tiny", "--ref-tokens", "4"]
    env = {**os.environ, "OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1"}
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout            # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert np.isfinite(d["ms_per_step"])
