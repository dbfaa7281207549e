"""Throughput of the fused MoE layer on GB300, one JSON line per run.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mm|reference]
                    [--workload decode_qwen3_30b_a3b|prefill_qwen3_30b_a3b|...]

A step is one pass of the whole layer (route, align, gate_up GEMM + SiLU*up,
down GEMM + weighted scatter-add, rounding) over one synthetic batch.
The default workload is the Qwen3-30B-A3B-shaped decode layer (T=64, H=2048,
E=128, k=8, I=768): every step streams the selected experts' weights (about
1.2 GB, far above the 129 MB L2) from HBM, so no L2 flush is needed. Batches
whose step reads less than twice the L2 size (--sweep-T 1) are timed step by
step, with the L2 flushed between steps (a write and a read of twice its
size) outside the timed events.

The line's value, roofline and e2e are the decode layer's (fraction of the
HBM copy peak). The same run also times the prefill layer of the same model
(T=4096) and reports it in the line's prefill_qwen3_30b_a3b object, as
flops / time against the bf16 tensor peak for the layer, gate_up and down.
One NVML sampler covers every timed region of the run.

--tp splits one layer over the ranks instead (tensor parallelism: each rank
a slice of the experts' intermediates, one fp32 all-reduce per step).

--impl reference times the CPU oracle on the host cores instead (a baseline,
not a target). Under torchrun every rank runs its own replica (the layer
shards by tokens with no exchange), and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
_CORES = os.cpu_count() or 1
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_layer_mm_gb300 import synthetic  # noqa: E402

METRIC = "MoE-layer tokens/s (Qwen3-30B-A3B shape) + % of BF16 TC / HBM roofline"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# The sources of each dominant kernel family: the single-CTA grouped GEMM
# (decode-shaped batches), the SM-pair grouped GEMM (prefill-shaped ones) and
# the single-launch layer (batches of at most 16 tokens).
_CSRC = "mixture_experts_layer_mm_gb300/csrc/"
KERNEL_SOURCES = {"gemm": [_CSRC + "gemm.cu", _CSRC + "mm_device.cuh"],
                  "pair": [_CSRC + "gemm_pair.cu", _CSRC + "mm_device.cuh"],
                  "single": [_CSRC + "decode.cu", _CSRC + "mm_device.cuh",
                             _CSRC + "route_finish.cuh"]}


def flush_l2(scratch):
    """Evicts the previous step's data from L2: a write of the scratch buffer
    (twice the L2 size), then a read of it. The write alone left part of the
    previous step in L2 on GB300 (a small batch ran ~6 us faster after it
    than after a read of the same size, with 2x and 4x L2 writes alike)."""
    scratch.zero_()
    scratch.sum()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def kernel_source_hash(family: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def kernel_family(shape) -> str:
    """The kernel family that runs this shape's dominant step."""
    if decode_fused(shape):
        return "single"
    return "pair" if tensor_regime(shape) else "gemm"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Replicas: each rank runs the whole layer on its own batch (tokens are
# independent units; the layer has no exchange step), so the only
# cross-rank traffic is the barrier around the timed region and the maximum
# of the per-rank times. These helpers work with the nccl (GPU) and gloo
# (CPU) process groups alike.

def replica_batch(shape, rank: int):
    """The shape whose seeded hidden batch rank `rank` times. The weights are
    drawn from the unmodified shape, so every replica holds the same layer."""
    return synthetic.MoEShape(**{**shape.__dict__, "seed": rank})


def barrier(ws: int) -> None:
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tp_combine(partial, ws: int):
    """The one exchange step of the tensor-parallel split: the ranks' fp32
    partial outputs summed over all ranks (in place; nccl on GPUs, gloo on
    CPU)."""
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(partial, op=dist.ReduceOp.SUM)
    return partial


def job_tokens_per_s(T: int, ws: int, ms: float) -> float:
    """Whole-job throughput: the tokens of all replicas over the slowest
    rank's time per step."""
    return T * ws / (ms * 1e-3)


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, read through
    NVML every 10 ms on a background thread while the timed region runs.
    Read-only queries; nothing about the GPU is changed."""
    # nvmlClocksEventReasons bits
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        import threading
        self.index = index
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            self._nvml, self._h, self._ct = lib, h, ctypes
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
                self.max_mhz = float(mx.value)
        except OSError:
            self._nvml = None

    def _run(self):
        ct, lib, h = self._ct, self._nvml, self._h
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0 and \
                    get_reasons(h, ct.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            self._stop.wait(0.01)

    def __enter__(self):
        import threading
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable" if self._nvml is None else "nvml"}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml, 10 ms"}


def algorithmic_work(shape, ids: np.ndarray):
    """Algorithmic bytes / flops of the layer and of its two GEMM kernels for
    one step, from the realised routing. Only what the layer has to move
    counts: each selected expert's weights once, the token rows read once and
    the output written once. Padding, re-reads, gathers, the act round trip
    between the GEMMs and the fp32 accumulator traffic are excluded."""
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.top_k, shape.I
    D = int(np.unique(ids).size)          # distinct experts selected in the batch
    M = T * k                             # real (token, expert) rows
    gu_bytes = D * 2 * I * H * 2 + T * H * 2     # gate/up rows of the selected experts + x
    dn_bytes = D * H * I * 2 + T * H * 2         # down rows of the selected experts + out
    layer_bytes = D * 3 * H * I * 2 + E * H * 2 + 2 * T * H * 2
    return {"D": D,
            "gate_up": {"bytes": gu_bytes, "flops": 2 * M * H * 2 * I},
            "down": {"bytes": dn_bytes, "flops": 2 * M * I * H},
            "layer": {"bytes": layer_bytes, "flops": 2 * T * E * H + 2 * M * 3 * H * I}}


def tensor_regime(shape) -> bool:
    """Whether the roofline fraction is taken against the bf16 tensor peak
    (flops / time) rather than the HBM peak (bytes / time): batches with more
    than 64 rows per expert on average (T*k > 64*E), where the GEMMs read
    their token rows in segment order and reuse every weight tile across
    many tokens (prefill, the large config, the sweep from T = 2048). Below
    that the layer streams the selected experts' weights (decode)."""
    return shape.T * shape.top_k > 64 * shape.E


def decode_fused(shape) -> bool:
    """Whether mm_moe_forward runs this shape's layer as its single
    cooperative launch (batches of at most 16 tokens whose shape that launch
    takes: T*k <= 512, E <= 256, H % 256 == 0 and H <= 2048, I % 128 == 0 and
    I <= 1024)."""
    return (1 <= shape.T <= 16 and shape.T * shape.top_k <= 512 and shape.E <= 256
            and shape.H % 256 == 0 and shape.H <= 2048 and shape.I % 128 == 0 and shape.I <= 1024)


def kernel_launches(shape, add_norm: bool = False) -> int:
    """Kernels one layer call launches for this shape (the launch sequence of
    the library's forward): route (which also groups when T <= 64), the
    grouping (one block up to 1024 tokens; count + place beyond; place alone
    from the tensor-core router's tile counts above 2048 tokens with E <= 128),
    the row copy into segment order when T*k > 64*E (inside the place launch
    when it runs from tile counts and E % 4 == 0), gate_up, down, finalize
    (which also adds the residual after the layer in the add-norm mode); plus
    the add + RMSNorm kernel in front when add_norm."""
    T, E, k = shape.T, shape.E, shape.top_k
    if decode_fused(shape):  # one launch for the whole layer
        return 1 + (1 if add_norm else 0)
    fused_align = T <= 64 and T * k <= 8192
    single_align = T <= 1024 and T * k <= 8192
    router_counts = T > 2048 and E <= 128
    rows_gathered = T * k > 64 * E
    separate_copy = rows_gathered and not (router_counts and E % 4 == 0)
    grouping = 0 if fused_align else 1 if (single_align or router_counts) else 2
    return 4 + grouping + (1 if separate_copy else 0) + (1 if add_norm else 0)


def load_traffic(workload: str, kernel: str, family: str):
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE))
    ent = d.get(workload, {}).get(kernel)
    if not ent or ent.get("family") != family or ent.get("source_hash") != kernel_source_hash(family):
        return None  # counters were taken on another version of the kernel
    return ent.get("bytes_per_launch")


def run_reference(args, shape, ws, rank):
    """The CPU oracle on the host cores, on a bounded sample of the workload."""
    if rank != 0:
        return
    from oracle import moe_oracle as O
    d = synthetic.make_inputs(shape)
    n_tok = min(shape.T, args.ref_tokens)
    sub = dict(d)
    sub["hidden"] = d["hidden"][:n_tok]

    def step():
        O.moe_layer(sub, shape.top_k, shape.renorm)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    v = n_tok * args.steps / dt
    sample = (f"first {n_tok} of the {shape.T} tokens of {shape.name} per step, "
              f"full routing + grouping + fp32 expert loop")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": shape.name, "T": shape.T, "H": shape.H, "E": shape.E,
                       "top_k": shape.top_k, "I": shape.I, "renorm": shape.renorm,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(shape, budget_s: float):
    """Times the oracle as it stands on a bounded sample (about budget_s)."""
    from oracle import moe_oracle as O
    d = synthetic.make_inputs(shape)
    n_tok = min(shape.T, 64)
    sub = dict(d)
    sub["hidden"] = d["hidden"][:n_tok]
    t0 = time.perf_counter()
    O.moe_layer(sub, shape.top_k, shape.renorm)
    one = time.perf_counter() - t0
    reps = max(1, min(20, int(budget_s / max(one, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(reps):
        O.moe_layer(sub, shape.top_k, shape.renorm)
    dt = time.perf_counter() - t0
    return {"value": n_tok * reps / dt, "unit": UNIT, "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle",
            "sample": f"{reps} oracle passes over the first {n_tok} tokens of {shape.name} "
                      f"({dt:.1f} s, numpy fp32 with OpenBLAS threads)"}


def run_dense(args, shape, ws, rank, dev, mm):
    """Times mm_gated_mlp on the workload's T tokens: a dense SwiGLU MLP with
    hidden H and intermediate k*I, the flops per token of the MoE layer's
    experts. Same timing rules as the layer (warm-up, events, NVML clocks,
    max over ranks); the roofline is taken over the whole call."""
    T, H, I = shape.T, shape.H, shape.top_k * shape.I
    w = synthetic.make_dense_weights(0, H, I)
    x_np = synthetic.make_hidden(synthetic.MoEShape(**{**shape.__dict__, "seed": rank}))

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    x, wgu, wdn = to_dev(x_np), to_dev(w["w_gate_up"]), to_dev(w["w_down"])
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd = lambda: mm.mm_gated_mlp(x, wgu, wdn, out=out)  # noqa: E731
    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    if args.steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            fwd()
        e1.record(stream)
        torch.cuda.synchronize()
        args.steps = int(min(5000, max(20, 600.0 / max(e0.elapsed_time(e1) / 5, 1e-3))))
    flops = 2 * T * H * 2 * I + 2 * T * I * H
    nbytes = 3 * H * I * 2 + 2 * T * H * 2
    # The weights (75 MB at H=2048, I=6144) fit in L2: a step whose bytes are
    # under twice the L2 size is timed alone, after the L2 is flushed (a write
    # and a read of twice its size) outside its events, as in the layer's timing.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = nbytes < 2 * l2_bytes
    scratch = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev) if flush else None
    barrier(ws)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        if flush:
            step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.steps)]
            for a, b in step_ev:
                flush_l2(scratch)
                a.record(stream)
                fwd()
                b.record(stream)
        else:
            t_start.record(stream)
            for _ in range(args.steps):
                fwd()
            t_end.record(stream)
        torch.cuda.synchronize()
    if flush:
        ms = sum(a.elapsed_time(b) for a, b in step_ev) / args.steps
    else:
        ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms, ws, dev)

    # End to end: x from pinned host memory, the call, out back to the host.
    x_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    o_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    x_dev = torch.empty_like(x)
    barrier(ws)
    torch.cuda.synchronize()
    e2e_total = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        if flush:  # the flush is kept out of the step's wall time
            flush_l2(scratch)
            stream.synchronize()
            t0 = time.perf_counter()
        x_dev.copy_(x_host, non_blocking=True)
        mm.mm_gated_mlp(x_dev, wgu, wdn, out=out)
        o_host.copy_(out, non_blocking=True)
        stream.synchronize()
        if flush:
            e2e_total += time.perf_counter() - t0
    if not flush:
        e2e_total = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_total / args.steps, ws, dev)
    st = mm.mm_poll_device_status()
    if st != mm.MM_OK:
        raise RuntimeError(f"device status after the timed region: {mm.status_string(st)}")
    pk, pk_kind = peaks()
    tensor = flops / nbytes > pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if tensor:
        ach = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "peak_kind": f"{pk_kind} bf16_tflops (burst)"}
    else:
        ach = nbytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"], "peak_kind": f"{pk_kind} hbm_gbs (copy bandwidth)"}
    roof["kernel"] = "mm_gated_mlp, whole call (grouping, gate_up, down, finalize)"
    roof["traffic"] = None
    line = {"metric": "dense SwiGLU MLP tokens/s", "value": T * ws / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normals, bf16)",
            "config": {"workload": f"dense_gated_mlp_T{T}_H{H}_I{I}", "T": T, "H": H, "I": I,
                       "parallelism": f"replicas x{ws}",
                       "l2": (f"L2 flushed between steps (a {2 * l2_bytes / 1e6:.0f} MB write and "
                              f"read outside each step's events): the {3 * H * I * 2 / 1e6:.0f} MB "
                              "of weights fit in L2") if flush else
                             f"weights {3 * H * I * 2 / 1e6:.0f} MB per step, inputs larger than L2"},
            "roofline": roof,
            "e2e": {"value": T * ws / e2e_s, "unit": "tokens/s",
                    "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2},
            "gpu_launches": 4 * args.steps, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def roofline(shape, work, stage_ms, ms, pk, pk_kind):
    """The roofline object of the dominant kernel (the gate_up grouped GEMM:
    the largest share of both bytes and flops), and of the whole layer.
    Decode-shaped batches are measured as algorithmic bytes / time against
    the HBM copy peak, prefill-shaped ones (tensor_regime) as flops / time
    against the bf16 burst peak; both fractions are in the object."""
    dom = "gate_up"
    dom_ms = stage_ms[dom]
    if decode_fused(shape):
        # the single-launch layer: its one kernel moves all of the layer's
        # bytes (its time is reported as the gate_up stage)
        dom = "layer"
    bw = work[dom]["bytes"] / (dom_ms * 1e-3) / 1e9
    tf = work[dom]["flops"] / (dom_ms * 1e-3) / 1e12
    if tensor_regime(shape):
        roof = {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"],
                "peak_kind": f"{pk_kind} bf16_tflops (burst)"}
    else:
        roof = {"bound": "hbm", "achieved": bw, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": bw / pk["hbm_gbs"], "peak_kind": f"{pk_kind} hbm_gbs (copy bandwidth)"}
    roof["frac_hbm"] = bw / pk["hbm_gbs"]
    roof["frac_tensor"] = tf / pk["bf16_tflops"]
    roof["intensity_flop_per_byte"] = work[dom]["flops"] / work[dom]["bytes"]
    fam = kernel_family(shape)
    kname = {"single": "moe_decode_kernel, whole layer", "pair": "grouped_gemm_pair_kernel<gate_up>",
             "gemm": "grouped_gemm_kernel<gate_up>"}[fam]
    roof["kernel"] = f"{kname} ({dom_ms * 1e3:.1f} us/launch, CUDA events)"
    roof["traffic"] = load_traffic(shape.name, dom, fam)
    dn_ms = stage_ms["down"]
    roof["down"] = {"frac_hbm": work["down"]["bytes"] / (dn_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "frac_tensor": work["down"]["flops"] / (dn_ms * 1e-3) / 1e12 /
                    pk["bf16_tflops"], "us_per_launch": dn_ms * 1e3}
    roof["layer"] = {"bytes_frac_hbm": work["layer"]["bytes"] / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "flops_frac_bf16": work["layer"]["flops"] / (ms * 1e-3) / 1e12 /
                     pk["bf16_tflops"]}
    return roof


class LayerRun:
    """One workload's device inputs and the three timed regions of bench.py:
    A the layer as a user calls it (device-resident inputs), B the same
    steps with stage events around each kernel, C end to end from pinned
    host memory through the C ABI."""

    def __init__(self, mm, shape, dev, weights, bias, rank, add_norm=False, eps=1e-6):
        self.mm, self.shape, self.dev = mm, shape, dev
        self.router_w, self.w_gu, self.w_dn = weights
        self.bias = bias
        self.add_norm, self.eps = add_norm, eps
        self.stream = torch.cuda.current_stream(dev)
        self.hidden = _to_dev(synthetic.make_hidden(replica_batch(shape, rank)), dev)
        self.out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev)
        if add_norm:  # x, the residual stream and the norm weight of the step before
            nrm = synthetic.make_norm_inputs(rank, shape.T, shape.H)
            self.x, self.res = _to_dev(nrm["x"], dev), _to_dev(nrm["residual"], dev)
            self.norm_w = _to_dev(nrm["norm_w"], dev)

    def fwd(self, hidden=None):
        mm, sh = self.mm, self.shape
        if self.add_norm:  # both residual adds; the residual stream is updated in place
            mm.mm_moe_forward_add_norm_residual(self.x if hidden is None else hidden, self.norm_w,
                                                self.eps, self.router_w, self.w_gu, self.w_dn,
                                                sh.top_k, sh.renorm, residual=self.res,
                                                out=self.out)
        else:
            mm.mm_moe_forward(self.hidden if hidden is None else hidden, self.router_w,
                              self.w_gu, self.w_dn, sh.top_k, sh.renorm, out=self.out,
                              router_bias=self.bias)

    def warmup(self, n):
        for _ in range(n):
            self.fwd()
        torch.cuda.synchronize()

    def auto_steps(self, seconds=0.6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(5):
            self.fwd()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return int(min(5000, max(20, seconds * 1e3 / max(e0.elapsed_time(e1) / 5, 1e-3))))

    def work(self):
        sh = self.shape
        ids, _ = self.mm.mm_route(self.hidden, self.router_w, sh.top_k, sh.renorm,
                                  router_bias=self.bias)
        return algorithmic_work(sh, ids.cpu().numpy())

    def measure(self, steps, ws, flush_bytes, l2_bytes, e2e=True):
        """Runs regions A, B (and C); returns ms per step, stage ms, e2e s per step."""
        mm, stream, dev = self.mm, self.stream, self.dev
        # A step whose bytes would stay in L2 is timed alone, after a write and
        # a read of twice the L2 size (outside its events) evict the previous
        # step's data.
        flush = flush_bytes < 2 * l2_bytes
        scratch = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev) if flush else None
        self.flushed = flush
        # ---- region A
        barrier(ws)
        torch.cuda.synchronize()
        if flush:
            step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(steps)]
            for a, b in step_ev:
                flush_l2(scratch)
                a.record(stream)
                self.fwd()
                b.record(stream)
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in step_ev) / steps
            # the same steps back to back (warm L2: the weights stay), reported
            # beside the cold headline
            t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for _ in range(steps):
                self.fwd()
            t_end.record(stream)
            torch.cuda.synchronize()
            self.warm_ms = max_over_ranks(t_start.elapsed_time(t_end) / steps, ws, dev)
        else:
            t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for _ in range(steps):
                self.fwd()
            t_end.record(stream)
            torch.cuda.synchronize()
            ms = t_start.elapsed_time(t_end) / steps
        barrier(ws)
        ms = max_over_ranks(ms, ws, dev)
        # ---- region B: stage events (the layer itself, without the norm step)
        sh = self.shape
        nb = min(steps, 200)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(mm.PROFILE_STAGES) + 1)]
               for _ in range(nb)]
        barrier(ws)
        torch.cuda.synchronize()
        for i in range(nb):
            if flush:
                flush_l2(scratch)  # before the call's first event
            mm.mm_moe_forward_profiled(self.hidden, self.router_w, self.w_gu, self.w_dn, sh.top_k,
                                       sh.renorm, evs[i], out=self.out, router_bias=self.bias)
        torch.cuda.synchronize()
        barrier(ws)
        stage_ms = {name: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1])
                                          for i in range(nb))
                    for j, name in enumerate(mm.PROFILE_STAGES)}
        e2e_s = None
        if e2e:
            e2e_s = self._measure_e2e(steps, ws, flush, scratch)
        st = mm.mm_poll_device_status()
        if st != mm.MM_OK:
            raise RuntimeError(f"device status after the timed regions: {mm.status_string(st)}")
        return ms, stage_ms, e2e_s

    def _measure_e2e(self, steps, ws, flush, scratch):
        # ---- region C: pinned host -> device, the call, device -> host
        stream, sh = self.stream, self.shape
        src = self.x if self.add_norm else self.hidden
        h_host = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, pin_memory=True)
        h_host.copy_(src.cpu())
        o_host = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, pin_memory=True)
        h_dev = torch.empty_like(src)
        if self.add_norm:  # the step's inputs are x and the residual; outputs out and residual
            r_host = torch.empty_like(h_host, pin_memory=True)
            r_host.copy_(self.res.cpu())
            r_back = torch.empty_like(h_host, pin_memory=True)
        self.io_bytes = sh.T * sh.H * 2 * (2 if self.add_norm else 1)
        barrier(ws)
        torch.cuda.synchronize()
        total = 0.0
        t0 = time.perf_counter()
        for _ in range(steps):
            if flush:  # the flush is kept out of the step's wall time
                flush_l2(scratch)
                stream.synchronize()
                t0 = time.perf_counter()
            h_dev.copy_(h_host, non_blocking=True)
            if self.add_norm:
                self.res.copy_(r_host, non_blocking=True)
            self.fwd(h_dev)
            if self.add_norm:
                r_back.copy_(self.res, non_blocking=True)
            o_host.copy_(self.out, non_blocking=True)
            stream.synchronize()
            if flush:
                total += time.perf_counter() - t0
        if not flush:
            total = time.perf_counter() - t0
        return max_over_ranks(total / steps, ws, self.dev)


def _to_dev(bits, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


def run_tp(args, shape, ws, rank, dev, mm):
    """Tensor-parallel split of one layer over the ws ranks ("The op layer:
    BaseOP and the layers", "Linear layers"): every rank routes the same
    batch with the replicated router and runs the experts on its slice of
    the intermediates (mm_moe_forward_partial), one all-reduce sums the fp32
    partials (tp_combine, nccl), and mm_round_bf16 rounds the sum. A step is
    the whole layer on the batch, so the job's tokens/s is T / step time
    (strong scaling: the work is split, not repeated)."""
    w = synthetic.make_weights(shape)
    gu_np, dn_np = mm.tp_slice(w["w_gate_up"], w["w_down"], rank, ws)
    router_w, gu, dn = _to_dev(w["router_w"], dev), _to_dev(gu_np, dev), _to_dev(dn_np, dev)
    del w, gu_np, dn_np
    hidden = _to_dev(synthetic.make_hidden(shape), dev)  # the same batch on every rank
    bias_np = synthetic.make_router_bias(shape)
    bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    T, H = shape.T, shape.H
    partial = torch.empty((T, H), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(h=hidden):
        mm.mm_moe_forward_partial(h, router_w, gu, dn, shape.top_k, shape.renorm,
                                  partial=partial, router_bias=bias)
        tp_combine(partial, ws)
        mm.mm_round_bf16(partial, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    steps = args.steps or 50
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, ws, dev)
    # end to end: the batch from pinned host memory, the step, out back
    h_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    h_host.copy_(hidden.cpu())
    o_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    h_dev = torch.empty_like(hidden)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        h_dev.copy_(h_host, non_blocking=True)
        step(h_dev)
        o_host.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / steps, ws, dev)
    st = mm.mm_poll_device_status()
    if st != mm.MM_OK:
        raise RuntimeError(f"device status after the timed regions: {mm.status_string(st)}")
    pk, pk_kind = peaks()
    ids, _ = mm.mm_route(hidden, router_w, shape.top_k, shape.renorm, router_bias=bias)
    work = algorithmic_work(shape, ids.cpu().numpy())["layer"]
    flops, nbytes = work["flops"], work["bytes"]
    if tensor_regime(shape):
        roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12,
                "peak": pk["bf16_tflops"] * ws, "unit": "TFLOP/s",
                "peak_kind": f"{pk_kind} bf16_tflops (burst) x {ws} GPUs"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9,
                "peak": pk["hbm_gbs"] * ws, "unit": "GB/s",
                "peak_kind": f"{pk_kind} hbm_gbs (copy bandwidth) x {ws} GPUs"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = "whole step (layer on the slice, all-reduce, rounding)"
    roof["traffic"] = None
    line = {"metric": METRIC, "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded normals, bf16; random-init weights of the named shape)",
            "config": {"workload": shape.name, "T": T, "H": H, "E": shape.E,
                       "top_k": shape.top_k, "I": shape.I, "I_per_rank": shape.I // ws,
                       "renorm": shape.renorm, "parallelism": f"tp{ws}",
                       "allreduce_bytes_per_step": T * H * 4},
            "roofline": roof,
            "e2e": {"value": T / e2e_s, "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                    "d2h_bytes_per_step": T * H * 2},
            # the layer's launches, mm_round_bf16 in place of the rounding pass
            "gpu_launches": kernel_launches(shape) * steps, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 0.6 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mm", "reference"], default="mm")
    ap.add_argument("--workload", default=synthetic.DECODE.name)
    ap.add_argument("--sweep-T", type=int, default=None, help="run the Zipf sweep shape at this T")
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="with the decode workload, skip the prefill measurement that the line "
                         "carries as its prefill_qwen3_30b_a3b object")
    ap.add_argument("--add-norm", action="store_true",
                    help="time mm_moe_forward_add_norm_residual: the residual add + RMSNorm "
                         "step before the layer, the layer, and the residual add after it, "
                         "in one call")
    ap.add_argument("--tp", action="store_true",
                    help="tensor-parallel split of one layer over the ranks (each rank a slice "
                         "of the experts' intermediates, one fp32 all-reduce per step) instead "
                         "of one replica per rank")
    ap.add_argument("--dense", action="store_true",
                    help="time mm_gated_mlp: a dense SwiGLU MLP of H x k*I on the workload's "
                         "tokens (the same flops per token as the MoE layer's experts)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    ws, rank, local = dist_info()
    shape = synthetic.SWEEP.with_T(args.sweep_T) if args.sweep_T else synthetic.WORKLOADS[args.workload]
    if ws > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 5  # each step is a full oracle pass over the sample
        run_reference(args, shape, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return

    import mixture_experts_layer_mm_gb300 as mm
    mm.lib()  # fails loudly if the CUDA library is missing
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.dense:
        run_dense(args, shape, ws, rank, dev, mm)
        return
    if args.tp:
        run_tp(args, shape, ws, rank, dev, mm)
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return
    if args.add_norm and synthetic.make_router_bias(shape) is not None:
        raise SystemExit("--add-norm takes no router bias (the Zipf sweep has one)")
    # Each replica gets its own batch (hidden seed = rank); the layer weights are shared.
    w = synthetic.make_weights(shape)
    weights = (_to_dev(w["router_w"], dev), _to_dev(w["w_gate_up"], dev),
               _to_dev(w["w_down"], dev))
    del w
    bias_np = synthetic.make_router_bias(shape)
    bias = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    run = LayerRun(mm, shape, dev, weights, bias, rank, add_norm=args.add_norm)
    run.warmup(args.warmup)
    if args.steps is None:  # size the timed region to about 0.6 s so clocks are sampled
        args.steps = int(max_over_ranks(float(run.auto_steps()), ws, dev))
    st = mm.mm_poll_device_status()
    if st != mm.MM_OK:
        raise RuntimeError(f"device status after warm-up: {mm.status_string(st)}")
    work = run.work()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    # The prefill-shaped layer of the same model, measured in the same run
    # (the metric's tensor-core half), when the workload is the decode layer.
    pre = None
    if shape.name == synthetic.DECODE.name and not args.no_prefill:
        pre_shape = synthetic.PREFILL
        pre = LayerRun(mm, pre_shape, dev, weights, None, rank, add_norm=args.add_norm)
        pre.warmup(args.warmup)
        pre_steps = int(min(200, max(args.steps, 50)))
        pre_work = pre.work()

    pk, pk_kind = peaks()
    # One NVML sampler spans every timed region of the run (A, B, C of the
    # workload, then A and B of the prefill layer).
    with ClockSampler(local) as clk:
        ms, stage_ms, e2e_s = run.measure(args.steps, ws, work["layer"]["bytes"], l2_bytes)
        if pre is not None:
            pre_ms, pre_stage, _ = pre.measure(pre_steps, ws, pre_work["layer"]["bytes"],
                                               l2_bytes, e2e=False)
    clocks = clk.summary()

    T_all = shape.T * ws
    value = job_tokens_per_s(shape.T, ws, ms)
    roof = roofline(shape, work, stage_ms, ms, pk, pk_kind)
    launches_per_step = kernel_launches(shape, args.add_norm)
    flush = run.flushed
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded normals, bf16; random-init weights of the named shape)",
            "config": {"workload": shape.name + ("+add_rmsnorm" if args.add_norm else ""),
                       "T": shape.T, "H": shape.H, "E": shape.E,
                       "top_k": shape.top_k, "I": shape.I, "renorm": shape.renorm,
                       "distinct_experts": work["D"], "parallelism": f"replicas x{ws}",
                       "l2": (f"L2 flushed between steps (a {2 * l2_bytes / 1e6:.0f} MB write and "
                              "read outside each step's events): the step's "
                              f"{work['layer']['bytes'] / 1e6:.0f} MB would fit in L2"
                              if flush else
                              "inputs larger than L2: each step streams the selected experts' "
                              f"weights ({work['layer']['bytes'] / 1e9:.2f} GB)")},
            "roofline": roof,
            "stage_ms": {n: round(v, 5) for n, v in stage_ms.items()},
            "stage_sum_ms": sum(stage_ms.values()),
            "e2e": {"value": T_all / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": int(run.io_bytes),
                    "d2h_bytes_per_step": int(run.io_bytes)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks}
    if flush:
        line["warm"] = {"ms_per_step": run.warm_ms,
                        "value": job_tokens_per_s(shape.T, ws, run.warm_ms), "unit": UNIT,
                        "bytes_frac_hbm": work["layer"]["bytes"] / (run.warm_ms * 1e-3) / 1e9 /
                        pk["hbm_gbs"],
                        "l2": "steps back to back: the step's weights stay in L2"}
    if pre is not None:
        proof = roofline(pre.shape, pre_work, pre_stage, pre_ms, pk, pk_kind)
        line[pre.shape.name + ("+add_rmsnorm" if args.add_norm else "")] = {
            "T": pre.shape.T, "steps": pre_steps, "ms_per_step": pre_ms,
            "value": job_tokens_per_s(pre.shape.T, ws, pre_ms), "unit": UNIT,
            "bound": "tensor", "peak": pk["bf16_tflops"], "peak_kind": proof["peak_kind"],
            "frac_tensor_layer": proof["layer"]["flops_frac_bf16"],
            "frac_tensor_gate_up": proof["frac_tensor"],
            "frac_tensor_down": proof["down"]["frac_tensor"],
            "frac_hbm_layer": proof["layer"]["bytes_frac_hbm"],
            "stage_ms": {n: round(v, 5) for n, v in pre_stage.items()},
            "layer_tflops": pre_work["layer"]["flops"] / (pre_ms * 1e-3) / 1e12,
            "gpu_launches": kernel_launches(pre.shape, args.add_norm) * pre_steps,
            "traffic_gate_up": proof["traffic"]}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
