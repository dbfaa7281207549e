"""Runs the MoE layer a few times on one of the seeded synthetic workloads.

    python -m mixture_experts_layer_mm_gb300.run_layer --workload decode_qwen3_30b_a3b --passes 4
    python -m mixture_experts_layer_mm_gb300.run_layer --sweep-T 8 --passes 4

A short, fixed sequence of forward calls (and nothing else on the GPU) for
checking an installation and for profilers: with --passes P the layer's
kernels run P times back to back, so a profiler can skip the first passes'
launches and capture the last one's. --single-launch calls
mm_moe_forward_single_launch instead of mm_moe_forward. Exits non-zero if
the device status word reports an error.
"""
import argparse
import sys

import numpy as np
import torch

from . import _lib as mm
from . import synthetic


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    g = p.add_mutually_exclusive_group()
    g.add_argument("--workload", default=synthetic.DECODE.name, choices=list(synthetic.WORKLOADS))
    g.add_argument("--sweep-T", type=int, default=None,
                   help="the Zipf-skewed sweep workload at this batch size")
    p.add_argument("--passes", type=int, default=4)
    p.add_argument("--single-launch", action="store_true")
    args = p.parse_args(argv)
    shape = (synthetic.SWEEP.with_T(args.sweep_T) if args.sweep_T
             else synthetic.WORKLOADS[args.workload])
    d = synthetic.make_inputs(shape)

    def dev(b):
        return torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)

    hidden, router_w = dev(d["hidden"]), dev(d["router_w"])
    w_gate_up, w_down = dev(d["w_gate_up"]), dev(d["w_down"])
    bias = None if d["router_bias"] is None else torch.from_numpy(d["router_bias"]).cuda()
    out = torch.empty_like(hidden)
    fwd = mm.mm_moe_forward_single_launch if args.single_launch else mm.mm_moe_forward
    for _ in range(args.passes):
        fwd(hidden, router_w, w_gate_up, w_down, shape.top_k, shape.renorm, out=out,
            router_bias=bias)
    torch.cuda.synchronize()
    status = mm.mm_poll_device_status()
    print(f"{shape.name}: {args.passes} passes, status {mm.status_string(status)}")
    return 0 if status == mm.MM_OK else 1


if __name__ == "__main__":
    sys.exit(main())
