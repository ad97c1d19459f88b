"""Profiling harness: runs the library's kernels on one workload a few times, for ncu captures.

    python -m ulysses_sequence_all_gb300.profile_case --kernel all --workload wan --iters 2

Allocates only what the chosen kernels need (the Wan-720p shape: 774,144,000 bytes per tensor
set, about 3.1 GB for the fused call's inputs and outputs), launches each kernel `iters` times,
synchronises and checks the device status word. It reports no timing. The backward (`bwd`)
holds six tensor sets (4.6 GB at the Wan shape; `wan_half` halves the sequence).
"""
from __future__ import annotations

import argparse

import torch

from . import binding as B
from . import workloads as wl

# half the Wan sequence (37,800 tokens; 387 MB per tensor set) for captures with many passes
WAN_HALF = wl.Workload("wan720p_half", 8, 1, (4725,) * 8, (5,) * 8, 128, "bfloat16", seed=1)
# the Wan-720p length with 16 heads of 64 or of 72 (DiT-XL's heads; a run-time row layout)
N16_D64 = wl.Workload("s75600_N16_d64", 8, 1, (9450,) * 8, (2,) * 8, 64, "bfloat16", seed=1)
N16_D72 = wl.Workload("s75600_N16_d72", 8, 1, (9450,) * 8, (2,) * 8, 72, "bfloat16", seed=1)
WORKLOADS = {"wan": wl.WAN, "wan_half": WAN_HALF, "long": wl.LONG_QKV, "tiny": wl.TINY,
             "n16_d64": N16_D64, "n16_d72": N16_D72}
ENGINES = {"auto": B.ULY_ENGINE_AUTO, "tma": B.ULY_ENGINE_TMA, "vec": B.ULY_ENGINE_VEC,
           "tensor": B.ULY_ENGINE_TENSOR}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["fused", "bwd", "mode0", "mode1", "all"], default="all")
    ap.add_argument("--engine", choices=sorted(ENGINES), default="auto")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="wan")
    ap.add_argument("--iters", type=int, default=2)
    args = ap.parse_args()
    cfg = WORKLOADS[args.workload]
    engine = ENGINES[args.engine]
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    dt = wl.torch_dtype(cfg.dtype)
    head = [torch.empty(cfg.head_side_shape(r), dtype=dt, device="cuda") for r in range(cfg.W)]
    if args.kernel in ("mode0", "all"):
        x = wl.seq_side_inputs(cfg, "cuda")
        for _ in range(args.iters):
            B.ulysses_a2a_4d_engine(plan, 0, engine, x, head)
        torch.cuda.synchronize()
        del x
    if args.kernel in ("mode1", "all"):
        y = wl.head_side_inputs(cfg, "cuda")
        seq = [torch.empty(cfg.seq_side_shape(q), dtype=dt, device="cuda") for q in range(cfg.W)]
        for _ in range(args.iters):
            B.ulysses_a2a_4d_engine(plan, 1, engine, y, seq)
        torch.cuda.synchronize()
        del y, seq
    if args.kernel in ("fused", "all"):
        q = wl.seq_side_inputs(cfg, "cuda", seed=3)
        k = wl.seq_side_inputs(cfg, "cuda", seed=4)
        w = wl.rms_weights(cfg.d).cuda()
        ko = [torch.empty_like(t) for t in head]
        for _ in range(args.iters):
            B.ulysses_a2a_4d_qk_fused(plan, q, k, head, ko, w, 1e-6, 1e4)
        torch.cuda.synchronize()
    if args.kernel in ("bwd", "all"):
        q = wl.seq_side_inputs(cfg, "cuda", seed=3)
        k = wl.seq_side_inputs(cfg, "cuda", seed=4)
        gq = wl.head_side_inputs(cfg, "cuda", seed=5)
        gk = wl.head_side_inputs(cfg, "cuda", seed=6)
        w = wl.rms_weights(cfg.d).cuda()
        dq = [torch.empty_like(t) for t in q]
        dk = [torch.empty_like(t) for t in k]
        dw = torch.empty((2, cfg.d), dtype=torch.float32, device="cuda")
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device="cuda")
        for _ in range(args.iters):
            B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw, 1e-6, 1e4, ws)
        torch.cuda.synchronize()
    status = B.ulysses_device_status()
    if status:
        raise SystemExit(f"device status word {status:#x}")


if __name__ == "__main__":
    main()
