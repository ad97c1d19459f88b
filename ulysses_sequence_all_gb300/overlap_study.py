"""Overlap study: the relayout running next to a GEMM chain on another stream.

    python -m ulysses_sequence_all_gb300.overlap_study [--gemms 24] [--pairs 24] [--reps 5]

The pages report that their collective hides almost completely under a concurrent GEMM chain
(fast-ulysses 0.1.0, "Results": 86% on B200, ~105% on A100). They do not define the figure; the
reading used here is the share of the relayout's own time that disappears when it runs beside the
chain: hidden = (T_gemm + T_relayout - T_both) / T_relayout, where T_both is the time from a common
start until both chains have finished. 100% means the relayout cost nothing; 0% means the two ran
one after the other.

Workload: the Wan-720p exchange (W=8, 75,600 tokens, 40 heads, d=128, bf16), `pairs` times a
mode-0 then mode-1 relayout on one stream; on a second stream `gemms` bf16 matrix products of
8192 x 8192 x 8192 (cuBLAS through torch.matmul; the load, not part of the library). Each engine
is measured alone, the chain alone, and both together, with the relayout stream at default and
at high priority, and for the SM engines under caps on their CTAs (`ulysses_plan_set_max_ctas`,
which leaves the other SMs to the GEMM). Prints one JSON object per case. CUDA events on the
launching streams; inputs are far larger than the L2.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import binding as B
from . import workloads as wl

ENGINES = {"tma": B.ULY_ENGINE_TMA, "vec": B.ULY_ENGINE_VEC, "ce": B.ULY_ENGINE_CE,
           "tensor": B.ULY_ENGINE_TENSOR}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gemms", type=int, default=24)
    ap.add_argument("--pairs", type=int, default=24)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--gemm-size", type=int, default=8192)
    ap.add_argument("--engines", default="tma,vec,ce,tensor")
    ap.add_argument("--max-ctas", default="0",
                    help="comma-separated CTA caps for the SM engines (0: no cap)")
    ap.add_argument("--priorities", default="default,high")
    args = ap.parse_args()

    cfg = wl.WAN
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    x = wl.seq_side_inputs(cfg, "cuda")
    head = [torch.empty(cfg.head_side_shape(r), dtype=torch.bfloat16, device="cuda")
            for r in range(cfg.W)]
    back = [torch.empty_like(t) for t in x]
    n = args.gemm_size
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    a = torch.randn((n, n), generator=gen, device="cuda").to(torch.bfloat16)
    bm = torch.randn((n, n), generator=gen, device="cuda").to(torch.bfloat16)
    c = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    bytes_pair = 2 * 2 * cfg.plane_bytes()  # mode 0 and mode 1, each read + write
    flops_gemm = 2.0 * n * n * n

    s_gemm = torch.cuda.Stream()
    streams = {"default": torch.cuda.Stream(), "high": torch.cuda.Stream(priority=-1)}

    def gemm_chain(st):
        with torch.cuda.stream(st):
            for _ in range(args.gemms):
                torch.matmul(a, bm, out=c)

    def relayout_chain(st, engine):
        for _ in range(args.pairs):
            B.ulysses_a2a_4d_engine(plan, 0, engine, x, head, st)
            B.ulysses_a2a_4d_engine(plan, 1, engine, head, back, st)

    def timed(fn_by_stream):
        """Start every stream on one event; return each stream's elapsed ms and the max."""
        start = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        start.record(cur)
        ends = {}
        for st, fn in fn_by_stream:
            st.wait_event(start)
            fn(st)
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
            ends[st] = e
        torch.cuda.synchronize()
        per = {st: start.elapsed_time(e) for st, e in ends.items()}
        return per, max(per.values())

    def median_of(fn_by_stream):
        runs = [timed(fn_by_stream) for _ in range(args.reps + 1)][1:]  # first run warms up
        per = {st: statistics.median(r[0][st] for r in runs) for st, _ in fn_by_stream}
        return per, statistics.median(r[1] for r in runs)

    (_, t_gemm) = median_of([(s_gemm, gemm_chain)])
    print(json.dumps({"case": "gemm alone", "ms": round(t_gemm, 3),
                      "TFLOP/s": round(args.gemms * flops_gemm / (t_gemm * 1e-3) / 1e12, 1)}),
          flush=True)
    cases = []
    for name in args.engines.split(","):
        caps = [0] if name == "ce" else [int(c) for c in args.max_ctas.split(",")]
        cases += [(name, cap) for cap in caps]
    for name, cap in cases:
        engine = ENGINES[name]
        B.ulysses_plan_set_max_ctas(plan, cap)
        st = streams["default"]
        _, t_rel = median_of([(st, lambda s, e=engine: relayout_chain(s, e))])
        print(json.dumps({"case": f"{name} alone", "max_ctas": cap, "ms": round(t_rel, 3),
                          "GB/s": round(args.pairs * bytes_pair / (t_rel * 1e-3) / 1e9, 1)}),
              flush=True)
        for prio in args.priorities.split(","):
            st = streams[prio]
            per, t_both = median_of([(s_gemm, gemm_chain),
                                     (st, lambda s, e=engine: relayout_chain(s, e))])
            hidden = (t_gemm + t_rel - t_both) / t_rel
            print(json.dumps({
                "case": f"{name} + gemm chain", "max_ctas": cap, "relayout_stream": prio,
                "ms_both": round(t_both, 3), "ms_gemm_part": round(per[s_gemm], 3),
                "ms_relayout_part": round(per[st], 3),
                "relayout_GB/s_under_load": round(args.pairs * bytes_pair / (per[st] * 1e-3) / 1e9, 1),
                "gemm_slowdown": round(per[s_gemm] / t_gemm, 3),
                "hidden": round(hidden, 3)}), flush=True)
    status = B.ulysses_device_status()
    if status:
        raise SystemExit(f"device status word {status:#x}")


if __name__ == "__main__":
    main()
