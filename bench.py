"""Benchmark of the Ulysses exchange around one attention block at the Wan-720p shape.

One step is one pass of the whole hot path over one batch of synthetic bf16 input, W=8 virtual
ranks, b=1, 75,600 tokens (9,450 per rank), 40 heads (5 per rank), d=128:
  1. q and k: mode 0 with QK RMSNorm + RoPE fused into the scatter (one launch),
  2. v: plain mode 0 (one launch),
  3. the attention output: plain mode 1 back to sequence shards (one launch).
Throughput counts algorithmic bytes (every tensor byte read once and written once) per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle on this machine's host cores on the same workload
geometry (a bounded sequence slice per step); it is a slow plain program, not a tuned baseline.
Under torchrun (N > 1) every rank runs its own replica of the workload on its own GPU (the path
does not shard across GPUs); the value is all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "relayout GB/s (read+write) at Wan-720p shape, W=8; % of HBM roofline"
EPS, THETA = 1e-6, 1e4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", action="store_true",
                    help="instead of the step: time modes 0 and 1 on every other configuration "
                         "(uneven W/dtype points, long packed QKV) and print one JSON line")
    return ap.parse_args()


def aggregate_throughput(local_ms: float, bytes_per_rank_step: int, dist=None, device="cpu"):
    """Whole-job throughput of replicas: every rank's bytes over the slowest rank's time.
    Returns (max ms per step over ranks, GB/s of all ranks together)."""
    world, ms = 1, float(local_ms)
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, bytes_per_rank_step * world / (ms * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------
def _reason_summary(rows):
    """Union of the active throttle reasons over sample rows (dicts with a 'reasons' set)."""
    out = set()
    for r in rows:
        out |= r["reasons"]
    return sorted(out)


class NvmlSampler:
    """SM clock, power and clock-event (throttle) reasons of one GPU, read through NVML
    (libnvidia-ml via ctypes; read-only queries, no setting is changed) every `period_s` on a
    background thread, each sample with its host time. At 2 ms a timed region of a few tens of
    milliseconds holds samples, which a 50 ms nvidia-smi poll would miss."""

    CLOCK_SM = 1  # NVML_CLOCK_SM
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                   ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        import ctypes
        self.ct = ctypes
        self.period = period_s
        self.samples = []
        self.marks = {}
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        ok = False
        try:  # the CUDA device's own UUID: robust to CUDA_VISIBLE_DEVICES renumbering
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            ok = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) == 0
        except Exception:  # noqa: BLE001
            ok = False
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [v for v in vis.split(",") if v.strip().isdigit()]
            idx = int(ids[cuda_index]) if cuda_index < len(ids) else cuda_index
            if self.lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.dev)) != 0:
                raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.dev, self.CLOCK_SM, ctypes.byref(mx)) == 0 else None)
        self._stop = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _read(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        t = time.perf_counter()
        sm = float(clk.value) if self.lib.nvmlDeviceGetClockInfo(self.dev, self.CLOCK_SM,
                                                                  ct.byref(clk)) == 0 else None
        watts = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.dev, ct.byref(pw)) == 0 else None
        bits = rs.value if self.reasons_fn(self.dev, ct.byref(rs)) == 0 else 0
        return {"t": t, "sm": sm, "w": watts,
                "reasons": {name for name, bit in self.REASON_BITS if bits & bit}}

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            self._stop.wait(self.period)

    def start(self):
        self.thread.start()
        time.sleep(0.05)

    def mark(self, which):
        self.marks[which] = time.perf_counter()

    def window(self, t0, t1):
        """Summary of the samples taken between host times t0 and t1."""
        inside = [r for r in self.samples if t0 <= r["t"] <= t1]
        sm = [r["sm"] for r in inside if r["sm"] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": _reason_summary(inside), "samples": len(inside),
                "power_w_max": max((r["w"] or 0.0) for r in inside) if inside else None}

    def stop(self):
        self._stop.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()
        t0, t1 = self.marks.get("t0"), self.marks.get("t1")
        if t0 is None or t1 is None:
            return None
        out = self.window(t0, t1)
        out["samples_in_timed_region"] = out.pop("samples")
        out["source"] = f"NVML every {self.period * 1e3:.0f} ms, samples inside the timed region"
        out["timed_region_ms_host"] = round((t1 - t0) * 1e3, 2)
        k0, k1 = self.marks.get("k0"), self.marks.get("k1")
        if k0 is not None and k1 is not None:
            out["per_kernel_pass"] = self.window(k0, k1)
        return out


class SmiSampler:
    """Fallback when NVML cannot be loaded: nvidia-smi samples (50 ms) of the same fields."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, which):
        self.marks[which] = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0, t1 = self.marks.get("t0"), self.marks.get("t1")
        rows = [(t, l.split(", ")) for t, l in self.lines if l.count(",") >= 8]
        inside = [r for t, r in rows if t0 is not None and t0 <= t <= t1]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][1][2]) if rows else None, "reasons": sorted(reasons),
                "samples_in_timed_region": len(inside),
                "source": "nvidia-smi every 50 ms, samples inside the timed region only "
                          "(none when the region is shorter than the period)",
                "power_w_max": max((num(r[3]) or 0.0) for r in inside) if inside else None}


def clock_sampler(cuda_index: int):
    try:
        return NvmlSampler(cuda_index)
    except (OSError, AttributeError):
        return SmiSampler(cuda_index)


# ------------------------------------------------------------------------------------------------
class Workload:
    def __init__(self, torch, B, wl, device):
        self.torch, self.B = torch, B
        cfg = wl.WAN
        self.cfg = cfg
        bf16 = torch.bfloat16
        self.plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
        self.q = wl.seq_side_inputs(cfg, device, seed=wl.FUSED.seed)
        self.k = wl.seq_side_inputs(cfg, device, seed=wl.FUSED.extra["k_seed"])
        self.v = wl.seq_side_inputs(cfg, device, seed=5)
        self.o = wl.head_side_inputs(cfg, device, seed=6)
        self.w = wl.rms_weights(cfg.d, seed=wl.FUSED.extra["w_seed"]).to(device)
        head = [cfg.head_side_shape(r) for r in range(cfg.W)]
        seq = [cfg.seq_side_shape(q) for q in range(cfg.W)]
        self.qo = [torch.empty(s, dtype=bf16, device=device) for s in head]
        self.ko = [torch.empty(s, dtype=bf16, device=device) for s in head]
        self.vo = [torch.empty(s, dtype=bf16, device=device) for s in head]
        self.oo = [torch.empty(s, dtype=bf16, device=device) for s in seq]
        self.side = cfg.plane_bytes()          # one tensor set, all ranks: 774,144,000 bytes
        self.bytes_fused = 4 * self.side       # q, k in; q, k out
        self.bytes_plain = 2 * self.side       # in + out
        self.bytes_step = self.bytes_fused + 2 * self.bytes_plain
        self.launches_per_step = (B.ulysses_plan_num_chunks(self.plan, 0) * 2 +
                                  B.ulysses_plan_num_chunks(self.plan, 1))

    def step(self, stream, ev=None):
        """One exchange step on `stream`; `ev`, if given, holds three events recorded after the
        fused call, after the v relayout and after the attention-output relayout."""
        B = self.B
        B.ulysses_a2a_4d_qk_fused(self.plan, self.q, self.k, self.qo, self.ko, self.w, EPS, THETA,
                                  stream)
        if ev:
            ev[0].record(stream)
        B.ulysses_a2a_4d(self.plan, 0, self.v, self.vo, stream)
        if ev:
            ev[1].record(stream)
        B.ulysses_a2a_4d(self.plan, 1, self.o, self.oo, stream)
        if ev:
            ev[2].record(stream)


def back_to_back_ms(torch, stream, fn, n):
    """Durations (ms) of n launches of fn enqueued back to back, from CUDA events recorded on
    `stream` between consecutive calls. One call is enqueued before the first event, so the GPU is
    busy whenever an event is recorded and the host's launch latency is not counted (an event
    recorded on an idle GPU would time the host's enqueueing of the next call as well)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    fn()
    evs[0].record(stream)
    for i in range(n):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]


def d2d_gbs(torch, nbytes, reps=20):
    """Flat device-to-device copy (cudaMemcpyAsync) of nbytes, counted as read + write."""
    a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    a.fill_(1)
    for _ in range(3):
        b.copy_(a)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        b.copy_(a)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / reps
    del a, b
    return 2 * nbytes / (ms * 1e-3) / 1e9


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_digest(files) -> str | None:
    """sha256 (first 16 hex digits) of the named csrc files, concatenated in the given order."""
    import hashlib
    h = hashlib.sha256()
    for name in files:
        try:
            with open(os.path.join(ROOT, "ulysses_sequence_all_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def read_traffic(kernel: str):
    """Per-launch DRAM bytes (read + write) from the committed ncu summary, or None when the
    kernel's sources have changed since the counters were taken. Lines of profiles/traffic.txt:
    kernel  comma-separated-source-files  digest  bytes-per-launch."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    except OSError:
        return None
    for parts in lines:
        if len(parts) >= 4 and parts[0] == kernel:
            return int(parts[3]) if source_digest(parts[1].split(",")) == parts[2] else None
    return None


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
def oracle_step_sample(tokens_per_rank: int, seed: int = 0):
    """Inputs for one oracle step on the Wan geometry with `tokens_per_rank` tokens per rank."""
    import numpy as np
    rng = np.random.default_rng(seed)
    W, N, d = 8, 40, 128
    seq = [tokens_per_rank] * W
    heads = [5] * W
    S = sum(seq)

    def bf16(shape):  # bf16 bit patterns of N(0, 1) values
        x = rng.standard_normal(shape, dtype=np.float32)
        return (x.view(np.uint32) >> 16).astype(np.uint16)

    q = [bf16((1, s, N, d)) for s in seq]
    k = [bf16((1, s, N, d)) for s in seq]
    v = [bf16((1, s, N, d)) for s in seq]
    o = [bf16((1, S, n, d)) for n in heads]
    w = 1.0 + 0.1 * rng.standard_normal((2, d))
    return seq, heads, q, k, v, o, w


def oracle_step(orc, sample):
    seq, heads, q, k, v, o, w = sample
    orc.qk_fused_A(q, seq, heads, w[0], EPS, THETA)
    orc.qk_fused_A(k, seq, heads, w[1], EPS, THETA)
    orc.a2a_4d(v, seq, heads, 0)
    orc.a2a_4d(o, seq, heads, 1)


def sample_bytes(tokens_per_rank: int) -> int:
    side = 8 * tokens_per_rank * 40 * 128 * 2
    return 4 * side + 2 * (2 * side)


def host_description():
    """The host's logical CPU count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def oracle_leg(budget_s: float = 15.0):
    """The single-threaded C oracle on one step of the Wan geometry, a token slice sized to
    about budget_s seconds."""
    import oracle
    orc = oracle.get()
    t = 64
    smp = oracle_step_sample(t)
    t0 = time.perf_counter()
    oracle_step(orc, smp)
    per_token = (time.perf_counter() - t0) / t
    tokens = max(64, min(9450, int(budget_s / max(per_token, 1e-9))))
    smp = oracle_step_sample(tokens, seed=1)
    t0 = time.perf_counter()
    oracle_step(orc, smp)
    dt = time.perf_counter() - t0
    return {"value": round(sample_bytes(tokens) / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": (f"one step (fused q,k mode 0 + v mode 0 + o mode 1) on the Wan-720p geometry "
                       f"with {tokens} of 9,450 tokens per rank (W=8, 40 heads, d=128, bf16), "
                       f"single-threaded C oracle, {dt:.1f} s")}


def memcpy_leg(reps: int = 5):
    """The multi-threaded CPU relayout (one memcpy per row and destination rank, rows shared
    among OpenMP threads; oracle/segment_memcpy.c, byte-equal to the oracle) on the full Wan-720p
    tensor set: mode 0 of a sequence-side set and mode 1 of a head-side set, every host thread,
    median of `reps` calls each."""
    import numpy as np
    import oracle
    seg = oracle.SegmentMemcpy()
    W, N, d, s_local = 8, 40, 128, 9450
    seq, heads = [s_local] * W, [5] * W
    rng = np.random.default_rng(3)
    v = [rng.integers(0, 1 << 16, (1, s_local, N, d), dtype=np.uint16) for _ in range(W)]
    o = [rng.integers(0, 1 << 16, (1, W * s_local, 5, d), dtype=np.uint16) for _ in range(W)]
    vo = [np.empty_like(x) for x in o]
    oo = [np.empty_like(x) for x in v]
    side = sum(x.nbytes for x in v)
    threads = seg.max_threads()
    per_mode = {}
    for mode, ins, outs in ((0, v, vo), (1, o, oo)):
        seg.a2a_4d(ins, seq, heads, mode, outs=outs)  # first touch of the outputs
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            seg.a2a_4d(ins, seq, heads, mode, outs=outs)
            ts.append(time.perf_counter() - t0)
        per_mode[f"mode{mode}"] = round(2 * side / statistics.median(ts) / 1e9, 3)
    value = 2 * (2 * side) / (2 * side / (per_mode["mode0"] * 1e9) + 2 * side / (per_mode["mode1"] * 1e9)) / 1e9
    return {"value": round(value, 3), "unit": "GB/s", "cores": threads,
            "kind": "segment_memcpy_openmp", **{f"{k}_GBps": v_ for k, v_ in per_mode.items()},
            "sample": (f"relayout only (no norm or rotation): modes 0 and 1 of the full Wan-720p "
                       f"tensor set ({side:,} bytes per side), {threads} OpenMP threads, median "
                       f"of {reps} calls per mode; value = both modes' bytes over both modes' "
                       f"time")}


def cpu_baseline(budget_s: float = 15.0):
    """Both CPU legs on the host cores: the oracle (single thread, the contract's reported
    baseline: its figure is `value`) and the multi-threaded memcpy relayout."""
    orc = oracle_leg(budget_s)
    out = dict(orc)
    out["host"] = host_description()
    out["legs"] = {"oracle_single_thread": orc, "segment_memcpy_all_threads": memcpy_leg()}
    return out


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    orc = oracle.get()
    smp = oracle_step_sample(32)
    t0 = time.perf_counter()
    oracle_step(orc, smp)
    per_token = (time.perf_counter() - t0) / 32
    total_steps = args.steps + args.warmup
    tokens = max(8, min(2048, int(60.0 / total_steps / max(per_token, 1e-9))))
    smp = oracle_step_sample(tokens, seed=2)
    for _ in range(args.warmup):
        oracle_step(orc, smp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(orc, smp)
    dt = time.perf_counter() - t0
    value = sample_bytes(tokens) * args.steps / dt / 1e9
    sample = (f"each step: fused q,k mode 0 + v mode 0 + o mode 1 on the Wan-720p geometry with "
              f"{tokens} of 9,450 tokens per rank, single-threaded C oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(), "gpu_launches": 0,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_description()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def workload_config():
    return {"workload": "wan720p_ulysses_attention_exchange", "W": 8, "b": 1, "s_global": 75600,
            "n_global": 40, "d": 128, "dtype": "bf16",
            "step": "fused q,k RMSNorm+RoPE mode 0 + v mode 0 + attention-out mode 1",
            "bytes_per_step": 8 * 774144000,
            "l2": "inputs larger than L2 (774,144,000 B per tensor set vs 126 MB L2), no flush",
            "parallelism": "replicas"}


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    from ulysses_sequence_all_gb300 import binding as B
    from ulysses_sequence_all_gb300 import workloads as wl

    wk = Workload(torch, B, wl, "cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        wk.step(stream)
    torch.cuda.synchronize()
    assert B.ulysses_device_status() == 0

    # outside the step: the interleaved (b, s, 3, N, d) QKV form of its first two launches
    qkv = [torch.stack([a, b, c], dim=2) for a, b, c in zip(wk.q, wk.k, wk.v)]
    for _ in range(3):
        B.ulysses_a2a_4d_qkv_fused(wk.plan, qkv, wk.qo, wk.ko, wk.vo, wk.w, EPS, THETA, stream)
    qkv_ms = back_to_back_ms(torch, stream, lambda: B.ulysses_a2a_4d_qkv_fused(
        wk.plan, qkv, wk.qo, wk.ko, wk.vo, wk.w, EPS, THETA, stream), min(args.steps, 20))
    del qkv

    # outside the step: QKVG packed as (b, s, 4, N, d) (the step's q, k, v and a gate plane), one
    # launch for all four planes
    cfg = wk.cfg
    gate = wl.seq_side_inputs(cfg, "cuda", seed=7)
    qkvg = [torch.stack([a, b, c, g], dim=2) for a, b, c, g in zip(wk.q, wk.k, wk.v, gate)]
    go = [torch.empty_like(t) for t in wk.vo]
    packed = lambda: B.ulysses_a2a_4d_packed_fused(  # noqa: E731
        wk.plan, 4, 0, 1, 4 * cfg.N * cfg.d * 2, qkvg, [wk.qo, wk.ko, wk.vo, go], wk.w, EPS, THETA,
        stream)
    for _ in range(3):
        packed()
    qkvg_ms = back_to_back_ms(torch, stream, packed, min(args.steps, 20))
    del gate, qkvg, go

    # outside the step: the backward of the fused call (dq, dk and dw from the gradients of q_out
    # and k_out; the step's own outputs serve as those gradients)
    dq = [torch.empty_like(t) for t in wk.q]
    dk = [torch.empty_like(t) for t in wk.k]
    dw = torch.empty((2, wk.cfg.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(wk.plan), dtype=torch.uint8,
                     device="cuda")
    bwd = lambda: B.ulysses_a2a_4d_qk_fused_backward(  # noqa: E731
        wk.plan, dq, dk, wk.q, wk.k, wk.qo, wk.ko, wk.w, dw, EPS, THETA, ws, stream)
    for _ in range(3):
        bwd()
    bwd_ms = back_to_back_ms(torch, stream, bwd, min(args.steps, 20))
    # the backward of the interleaved form: packed dqkv from the three output gradients
    qkv = [torch.stack([a, b, c], dim=2) for a, b, c in zip(wk.q, wk.k, wk.v)]
    dqkv = [torch.empty_like(t) for t in qkv]
    qkv_bwd = lambda: B.ulysses_a2a_4d_qkv_fused_backward(  # noqa: E731
        wk.plan, dqkv, qkv, wk.qo, wk.ko, wk.vo, wk.w, dw, EPS, THETA, ws, stream)
    for _ in range(3):
        qkv_bwd()
    qkv_bwd_ms = back_to_back_ms(torch, stream, qkv_bwd, min(args.steps, 20))
    del dq, dk, dw, ws, qkv, dqkv

    # Per-kernel durations: the same steps enqueued back to back, one event per kernel boundary
    # (bounds[3 i] precedes step i's fused call, bounds[3 i + 1..3] follow its three launches).
    # The GPU stays busy across the pass, so consecutive events time each launch without the
    # host's launch latency. Kept out of the timed region, whose steps carry no extra events.
    clocks = clock_sampler(local)
    clocks.start()
    nk = max(2, min(args.steps, 50))
    bounds = [torch.cuda.Event(enable_timing=True) for _ in range(3 * nk + 1)]
    wk.step(stream)  # keeps the GPU busy while bounds[0] is recorded
    bounds[0].record(stream)
    clocks.mark("k0")
    for i in range(nk):
        wk.step(stream, bounds[3 * i + 1:3 * i + 4])
    torch.cuda.synchronize()
    clocks.mark("k1")
    kt = {name: [bounds[3 * i + j].elapsed_time(bounds[3 * i + j + 1]) for i in range(nk)]
          for j, name in enumerate(("fused_qk", "mode0", "mode1"))}
    del bounds

    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    start.record(stream)
    for _ in range(args.steps):
        wk.step(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    if pg:
        pg.barrier()
    clock_info = clocks.stop()
    ms, value = aggregate_throughput(start.elapsed_time(end) / args.steps, wk.bytes_step, pg, "cuda")
    if clock_info and clock_info.get("sm_mhz"):
        clock_info["ms_per_step_x_sm_mhz"] = round(ms * clock_info["sm_mhz"], 1)
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"

    # end to end through the host-buffer entry points: pinned host in, device, pinned host out
    e2e = run_e2e(torch, B, wk, stream, args)
    e2e["ms_per_step"], e2e_value = aggregate_throughput(e2e["ms_per_step"], wk.bytes_step, pg, "cuda")
    e2e["value"] = round(e2e_value, 3)

    tg = torch_gpu_step(torch, wk, stream) if rank == 0 else None
    med = {k: statistics.median(v) for k, v in kt.items()}
    gbs = {"fused_qk": wk.bytes_fused / (med["fused_qk"] * 1e-3) / 1e9,
           "mode0": wk.bytes_plain / (med["mode0"] * 1e-3) / 1e9,
           "mode1": wk.bytes_plain / (med["mode1"] * 1e-3) / 1e9}
    dominant = max(med, key=lambda k: med[k])
    peak, peak_kind = read_peaks()
    relayout_kernel = ("relayout_tensor_kernel" if B.ulysses_plan_auto_engine(wk.plan) ==
                       B.ULY_ENGINE_TENSOR else "relayout_rows_kernel")
    fused_kernel = ("fused_qk_tensor_kernel" if B.ulysses_plan_fused_kernel(wk.plan) ==
                    B.ULY_ENGINE_TENSOR else "fused_qk_kernel")
    kernel_name = {"fused_qk": fused_kernel, "mode0": f"{relayout_kernel}<0>",
                   "mode1": f"{relayout_kernel}<1>"}[dominant]
    traffic = read_traffic(kernel_name)
    d2d = d2d_gbs(torch, wk.side) if rank == 0 else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, Wan-720p-shaped; no dataset)",
        "config": workload_config(),
        "clocks": clock_info,
        "e2e": {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")},
        "e2e_detail": {"ms_per_step": round(e2e["ms_per_step"], 3),
                       "per_call_ms": e2e["per_call_ms"],
                       "window_ms": e2e["window_ms"], "steps_per_window": max(3, args.e2e_steps)},
        "gpu_launches": wk.launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "kernel": kernel_name,
                     "achieved": round(gbs[dominant], 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs[dominant] / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": {"fused_qk": wk.bytes_fused,
                                                      "mode0": wk.bytes_plain,
                                                      "mode1": wk.bytes_plain}[dominant]},
        "kernels": {k: {"kernel": {"fused_qk": fused_kernel}.get(k, relayout_kernel),
                        "median_ms": round(med[k], 4), "min_ms": round(min(kt[k]), 4),
                        "launches_timed": len(kt[k]), "GB/s": round(gbs[k], 1),
                        "frac_of_peak": round(gbs[k] / peak, 4),
                        "frac_of_d2d": round(gbs[k] / d2d, 4) if d2d else None} for k in med},
        "d2d_copy_GBps": round(d2d, 1) if d2d else None,
        "torch_gpu": None if tg is None else {
            "note": "context: the same three operations as plain PyTorch GPU ops (torch.cat per "
                    "output rank; fp32 RMSNorm + RoPE as separate kernels before the cat), same "
                    "tensors, CUDA events; speedup = its time / this library's kernel time",
            **{k: dict(v, speedup=round(v["median_ms"] / med[k], 2)) for k, v in tg.items()},
            "step_ms": round(sum(v["median_ms"] for v in tg.values()), 4)},
        "qkv_fused": {
            "note": "outside the step: q, k, v interleaved (b, s, 3, N, d), one launch in place of "
                    "the step's fused_qk + mode0 launches",
            "median_ms": round(statistics.median(qkv_ms), 4),
            "GB/s": round(6 * wk.side / (statistics.median(qkv_ms) * 1e-3) / 1e9, 1),
            "frac_of_peak": round(6 * wk.side / (statistics.median(qkv_ms) * 1e-3) / 1e9 / peak, 4)},
        "packed_qkvg_fused": {
            "note": "outside the step: q, k, v and a gate plane packed as (b, s, 4, N, d), one "
                    "launch: q, k normalised and rotated, v and g moved (mode 0)",
            "median_ms": round(statistics.median(qkvg_ms), 4),
            "GB/s": round(8 * wk.side / (statistics.median(qkvg_ms) * 1e-3) / 1e9, 1),
            "frac_of_peak": round(8 * wk.side / (statistics.median(qkvg_ms) * 1e-3) / 1e9 / peak, 4)},
        "qk_fused_backward": {
            "note": "outside the step: dq, dk (bf16) and dw (fp32) of the fused call, the RMSNorm + "
                    "RoPE VJP inside the mode-1 gather (2 launches: kernel + dw reduction); reads "
                    "q, k and the two output gradients, writes dq and dk",
            "median_ms": round(statistics.median(bwd_ms), 4),
            "GB/s": round(6 * wk.side / (statistics.median(bwd_ms) * 1e-3) / 1e9, 1),
            "frac_of_peak": round(6 * wk.side / (statistics.median(bwd_ms) * 1e-3) / 1e9 / peak, 4)},
        "qkv_fused_backward": {
            "note": "outside the step: the interleaved call's backward, packed dq, dk, dv (b, s, 3, "
                    "N, d) from the three output gradients (2 launches); reads the q and k planes "
                    "and three gradients, writes three planes",
            "median_ms": round(statistics.median(qkv_bwd_ms), 4),
            "GB/s": round(8 * wk.side / (statistics.median(qkv_bwd_ms) * 1e-3) / 1e9, 1),
            "frac_of_peak": round(8 * wk.side / (statistics.median(qkv_bwd_ms) * 1e-3) / 1e9 / peak, 4)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def torch_gpu_step(torch, wk, stream, reps=5):
    """Context baseline: the step's three operations written with plain PyTorch ops on the GPU
    (the single-GPU analogue of the pages' baseline, a permute + all-to-all + permute with the
    norm and the rotation as separate kernels): per output rank one torch.cat of the slices each
    input rank sends, and for q and k an fp32 RMSNorm and adjacent-pair RoPE (cos/sin of every
    position built once, outside the timing) before the cat. Not the product path; timed back to
    back with CUDA events like the library's calls, on the same tensors, median of `reps`."""
    cfg = wk.cfg
    W, d = cfg.W, cfg.d
    seq_off = [sum(cfg.seq_splits[:q]) for q in range(W)]
    head_off = [sum(cfg.head_splits[:r]) for r in range(W)]
    j = torch.arange(d // 2, dtype=torch.float64, device="cuda")
    ang = torch.arange(cfg.S, dtype=torch.float64, device="cuda")[:, None] * (THETA ** (-2.0 * j / d))
    cos, sin = torch.cos(ang).float(), torch.sin(ang).float()

    def norm_rope(x, w, q):
        xf = x.float()
        y = xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + EPS) * w
        c = cos[seq_off[q]:seq_off[q] + x.shape[1]][None, :, None, :]
        sn = sin[seq_off[q]:seq_off[q] + x.shape[1]][None, :, None, :]
        e, o = y[..., 0::2], y[..., 1::2]
        return torch.stack((e * c - o * sn, e * sn + o * c), dim=-1).flatten(-2).to(x.dtype)

    def mode0(xs, outs):
        for r in range(W):
            n = cfg.head_splits[r]
            torch.cat([x[:, :, head_off[r]:head_off[r] + n] for x in xs], dim=1, out=outs[r])

    def mode1(ys, outs):
        for q in range(W):
            s = cfg.seq_splits[q]
            torch.cat([y[:, seq_off[q]:seq_off[q] + s] for y in ys], dim=2, out=outs[q])

    ops = {
        "fused_qk": (lambda: (mode0([norm_rope(x, wk.w[0], q) for q, x in enumerate(wk.q)], wk.qo),
                              mode0([norm_rope(x, wk.w[1], q) for q, x in enumerate(wk.k)], wk.ko)),
                     wk.bytes_fused),
        "mode0": (lambda: mode0(wk.v, wk.vo), wk.bytes_plain),
        "mode1": (lambda: mode1(wk.o, wk.oo), wk.bytes_plain),
    }
    out = {}
    with torch.cuda.stream(stream):
        for name, (fn, nbytes) in ops.items():
            fn()
            ms = statistics.median(back_to_back_ms(torch, stream, fn, reps))
            out[name] = {"median_ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return out


def run_e2e(torch, B, wk, stream, args):
    """The same step with every input copied from pinned host memory and every output read
    back into pinned host memory inside the timed region (host-buffer C ABI entry points)."""
    pin = lambda ts: [t.cpu().pin_memory() for t in ts]  # noqa: E731
    hq, hk, hv, ho = pin(wk.q), pin(wk.k), pin(wk.v), pin(wk.o)
    hqo = [torch.empty_like(t, device="cpu").pin_memory() for t in wk.qo]
    hko = [torch.empty_like(t, device="cpu").pin_memory() for t in wk.ko]
    hvo = [torch.empty_like(t, device="cpu").pin_memory() for t in wk.vo]
    hoo = [torch.empty_like(t, device="cpu").pin_memory() for t in wk.oo]

    def step():
        B.ulysses_a2a_4d_qk_fused_host(wk.plan, hq, hk, hqo, hko, wk.q, wk.k, wk.qo, wk.ko, wk.w,
                                       EPS, THETA, stream)
        B.ulysses_a2a_4d_host(wk.plan, 0, hv, hvo, wk.v, wk.vo, stream)
        B.ulysses_a2a_4d_host(wk.plan, 1, ho, hoo, wk.o, wk.oo, stream)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    # Host<->device bandwidth is shared with the rest of the machine and moves from second to
    # second, so the step is timed over several short windows of back-to-back steps and the
    # median window is reported (all windows are listed in e2e_detail).
    n = max(3, args.e2e_steps)
    windows = []
    for _ in range(5):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(n):
            step()
        e.record(stream)
        torch.cuda.synchronize()
        windows.append(s.elapsed_time(e) / n)
    ms = statistics.median(windows)
    h2d = sum(t.numel() * t.element_size() for t in hq + hk + hv + ho)
    d2h = sum(t.numel() * t.element_size() for t in hqo + hko + hvo + hoo)

    # outside the timed region: each host-buffer call on its own (median of 3)
    calls = {
        "fused_qk": lambda: B.ulysses_a2a_4d_qk_fused_host(wk.plan, hq, hk, hqo, hko, wk.q, wk.k,
                                                           wk.qo, wk.ko, wk.w, EPS, THETA, stream),
        "mode0": lambda: B.ulysses_a2a_4d_host(wk.plan, 0, hv, hvo, wk.v, wk.vo, stream),
        "mode1": lambda: B.ulysses_a2a_4d_host(wk.plan, 1, ho, hoo, wk.o, wk.oo, stream),
    }
    per_call = {}
    for name, fn in calls.items():
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        per_call[name] = round(statistics.median(ts), 3)
    return {"value": round(wk.bytes_step / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "per_call_ms": per_call, "window_ms": [round(w, 3) for w in windows]}


def tiny_latency(torch, B, wl, stream, reps=200, in_graph=100):
    """The tiny configuration (W=2, b=1, 16 tokens per rank, 8 heads, d=128, bf16; 65,536 bytes
    per side) is a latency point. Reported: the device time of one round trip (mode 0 then mode 1
    back), from a CUDA graph of `in_graph` round trips replayed on an otherwise idle GPU (no host
    launch cost inside; median of 5 replays); the host time of a round trip through the C ABI from
    Python (perf_counter over `reps` round trips, one synchronize at the end), which is what a
    caller launching one call at a time sees; and a bit-exact check of the round trip."""
    cfg = wl.TINY
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    x = wl.seq_side_inputs(cfg, "cuda")
    y = [torch.empty(cfg.head_side_shape(r), dtype=torch.bfloat16, device="cuda") for r in range(cfg.W)]
    z = [torch.empty_like(t) for t in x]

    def round_trip():  # on the current stream
        B.ulysses_a2a_4d(plan, 0, x, y)
        B.ulysses_a2a_4d(plan, 1, y, z)

    for _ in range(10):
        round_trip()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(in_graph):
            round_trip()
    graph.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    device_us = statistics.median(ts) * 1e3 / in_graph
    t0 = time.perf_counter()
    for _ in range(reps):
        round_trip()
    torch.cuda.synchronize()
    host_us = (time.perf_counter() - t0) / reps * 1e6
    exact = all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(x, z))
    assert exact, "tiny round trip did not return its input"
    return {"config": cfg.name, "kernel": "relayout round trip (latency point)", "W": cfg.W,
            "dtype": cfg.dtype, "bytes": 2 * cfg.relayout_bytes(),
            "round_trip_device_us": round(device_us, 2), "round_trip_host_us": round(host_us, 2),
            "launches_per_round_trip": 2, "round_trip_bit_exact": exact}


def run_configs(args):
    """The tiny configuration's latency (tiny_latency), then modes 0 and 1 on the parity-test
    configurations (not the headline): the 12 uneven
    (W, dtype) points (b=2, 75,000 tokens, 40 heads, d=128) and the long packed-QKV geometry
    (W=4, 250,000 tokens, 56 heads; three planes of 896,000,000 bytes per rank, one call per
    plane on views of a (3, b, s, N, d) buffer per rank); then the fused call and its backward on
    the fp16 uneven plans, the long geometry's q and k, and the Wan shape in fp16 with
    rotate-half pairs. Inputs already in HBM and larger than L2; CUDA events, median of 20
    launches after 5 warm-up launches."""
    import torch
    from ulysses_sequence_all_gb300 import binding as B
    from ulysses_sequence_all_gb300 import workloads as wl

    peak, peak_kind = read_peaks()
    stream = torch.cuda.current_stream()

    def timed(fn, reps=20, warm=5):
        for _ in range(warm):
            fn()
        return statistics.median(back_to_back_ms(torch, stream, fn, reps))

    def engine_name(plan):  # the relayout kernel the automatic engine takes
        return ("tensor" if B.ulysses_plan_auto_engine(plan) == B.ULY_ENGINE_TENSOR
                else "row_tiles")

    def fused_name(plan):  # the fused forward's kernel
        return ("row_blocks" if B.ulysses_plan_fused_kernel(plan) == B.ULY_ENGINE_TENSOR
                else "token_units")

    rows = [tiny_latency(torch, B, wl, stream)]
    for cfg in wl.UNEVEN:
        plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
        dt = wl.torch_dtype(cfg.dtype)
        seq = wl.seq_side_inputs(cfg, "cuda")
        head = [torch.empty(cfg.head_side_shape(r), dtype=dt, device="cuda") for r in range(cfg.W)]
        seq_out = [torch.empty_like(t) for t in seq]
        nbytes = cfg.relayout_bytes()
        for mode, ins, outs in ((0, seq, head), (1, head, seq_out)):
            ms = timed(lambda: B.ulysses_a2a_4d(plan, mode, ins, outs, stream))
            gbs = nbytes / (ms * 1e-3) / 1e9
            rows.append({"config": cfg.name, "kernel": "relayout", "W": cfg.W,
                         "dtype": cfg.dtype, "mode": mode, "engine": engine_name(plan),
                         "bytes": nbytes, "median_ms": round(ms, 4), "GB/s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4)})
        del seq, head, seq_out
    cfg = wl.LONG_QKV
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    dt = wl.torch_dtype(cfg.dtype)
    packed_in = [torch.empty((3,) + cfg.seq_side_shape(q), dtype=dt, device="cuda")
                 for q in range(cfg.W)]
    for p in range(3):
        for q, t in enumerate(wl.seq_side_inputs(cfg, "cuda", plane=p)):
            packed_in[q][p].copy_(t)
    packed_out = [torch.empty((3,) + cfg.head_side_shape(r), dtype=dt, device="cuda")
                  for r in range(cfg.W)]
    nbytes = cfg.relayout_bytes()
    for mode in (0, 1):
        src, dst = (packed_in, packed_out) if mode == 0 else (packed_out, packed_in)

        def planes():
            for p in range(3):
                B.ulysses_a2a_4d(plan, mode, [t[p] for t in src], [t[p] for t in dst], stream)

        ms = timed(planes, reps=10, warm=2)
        gbs = 3 * nbytes / (ms * 1e-3) / 1e9
        rows.append({"config": cfg.name + "_3planes", "kernel": "relayout", "W": cfg.W,
                     "dtype": cfg.dtype, "mode": mode, "bytes": 3 * nbytes, "median_ms": round(ms, 4),
                     "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)})
    del packed_in, packed_out

    # the fused call (q, k: mode 0 + RMSNorm + RoPE) and its backward on other geometries
    fused_cfgs = [(c, "adjacent") for c in wl.UNEVEN if c.dtype == "float16"]
    fused_cfgs += [(wl.Workload("long_qk", 4, 1, (62500,) * 4, (14,) * 4, 128, "bfloat16", seed=20),
                    "adjacent"),
                   (wl.Workload("wan720p_fp16", 8, 1, (9450,) * 8, (5,) * 8, 128, "float16", seed=1),
                    "half")]
    # head dimensions beside 128 at the Wan-720p length (W=8, 75,600 tokens): DiT-XL's 16 heads of
    # 72, and 64, 80, 96, 120 (the non-powers of two take the run-time row layouts)
    fused_cfgs += [(wl.Workload(f"s75600_N{8 * n}_d{d}", 8, 1, (9450,) * 8, (n,) * 8, d, "bfloat16",
                                seed=1), "adjacent")
                   for n, d in ((2, 72), (2, 64), (5, 80), (3, 96), (2, 120))]
    for cfg, pairs in fused_cfgs:
        plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
        if pairs == "half":
            B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
        dt = wl.torch_dtype(cfg.dtype)
        q = wl.seq_side_inputs(cfg, "cuda", seed=3)
        k = wl.seq_side_inputs(cfg, "cuda", seed=4)
        w = wl.rms_weights(cfg.d).cuda()
        qo = [torch.empty(cfg.head_side_shape(r), dtype=dt, device="cuda") for r in range(cfg.W)]
        ko = [torch.empty_like(t) for t in qo]
        side = cfg.plane_bytes()
        ms = timed(lambda: B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA, stream))
        gbs = 4 * side / (ms * 1e-3) / 1e9
        rows.append({"config": cfg.name, "kernel": "fused_qk", "W": cfg.W, "dtype": cfg.dtype,
                     "rope_pairs": pairs, "fused_kernel": fused_name(plan), "bytes": 4 * side,
                     "median_ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4)})
        dq = [torch.empty_like(t) for t in q]
        dk = [torch.empty_like(t) for t in k]
        dw = torch.empty((2, cfg.d), dtype=torch.float32, device="cuda")
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device="cuda")
        ms = timed(lambda: B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, qo, ko, w, dw,
                                                              EPS, THETA, ws, stream))
        gbs = 6 * side / (ms * 1e-3) / 1e9
        rows.append({"config": cfg.name, "kernel": "fused_qk_backward", "W": cfg.W,
                     "dtype": cfg.dtype, "rope_pairs": pairs, "bytes": 6 * side,
                     "median_ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4)})
        del q, k, qo, ko, dq, dk, ws

    # the interleaved (b, s, 3, N, d) call and its backward on the long packed-QKV geometry
    cfg = wl.Workload("long_qkv_interleaved", 4, 1, (62500,) * 4, (14,) * 4, 128, "bfloat16",
                      seed=20)
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    qkv = [torch.stack(list(planes), dim=2) for planes in
           zip(*(wl.seq_side_inputs(cfg, "cuda", seed=sd) for sd in (3, 4, 5)))]
    w = wl.rms_weights(cfg.d).cuda()
    outs = [[torch.empty(cfg.head_side_shape(r), dtype=torch.bfloat16, device="cuda")
             for r in range(cfg.W)] for _ in range(3)]
    side = cfg.plane_bytes()
    ms = timed(lambda: B.ulysses_a2a_4d_qkv_fused(plan, qkv, outs[0], outs[1], outs[2], w, EPS,
                                                  THETA, stream))
    gbs = 6 * side / (ms * 1e-3) / 1e9
    rows.append({"config": cfg.name, "kernel": "qkv_fused", "W": cfg.W, "dtype": cfg.dtype,
                 "rope_pairs": "adjacent", "fused_kernel": fused_name(plan), "bytes": 6 * side, "median_ms": round(ms, 4),
                 "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)})
    dqkv = [torch.empty_like(t) for t in qkv]
    dw = torch.empty((2, cfg.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    ms = timed(lambda: B.ulysses_a2a_4d_qkv_fused_backward(plan, dqkv, qkv, outs[0], outs[1],
                                                           outs[2], w, dw, EPS, THETA, ws, stream))
    gbs = 8 * side / (ms * 1e-3) / 1e9
    rows.append({"config": cfg.name, "kernel": "qkv_fused_backward", "W": cfg.W,
                 "dtype": cfg.dtype, "rope_pairs": "adjacent", "bytes": 8 * side,
                 "median_ms": round(ms, 4), "GB/s": round(gbs, 1),
                 "frac_of_peak": round(gbs / peak, 4)})
    del qkv, outs, dqkv, ws
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"
    print(json.dumps({"configs": rows, "peak": peak, "peak_source": f"{peak_kind} hbm_gbs",
                      "note": "parity-test configurations, timed for context; not bench lines"}),
          flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.configs:
        run_configs(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
