"""Full-size, element-by-element parity of the fused kernels against the oracle.

Every output element of the fused forward, the interleaved QKV call, the packed QKVG call and the
two backwards is compared at the Wan-720p shape (W=8, b=1, 75,600 tokens, 40 heads, d=128), and the fused forward
and backward also on the long packed-QKV geometry (W=4, 250,000 tokens, 56 heads, positions to
249,999). The
plans, and so the launch configurations (grid, work units, stages, CTAs per SM), are the ones the
benchmark times; its inputs too where it draws them: q, k, v of the step (seeds 3, 4, 5, weights
seed 2), the long geometry's q, k (seeds 3, 4), the fp16 rotate-half Wan shape (seeds 3, 4).

The oracle computes each call in parts on all host cores (ranges of shards and rows; the parts
write disjoint rows and are pinned on the CPU to reproduce the whole call). Its double results are
copied to the device rank by rank and compared there with plain torch arithmetic in double (the
library's outputs widened exactly), which keeps a full-size check to seconds.

Tolerances (as the smaller tests):
* forward outputs: |gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's unrounded double, and
  one rounding of an fp32 result: 2^-8 |ref| + 1e-5 (bf16) or 2^-10 |ref| + 1e-5 (fp16);
* dx of the backwards: the same with 1e-4 absolute (fp32 cancellation in u w - x k at unit-scale
  data);
* v planes: byte-exact;
* dw: within min(n 2^-20, 1e-4 sqrt(n)) + 1e-4 of the oracle's double sum over n rows (see
  check_dw); each test also confirms that one row's own contribution to dw exceeds that bound,
  so a row dropped or counted twice could not pass.
NaN anywhere fails every bound.
"""
import os

import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from test_gpu_fused import EPS, THETA
from test_gpu_fused_bwd import check_dw, dw_bound
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

THREADS = max(1, os.cpu_count() or 1)


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def check_all(got: torch.Tensor, ref: np.ndarray, rel: float, atol: float, what: str):
    """Every element of a device tensor (bf16 or fp16) against the oracle's double result."""
    g = got.to(torch.float64)  # exact widening
    r = torch.from_numpy(ref).to(g.device)
    assert tuple(g.shape) == tuple(r.shape), what
    if r.numel() == 0:
        return
    err = (g - r).abs_()
    ar = r.abs()
    loose = ~(err <= 1e-2 + 1e-2 * ar)  # NaN is never within a bound
    n_loose = int(loose.sum())
    assert n_loose == 0, f"{what}: {n_loose} elements beyond 1e-2 + 1e-2|ref|"
    tight = ~(err <= rel * ar + atol)
    n_tight = int(tight.sum())
    assert n_tight == 0, (f"{what}: {n_tight} elements beyond one rounding "
                          f"(max err {float(err.max()):.3e})")


def check_bytes(got: torch.Tensor, want_u16: np.ndarray, what: str):
    assert np.array_equal(host_raw(got), want_u16), f"{what}: bytes differ"


def _wan_plan(dtype="bfloat16", half=False):
    cfg = wl.WAN
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, dtype)
    if half:
        B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    return cfg, plan


def _head_outputs(cfg, dtype, planes):
    return [GuardedOutputs([cfg.head_side_shape(r) for r in range(cfg.W)], dtype)
            for _ in range(planes)]


def _seq_outputs(cfg, dtype, shape_of=None):
    shape_of = shape_of or cfg.seq_side_shape
    return GuardedOutputs([shape_of(q) for q in range(cfg.W)], dtype)


def _sensitivity(oracle, cfg, xs, gys, w, f16, half, bound, what, rows=16):
    """dw bound below what one row moves: for sampled rows, the largest element of the row's own
    dw contribution (the oracle's row backward of forward input row (q, i, h) and the gradient
    row that mode 0 made of it: rank r's row seq_off(q) + i, head h - head_off(r)) exceeds it."""
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(99)
    for _ in range(rows):
        q = int(rng.integers(0, cfg.W))
        i = int(rng.integers(0, cfg.seq_splits[q]))
        h = int(rng.integers(0, cfg.N))
        r = int(np.searchsorted(head_off, h, side="right") - 1)
        x = oracle.decode(host_raw(xs[q][0, i, h]), f16)
        g = oracle.decode(host_raw(gys[r][0, seq_off[q] + i, h - head_off[r]]), f16)
        _, dw_row = oracle.fused_row_bwd_var(x, g, half, w, EPS, seq_off[q] + i, THETA)
        assert np.abs(dw_row).max() > bound, f"{what}: a row's dw contribution is within the bound"


# ---- forward ----------------------------------------------------------------------------------
def test_fused_wan720p_full(oracle):
    """The step's fused call: q (seed 3) and k (seed 4), weights seed 2, every element, on the
    automatic choice and on both kernels."""
    cfg, plan = _wan_plan()
    q = wl.seq_side_inputs(cfg, "cuda", seed=wl.FUSED.seed)
    k = wl.seq_side_inputs(cfg, "cuda", seed=wl.FUSED.extra["k_seed"])
    w = wl.rms_weights(cfg.d, seed=wl.FUSED.extra["w_seed"]).cuda()
    outs = {}
    for name, engine in (("auto", B.ULY_ENGINE_AUTO), ("tokens", B.ULY_ENGINE_TMA),
                         ("tensor", B.ULY_ENGINE_TENSOR)):
        B.ulysses_plan_set_fused_engine(plan, engine)
        qo, ko = _head_outputs(cfg, torch.bfloat16, 2)
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo.tensors, ko.tensors, w, EPS, THETA)
        torch.cuda.synchronize()
        assert qo.guards_intact() and ko.guards_intact(), f"{name}: a kernel wrote outside its output"
        outs[name] = (qo, ko)
    wn = w.cpu().numpy().astype(np.float64)
    for t, xin in enumerate((q, k)):
        ref = oracle.qk_fused_A([host_raw(x) for x in xin], cfg.seq_splits, cfg.head_splits,
                                wn[t], EPS, THETA, threads=THREADS)
        for name, pair in outs.items():
            for r in range(cfg.W):
                check_all(pair[t].tensors[r], ref[r], 2.0 ** -8, 1e-5, f"{name} tensor {t} rank {r}")
        del ref


def test_fused_wan720p_f16_half_full(oracle):
    """The Wan shape in fp16 with rotate-half pairs (the benchmark's variant configuration):
    every element of q and k."""
    cfg, plan = _wan_plan("float16", half=True)
    cfg16 = wl.Workload("wan720p_fp16", cfg.W, 1, cfg.seq_splits, cfg.head_splits, cfg.d,
                        "float16", seed=1)
    q = wl.seq_side_inputs(cfg16, "cuda", seed=3)
    k = wl.seq_side_inputs(cfg16, "cuda", seed=4)
    w = wl.rms_weights(cfg.d).cuda()
    outs = {}
    for name, engine in (("tokens", B.ULY_ENGINE_TMA), ("tensor", B.ULY_ENGINE_TENSOR)):
        B.ulysses_plan_set_fused_engine(plan, engine)
        qo, ko = _head_outputs(cfg, torch.float16, 2)
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo.tensors, ko.tensors, w, EPS, THETA)
        torch.cuda.synchronize()
        assert qo.guards_intact() and ko.guards_intact(), f"{name}: a kernel wrote outside its output"
        outs[name] = (qo, ko)
    wn = w.cpu().numpy().astype(np.float64)
    for t, xin in enumerate((q, k)):
        ref = oracle.qk_fused_var([host_raw(x) for x in xin], cfg.seq_splits, cfg.head_splits,
                                  wn[t], EPS, THETA, 1, 1, threads=THREADS)
        for name, pair in outs.items():
            for r in range(cfg.W):
                check_all(pair[t].tensors[r], ref[r], 2.0 ** -10, 1e-5, f"{name} tensor {t} rank {r}")
        del ref


def test_qkv_wan720p_full(oracle):
    """The interleaved call on the step's q, k, v stacked as (b, s, 3, N, d): every element of
    q and k, v byte for byte."""
    cfg, plan = _wan_plan()
    planes = [wl.seq_side_inputs(cfg, "cuda", seed=sd) for sd in (3, 4, 5)]
    qkv = [torch.stack(list(p), dim=2) for p in zip(*planes)]
    del planes
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    outs = _head_outputs(cfg, torch.bfloat16, 3)
    B.ulysses_a2a_4d_qkv_fused(plan, qkv, outs[0].tensors, outs[1].tensors, outs[2].tensors, w,
                               EPS, THETA)
    torch.cuda.synchronize()
    assert all(o.guards_intact() for o in outs), "a kernel wrote outside its output"
    wn = w.cpu().numpy().astype(np.float64)
    qo, ko, vo = oracle.qkv_fused([host_raw(x) for x in qkv], cfg.seq_splits, cfg.head_splits,
                                  wn[0], wn[1], EPS, THETA, threads=THREADS)
    for r in range(cfg.W):
        check_all(outs[0].tensors[r], qo[r], 2.0 ** -8, 1e-5, f"q rank {r}")
        check_all(outs[1].tensors[r], ko[r], 2.0 ** -8, 1e-5, f"k rank {r}")
        check_bytes(outs[2].tensors[r], vo[r], f"v rank {r}")


def test_fused_long_sequence_full(oracle):
    """The long packed-QKV geometry's q and k (W=4, 250,000 tokens, 56 heads, d=128, 896,000,000
    bytes per rank and tensor; seeds 3, 4 as the benchmark's configuration table): every element,
    positions up to 249,999."""
    cfg = wl.Workload("long_qk", 4, 1, (62500,) * 4, (14,) * 4, 128, "bfloat16", seed=20)
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    q = wl.seq_side_inputs(cfg, "cuda", seed=3)
    k = wl.seq_side_inputs(cfg, "cuda", seed=4)
    w = wl.rms_weights(cfg.d).cuda()
    qo, ko = _head_outputs(cfg, torch.bfloat16, 2)
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo.tensors, ko.tensors, w, EPS, THETA)
    torch.cuda.synchronize()
    assert qo.guards_intact() and ko.guards_intact(), "a kernel wrote outside its output"
    wn = w.cpu().numpy().astype(np.float64)
    for t, (xin, out) in enumerate(((q, qo), (k, ko))):
        ref = oracle.qk_fused_A([host_raw(x) for x in xin], cfg.seq_splits, cfg.head_splits,
                                wn[t], EPS, THETA, threads=THREADS)
        for r in range(cfg.W):
            check_all(out.tensors[r], ref[r], 2.0 ** -8, 1e-5, f"tensor {t} rank {r}")
            ref[r] = None  # free as we go: 3.6 GB of doubles per rank
        del ref


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_AUTO, B.ULY_ENGINE_TMA], ids=["auto", "tokens"])
def test_packed_qkvg_wan720p_full(oracle, engine):
    """QKVG packed as (b, s, 4, N, d) (q, k, v of the step, seeds 3, 4, 5, and a gate plane, seed
    6): one call; every element of q and k, v and g byte for byte (the automatic choice, row
    blocks at this shape, and the token units)."""
    cfg, plan = _wan_plan()
    B.ulysses_plan_set_fused_engine(plan, engine)
    planes = [wl.seq_side_inputs(cfg, "cuda", seed=sd) for sd in (3, 4, 5, 6)]
    packed = [torch.stack(list(p), dim=2) for p in zip(*planes)]
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    outs = _head_outputs(cfg, torch.bfloat16, 4)
    B.ulysses_a2a_4d_packed_fused(plan, 4, 0, 1, 4 * cfg.N * cfg.d * 2, packed,
                                  [o.tensors for o in outs], w, EPS, THETA)
    torch.cuda.synchronize()
    assert all(o.guards_intact() for o in outs), "a kernel wrote outside its output"
    del packed
    wn = w.cpu().numpy().astype(np.float64)
    # the packed oracle is the planes' slices through the fused transform and mode 0 (pinned)
    for t in (0, 1):
        ref = oracle.qk_fused_A([host_raw(x) for x in planes[t]], cfg.seq_splits,
                                cfg.head_splits, wn[t], EPS, THETA, threads=THREADS)
        for r in range(cfg.W):
            check_all(outs[t].tensors[r], ref[r], 2.0 ** -8, 1e-5, f"plane {t} rank {r}")
        del ref
    for c in (2, 3):
        want = oracle.a2a_4d([host_raw(x) for x in planes[c]], cfg.seq_splits, cfg.head_splits, 0)
        for r in range(cfg.W):
            check_bytes(outs[c].tensors[r], want[r], f"plane {c} rank {r}")


# ---- backward ---------------------------------------------------------------------------------
def _wan_grads(cfg, dtype, seeds):
    """Output gradients of q and k, N(0, 1) head-side tensors (independent of the outputs, so
    the dw terms average to zero and one row's contribution stands out of the rounding)."""
    return [wl.head_side_inputs(wl.Workload("g", cfg.W, 1, cfg.seq_splits, cfg.head_splits, cfg.d,
                                            dtype, seed=sd), "cuda") for sd in seeds]


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_AUTO, B.ULY_ENGINE_TMA], ids=["auto", "tokens"])
def test_backward_wan720p_full(oracle, engine):
    """Backward at the Wan shape on the step's q, k (seeds 3, 4), weights seed 2, output
    gradients N(0, 1) (seeds 52, 53): every element of dq and dk, and dw."""
    cfg, plan = _wan_plan()
    B.ulysses_plan_set_fused_engine(plan, engine)
    q = wl.seq_side_inputs(cfg, "cuda", seed=3)
    k = wl.seq_side_inputs(cfg, "cuda", seed=4)
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    gq, gk = _wan_grads(cfg, "bfloat16", (52, 53))
    dqo, dko = _seq_outputs(cfg, torch.bfloat16), _seq_outputs(cfg, torch.bfloat16)
    dwo = GuardedOutputs([(2, cfg.d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, gq, gk, w,
                                       dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact() and dwo.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = cfg.S * cfg.N
    for t, (x, gy, got) in enumerate(((q, gq, dqo), (k, gk, dko))):
        xh = [host_raw(v) for v in x]
        ref_dx, ref_dw = oracle.qk_fused_bwd(xh, [host_raw(v) for v in gy], cfg.seq_splits,
                                             cfg.head_splits, wn[t], EPS, THETA, threads=THREADS)
        for qr in range(cfg.W):
            check_all(got.tensors[qr], ref_dx[qr], 2.0 ** -8, 1e-4, f"tensor {t} rank {qr}")
        del ref_dx
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"dw {t}")
        _sensitivity(oracle, cfg, x, gy, wn[t], 0, 0, dw_bound(n_rows), f"dw {t}")


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_AUTO, B.ULY_ENGINE_TMA], ids=["auto", "tokens"])
def test_qkv_backward_wan720p_full(oracle, engine):
    """Backward of the interleaved call at the Wan shape: packed q, k, v of the step (seeds
    3, 4, 5), output gradients N(0, 1) (seeds 52, 53, 54): every element of the q and k planes of
    dqkv, the v plane byte for byte (mode 1 of its gradient), and dw."""
    cfg, plan = _wan_plan()
    B.ulysses_plan_set_fused_engine(plan, engine)
    planes = [wl.seq_side_inputs(cfg, "cuda", seed=sd) for sd in (3, 4, 5)]
    qkv = [torch.stack(list(p), dim=2) for p in zip(*planes)]
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    gq, gk, gv = _wan_grads(cfg, "bfloat16", (52, 53, 54))
    packed = lambda q: (1, cfg.seq_splits[q], 3, cfg.N, cfg.d)  # noqa: E731
    dqkv = _seq_outputs(cfg, torch.bfloat16, packed)
    dwo = GuardedOutputs([(2, cfg.d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qkv_fused_backward(plan, dqkv.tensors, qkv, gq, gk, gv, w, dwo.tensors[0],
                                        EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dqkv.guards_intact() and dwo.guards_intact(), "a kernel wrote outside its output"
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = cfg.S * cfg.N
    want_v = oracle.a2a_4d([host_raw(x) for x in gv], cfg.seq_splits, cfg.head_splits, 1)
    for qr in range(cfg.W):
        check_bytes(dqkv.tensors[qr][:, :, 2].contiguous(), want_v[qr], f"v rank {qr}")
    del want_v
    for t, gy in enumerate((gq, gk)):
        ref_dx, ref_dw = oracle.qk_fused_bwd([host_raw(p) for p in planes[t]],
                                             [host_raw(v) for v in gy], cfg.seq_splits,
                                             cfg.head_splits, wn[t], EPS, THETA, threads=THREADS)
        for qr in range(cfg.W):
            check_all(dqkv.tensors[qr][:, :, t], ref_dx[qr], 2.0 ** -8, 1e-4,
                      f"plane {t} rank {qr}")
        del ref_dx
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"dw {t}")


def test_packed_qkvg_backward_wan720p_full(oracle):
    """Backward of the QKVG packed call at the Wan shape: packed q, k, v, g (seeds 3, 4, 5, 6),
    output gradients N(0, 1) (seeds 52, 53, 54, 55): every element of the q and k planes of the
    packed gradient, the v and g planes byte for byte (mode 1 of their gradients), and dw."""
    cfg, plan = _wan_plan()
    planes = [wl.seq_side_inputs(cfg, "cuda", seed=sd) for sd in (3, 4, 5, 6)]
    packed = [torch.stack(list(p), dim=2) for p in zip(*planes)]
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    grads = _wan_grads(cfg, "bfloat16", (52, 53, 54, 55))
    shape = lambda q: (1, cfg.seq_splits[q], 4, cfg.N, cfg.d)  # noqa: E731
    dpk = _seq_outputs(cfg, torch.bfloat16, shape)
    dwo = GuardedOutputs([(2, cfg.d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_packed_fused_backward(plan, 4, 0, 1, 4 * cfg.N * cfg.d * 2, dpk.tensors,
                                           packed, grads, w, dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dpk.guards_intact() and dwo.guards_intact(), "a kernel wrote outside its output"
    del packed
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = cfg.S * cfg.N
    for c in (2, 3):
        want = oracle.a2a_4d([host_raw(x) for x in grads[c]], cfg.seq_splits, cfg.head_splits, 1)
        for qr in range(cfg.W):
            check_bytes(dpk.tensors[qr][:, :, c].contiguous(), want[qr], f"plane {c} rank {qr}")
        del want
    # the packed backward oracle is the planes' slices through the pinned backward (pinned)
    for t in (0, 1):
        ref_dx, ref_dw = oracle.qk_fused_bwd([host_raw(x) for x in planes[t]],
                                             [host_raw(v) for v in grads[t]], cfg.seq_splits,
                                             cfg.head_splits, wn[t], EPS, THETA, threads=THREADS)
        for qr in range(cfg.W):
            check_all(dpk.tensors[qr][:, :, t], ref_dx[qr], 2.0 ** -8, 1e-4, f"plane {t} rank {qr}")
        del ref_dx
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"dw {t}")


def test_backward_long_sequence_full(oracle):
    """Backward on the long packed-QKV geometry's q and k (W=4, 250,000 tokens, 56 heads, d=128;
    seeds 3, 4 as the benchmark's configuration table), output gradients N(0, 1) (seeds 52, 53):
    every element of dq and dk, positions to 249,999, and dw (n = 14,000,000 rows per tensor)."""
    cfg = wl.Workload("long_qk", 4, 1, (62500,) * 4, (14,) * 4, 128, "bfloat16", seed=20)
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    q = wl.seq_side_inputs(cfg, "cuda", seed=3)
    k = wl.seq_side_inputs(cfg, "cuda", seed=4)
    w = wl.rms_weights(cfg.d).cuda()
    gq, gk = _wan_grads(cfg, "bfloat16", (52, 53))
    dqo, dko = _seq_outputs(cfg, torch.bfloat16), _seq_outputs(cfg, torch.bfloat16)
    dwo = GuardedOutputs([(2, cfg.d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, gq, gk, w,
                                       dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact() and dwo.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = cfg.S * cfg.N
    for t, (x, gy, got) in enumerate(((q, gq, dqo), (k, gk, dko))):
        ref_dx, ref_dw = oracle.qk_fused_bwd([host_raw(v) for v in x], [host_raw(v) for v in gy],
                                             cfg.seq_splits, cfg.head_splits, wn[t], EPS, THETA,
                                             threads=THREADS)
        for qr in range(cfg.W):
            check_all(got.tensors[qr], ref_dx[qr], 2.0 ** -8, 1e-4, f"tensor {t} rank {qr}")
            ref_dx[qr] = None  # free as we go: 3.6 GB of doubles per rank
        del ref_dx
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"dw {t}")
        _sensitivity(oracle, cfg, x, gy, wn[t], 0, 0, dw_bound(n_rows), f"dw {t}")


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_AUTO, B.ULY_ENGINE_TMA], ids=["auto", "tokens"])
def test_backward_wan720p_f16_half_full(oracle, engine):
    """Backward of the fp16 rotate-half variant at the Wan shape (q, k seeds 3, 4; gradients
    N(0, 1) seeds 52, 53): every element of dq and dk, and dw."""
    cfg, plan = _wan_plan("float16", half=True)
    B.ulysses_plan_set_fused_engine(plan, engine)
    cfg16 = wl.Workload("wan720p_fp16", cfg.W, 1, cfg.seq_splits, cfg.head_splits, cfg.d,
                        "float16", seed=1)
    q = wl.seq_side_inputs(cfg16, "cuda", seed=3)
    k = wl.seq_side_inputs(cfg16, "cuda", seed=4)
    w = wl.rms_weights(cfg.d).cuda()
    gq, gk = _wan_grads(cfg, "float16", (52, 53))
    dqo, dko = _seq_outputs(cfg, torch.float16), _seq_outputs(cfg, torch.float16)
    dwo = GuardedOutputs([(2, cfg.d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, gq, gk, w,
                                       dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact() and dwo.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = cfg.S * cfg.N
    for t, (x, gy, got) in enumerate(((q, gq, dqo), (k, gk, dko))):
        ref_dx, ref_dw = oracle.qk_fused_bwd_var([host_raw(v) for v in x], [host_raw(v) for v in gy],
                                                 cfg.seq_splits, cfg.head_splits, wn[t], EPS,
                                                 THETA, 1, 1, threads=THREADS)
        for qr in range(cfg.W):
            check_all(got.tensors[qr], ref_dx[qr], 2.0 ** -10, 1e-4, f"tensor {t} rank {qr}")
        del ref_dx
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"dw {t}")
        _sensitivity(oracle, cfg, x, gy, wn[t], 1, 1, dw_bound(n_rows), f"dw {t}")

