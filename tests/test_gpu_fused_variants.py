"""GPU parity of the fused call's variants (fp16 elements; rotate-half RoPE pairs) against the
CPU oracle, forward, interleaved QKV and backward.

Tolerances: as the bf16 tests (|gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's unrounded
double), plus one rounding of an fp32 result to the element type: 2^-8 |ref| (bf16) or
2^-10 |ref| (fp16), with 1e-5 absolute for the forward and 1e-4 for the backward's dx; dw within
n 2^-20 + 1e-4 for a sum of n rows.
"""
import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from test_gpu_fused import EPS, THETA
from test_gpu_fused_bwd import check_dw
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

VARIANTS = [(f16, half) for f16 in (0, 1) for half in (0, 1)]
VIDS = [f"{'f16' if f else 'bf16'}-{'half' if h else 'adjacent'}" for f, h in VARIANTS]
GEOMS = [
    (2, 1, [16, 16], [4, 4], 128),
    (3, 2, [5, 0, 7], [3, 2, 1], 64),
    (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128),
    (4, 2, [3, 1, 0, 2], [1, 0, 2, 1], 16),
    (2, 1, [7, 2], [3, 1], 8),
    (1, 1, [4], [100], 256),
    (2, 1, [75000, 600], [1, 1], 128),
    # equal head groups: the shapes the row-block (tensor-map) kernel takes
    (3, 2, [5, 0, 7], [2, 2, 2], 64),
    (4, 2, [3, 1, 0, 2], [1, 1, 1, 1], 16),
    (2, 1, [7, 2], [3, 3], 8),
    (8, 1, [37, 41, 29, 33, 40, 35, 31, 38], [5] * 8, 128),
]


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def _dtype(f16):
    return torch.float16 if f16 else torch.bfloat16


def _plan(g, f16, half, cap=None):
    plan = B.ulysses_plan(*g, "float16" if f16 else "bfloat16")
    if half:
        B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    return plan


def _check(oracle, got_raw, ref, f16, atol, what):
    got = oracle.decode(got_raw, f16)
    assert got.shape == ref.shape, what
    if ref.size == 0:
        return
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {err.max():.3e}"
    rel = 2.0 ** -10 if f16 else 2.0 ** -8
    tight = err <= rel * np.abs(ref) + atol
    assert tight.all(), f"{what}: {int((~tight).sum())} elements beyond one rounding"


def _inputs(g, f16, seed, planes=2):
    W, b, seq, heads, d = g
    N = sum(heads)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    xs = [[torch.randn((b, s, N, d), generator=gen).to(_dtype(f16)).cuda() for s in seq]
          for _ in range(planes)]
    return xs, wl.rms_weights(d, seed=seed + 1).cuda()


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_TMA, B.ULY_ENGINE_TENSOR], ids=["tokens", "tensor"])
@pytest.mark.parametrize("variant", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("g", GEOMS, ids=[f"g{i}" for i in range(len(GEOMS))])
def test_forward_variant(oracle, g, variant, engine):
    f16, half = variant
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, f16, seed=sum(seq) + d + 10 * f16 + half)
    plan = _plan(g, f16, half)
    B.ulysses_plan_set_fused_engine(plan, engine)
    shapes = [(b, sum(seq), n, d) for n in heads]
    qo, ko = GuardedOutputs(shapes, _dtype(f16)), GuardedOutputs(shapes, _dtype(f16))
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo.tensors, ko.tensors, w, EPS, THETA)
    torch.cuda.synchronize()
    assert qo.guards_intact() and ko.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    for t, (x, out) in enumerate(((q, qo), (k, ko))):
        ref = oracle.qk_fused_var([host_raw(v) for v in x], seq, heads, wn[t], EPS, THETA, f16, half)
        for r in range(W):
            _check(oracle, host_raw(out.tensors[r]), ref[r], f16, 1e-5, f"{g} t{t} r{r}")


@pytest.mark.parametrize("variant", VARIANTS[1:], ids=VIDS[1:])
def test_qkv_variant(oracle, variant):
    """Interleaved (b, s, 3, N, d): q and k as the variant's fused call, v bit-exact."""
    f16, half = variant
    g = (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128)
    W, b, seq, heads, d = g
    (q, k, v), w = _inputs(g, f16, seed=77, planes=3)
    qkv = [torch.stack([a, bb, c], dim=2) for a, bb, c in zip(q, k, v)]
    plan = _plan(g, f16, half)
    shapes = [(b, sum(seq), n, d) for n in heads]
    outs = [GuardedOutputs(shapes, _dtype(f16)) for _ in range(3)]
    B.ulysses_a2a_4d_qkv_fused(plan, qkv, outs[0].tensors, outs[1].tensors, outs[2].tensors, w,
                               EPS, THETA)
    torch.cuda.synchronize()
    assert all(o.guards_intact() for o in outs)
    wn = w.cpu().numpy().astype(np.float64)
    for t, x in enumerate((q, k)):
        ref = oracle.qk_fused_var([host_raw(v_) for v_ in x], seq, heads, wn[t], EPS, THETA, f16,
                                  half)
        for r in range(W):
            _check(oracle, host_raw(outs[t].tensors[r]), ref[r], f16, 1e-5, f"qkv t{t} r{r}")
    want_v = oracle.a2a_4d([host_raw(x) for x in v], seq, heads, 0)
    for r in range(W):
        assert np.array_equal(host_raw(outs[2].tensors[r]), want_v[r])


@pytest.mark.parametrize("variant", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("g", GEOMS, ids=[f"g{i}" for i in range(len(GEOMS))])
def test_backward_variant(oracle, g, variant):
    f16, half = variant
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, f16, seed=3 * sum(seq) + d + 10 * f16 + half)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(sum(heads) + d)
    S = sum(seq)
    dq = [torch.randn((b, S, n, d), generator=gen).to(_dtype(f16)).cuda() for n in heads]
    dk = [torch.randn((b, S, n, d), generator=gen).to(_dtype(f16)).cuda() for n in heads]
    plan = _plan(g, f16, half)
    shapes = [(b, s, sum(heads), d) for s in seq]
    dqo, dko = GuardedOutputs(shapes, _dtype(f16)), GuardedOutputs(shapes, _dtype(f16))
    dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, dq, dk, w, dw, EPS,
                                       THETA, ws)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = b * S * sum(heads)
    for t, (x, gy, got) in enumerate(((q, dq, dqo), (k, dk, dko))):
        ref_dx, ref_dw = oracle.qk_fused_bwd_var([host_raw(v) for v in x],
                                                 [host_raw(v) for v in gy], seq, heads, wn[t],
                                                 EPS, THETA, f16, half)
        for r in range(W):
            _check(oracle, host_raw(got.tensors[r]), ref_dx[r], f16, 1e-4, f"{g} dx t{t} r{r}")
        check_dw(dw[t].cpu().numpy(), ref_dw, n_rows, f"{g} dw t{t}")


def test_variant_chunked_equals_unchunked():
    g = (5, 2, [100, 110, 90, 105, 95], [9, 8, 8, 8, 7], 128)
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, 1, seed=90)
    res = []
    for cap in (None, 1 << 20):
        plan = _plan(g, 1, 1, cap)
        qo = [torch.empty((b, sum(seq), n, d), dtype=torch.float16, device="cuda") for n in heads]
        ko = [torch.empty_like(x) for x in qo]
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
        torch.cuda.synchronize()
        res.append(qo + ko)
    for x, y in zip(*res):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_wan720p_f16_half_sampled(oracle):
    """The Wan shape with fp16 elements and rotate-half pairs: 500 sampled rows per tensor of
    the forward and of the backward against the oracle's single-row rules."""
    cfg = wl.WAN
    g = (cfg.W, 1, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    q = [torch.randn((1, s, cfg.N, cfg.d), generator=gen, device="cuda").half() for s in cfg.seq_splits]
    k = [torch.randn((1, s, cfg.N, cfg.d), generator=gen, device="cuda").half() for s in cfg.seq_splits]
    gq = [torch.randn((1, cfg.S, n, cfg.d), generator=gen, device="cuda").half() for n in cfg.head_splits]
    gk = [torch.randn((1, cfg.S, n, cfg.d), generator=gen, device="cuda").half() for n in cfg.head_splits]
    w = wl.rms_weights(cfg.d, seed=6).cuda()
    plan = _plan(g, 1, 1)
    qo = [torch.empty((1, cfg.S, n, cfg.d), dtype=torch.float16, device="cuda") for n in cfg.head_splits]
    ko = [torch.empty_like(x) for x in qo]
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dw = torch.empty((2, cfg.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    wn = w.cpu().numpy().astype(np.float64)
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(7)
    for t, (x, out, gy, dx) in enumerate(((q, qo, gq, dq), (k, ko, gk, dk))):
        for _ in range(500):
            qr = int(rng.integers(0, cfg.W))
            i = int(rng.integers(0, cfg.seq_splits[qr]))
            hg = int(rng.integers(0, cfg.N))
            r = int(np.searchsorted(head_off, hg, side="right") - 1)
            p = seq_off[qr] + i
            raw = host_raw(x[qr][0, i, hg])
            want = oracle.fused_row_var(raw, 1, 1, wn[t], EPS, p, THETA)
            _check(oracle, host_raw(out[r][0, p, hg - head_off[r]]), want, 1, 1e-5, f"fwd t{t} p{p}")
            grow = oracle.decode(host_raw(gy[r][0, p, hg - head_off[r]]), 1)
            want_dx, _ = oracle.fused_row_bwd_var(oracle.decode(raw, 1), grow, 1, wn[t], EPS, p, THETA)
            _check(oracle, host_raw(dx[qr][0, i, hg]), want_dx, 1, 1e-4, f"bwd t{t} p{p}")


def test_host_buffer_form_variant():
    """The host-buffer form with fp16 elements and rotate-half pairs gives the device form's bytes."""
    g = (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128)
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, 1, seed=91)
    plan = _plan(g, 1, 1)
    qo = [torch.empty((b, sum(seq), n, d), dtype=torch.float16, device="cuda") for n in heads]
    ko = [torch.empty_like(x) for x in qo]
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
    hq = [x.cpu().pin_memory() for x in q]
    hk = [x.cpu().pin_memory() for x in k]
    hqo = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in qo]
    hko = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in ko]
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dqo = [torch.empty_like(x) for x in qo]
    dko = [torch.empty_like(x) for x in ko]
    B.ulysses_a2a_4d_qk_fused_host(plan, hq, hk, hqo, hko, dq, dk, dqo, dko, w, EPS, THETA)
    torch.cuda.synchronize()
    for a, c in zip(hqo + hko, qo + ko):
        assert torch.equal(a.view(torch.int16), c.cpu().view(torch.int16))

