"""GPU parity of the fused calls at head dimensions that are not powers of two (any multiple of 8
up to 256: DiT-XL's 72, 80, 96, 120, ...), which run the fused kernels (token units and row
blocks) with the run-time row layouts: a row takes d / 16 lanes of eight RoPE pairs where 16
divides d, else d / 8 lanes of four, rows in consecutive lane groups, the lanes past the last
whole group idle.

Forward, backward (dx and dw), the packed call (QKV, QKVG) and its backward, in bf16 and fp16,
adjacent and rotate-half pairs, against the CPU oracle; tolerances as the other fused tests
(within 1e-2 + 1e-2 |ref| of the oracle's unrounded double, and one rounding of an fp32 result:
2^-8 |ref| for bf16, 2^-10 |ref| for fp16, plus 1e-5 forward and 1e-4 for dx; dw within the
bound of test_gpu_fused_bwd). Every geometry spans several token blocks with a ragged tail.
"""
import os

import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from test_gpu_fused_bwd import check_dw
from test_gpu_fullsize import check_all
from test_gpu_fused_variants import _check, _dtype, _inputs, _plan
from test_gpu_packed import _check_dx_pp, _packed_inputs, run_packed
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4
VARIANTS = [(f16, half) for f16 in (0, 1) for half in (0, 1)]
VIDS = [f"{'f16' if f else 'bf16'}-{'half' if h else 'adjacent'}" for f, h in VARIANTS]

# W, b, seq_splits, head_splits, d: rows of 3 to 31 lanes in both run-time layouts
GEOMS = [
    (2, 1, [90, 73], [3, 3], 24),                             # 4 pairs a lane: 3 lanes a row
    (3, 2, [47, 0, 65], [3, 2, 1], 40),
    (2, 1, [70, 50], [4, 4], 48),                             # 8 pairs a lane: 3 lanes a row
    (8, 1, [60, 61, 59, 60, 62, 58, 60, 60], [2] * 8, 72),    # DiT-XL heads: 16 of 72
    (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 80),
    (4, 2, [23, 19, 0, 27], [3, 0, 5, 2], 96),
    (3, 1, [31, 29, 40], [3, 3, 3], 112),
    (2, 1, [75000, 600], [1, 1], 120),                        # positions to 75,599
    (3, 1, [11, 13, 9], [2, 1, 2], 136),
    (2, 2, [13, 17], [2, 2], 160),
    (1, 1, [37], [5], 200),
    (2, 1, [9, 14], [4, 4], 240),                             # 15 lanes of 8 pairs
    (2, 1, [9, 14], [3, 3], 248),                             # 31 lanes of 4 pairs
]


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


ENGINES = {"tokens": B.ULY_ENGINE_TMA, "row_blocks": B.ULY_ENGINE_TENSOR}


def _fits_row_blocks(g):
    """Equal, non-empty head groups with runs of at most 2,048 bytes (2-byte elements)."""
    W, b, seq, heads, d = g
    return len(set(heads)) == 1 and heads[0] > 0 and heads[0] * d * 2 <= 2048


def _forward(g, f16, half, q, k, w, engine=B.ULY_ENGINE_AUTO, cap=None):
    W, b, seq, heads, d = g
    plan = _plan(g, f16, half, cap)
    B.ulysses_plan_set_fused_engine(plan, engine)
    if engine != B.ULY_ENGINE_AUTO:
        want = engine if _fits_row_blocks(g) else B.ULY_ENGINE_TMA
        assert B.ulysses_plan_fused_kernel(plan) == want
    shapes = [(b, sum(seq), n, d) for n in heads]
    qo, ko = GuardedOutputs(shapes, _dtype(f16)), GuardedOutputs(shapes, _dtype(f16))
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo.tensors, ko.tensors, w, EPS, THETA)
    torch.cuda.synchronize()
    assert qo.guards_intact() and ko.guards_intact(), "a kernel wrote outside its output"
    return qo.tensors, ko.tensors


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("variant", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("g", GEOMS, ids=[f"d{g[4]}" for g in GEOMS])
def test_forward_head_dims(oracle, g, variant, engine):
    """Every element of q_out and k_out against the oracle, with each kernel (plans the row
    blocks do not fit take the token units)."""
    f16, half = variant
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, f16, seed=sum(seq) + d + 10 * f16 + half)
    qo, ko = _forward(g, f16, half, q, k, w, engine=ENGINES[engine])
    wn = w.cpu().numpy().astype(np.float64)
    for t, (x, out) in enumerate(((q, qo), (k, ko))):
        ref = oracle.qk_fused_var([host_raw(v) for v in x], seq, heads, wn[t], EPS, THETA, f16, half)
        for r in range(W):
            _check(oracle, host_raw(out[r]), ref[r], f16, 1e-5, f"{g} t{t} r{r}")


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("variant", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("g", GEOMS, ids=[f"d{g[4]}" for g in GEOMS])
def test_backward_head_dims(oracle, g, variant, engine):
    """Every element of dq and dk, and dw, against the oracle's backward, with each kernel."""
    f16, half = variant
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, f16, seed=3 * sum(seq) + d + 10 * f16 + half)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(sum(heads) + d)
    S = sum(seq)
    dq = [torch.randn((b, S, n, d), generator=gen).to(_dtype(f16)).cuda() for n in heads]
    dk = [torch.randn((b, S, n, d), generator=gen).to(_dtype(f16)).cuda() for n in heads]
    plan = _plan(g, f16, half)
    B.ulysses_plan_set_fused_engine(plan, ENGINES[engine])
    want = ENGINES[engine] if _fits_row_blocks(g) else B.ULY_ENGINE_TMA
    assert B.ulysses_plan_fused_backward_kernel(plan) == want
    shapes = [(b, s, sum(heads), d) for s in seq]
    dqo, dko = GuardedOutputs(shapes, _dtype(f16)), GuardedOutputs(shapes, _dtype(f16))
    dwo = GuardedOutputs([(2, d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, dq, dk, w,
                                       dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact() and dwo.guards_intact()
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = b * S * sum(heads)
    for t, (x, gy, got) in enumerate(((q, dq, dqo), (k, dk, dko))):
        ref_dx, ref_dw = oracle.qk_fused_bwd_var([host_raw(v) for v in x],
                                                 [host_raw(v) for v in gy], seq, heads, wn[t],
                                                 EPS, THETA, f16, half)
        for r in range(W):
            _check(oracle, host_raw(got.tensors[r]), ref_dx[r], f16, 1e-4, f"{g} dx t{t} r{r}")
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw, n_rows, f"{g} dw t{t}")


# (geometry, planes, q_plane, k_plane, extra elements per token)
PACKED = [
    ((8, 1, [40, 41, 39, 40, 42, 38, 40, 40], [2] * 8, 72), 3, 0, 1, 0),   # QKV, DiT-XL heads
    ((5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 80), 4, 0, 1, 0),        # QKVG
    ((3, 2, [5, 0, 7], [3, 2, 1], 40), 4, 2, 0, 8),                         # k before q, extra
    ((4, 1, [30, 28, 31, 29], [4] * 4, 112), 4, 0, 1, 0),                   # QKVG, row blocks
]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("case", PACKED, ids=[f"p{c[0][4]}" for c in PACKED])
def test_packed_head_dims(oracle, case, engine):
    """The packed call with each kernel: q and k planes against the oracle's packed form, the
    others byte-exact."""
    g, planes, qp, kp, extra = case
    W, b, seq, heads, d = g
    xs, pitch = _packed_inputs(g, planes, extra, seed=sum(seq) + planes + d)
    w = wl.rms_weights(d, seed=planes + d).cuda()
    outs = run_packed(g, planes, qp, kp, xs, pitch, w, engine=ENGINES[engine])
    wn = w.cpu().numpy().astype(np.float64)
    qo, ko, plain = oracle.packed_fused([host_raw(x) for x in xs], seq, heads, d, planes, qp, kp,
                                        pitch, wn[0], wn[1], EPS, THETA)
    for r in range(W):
        _check(oracle, host_raw(outs[qp][r]), qo[r], 0, 1e-5, f"{case} q rank {r}")
        _check(oracle, host_raw(outs[kp][r]), ko[r], 0, 1e-5, f"{case} k rank {r}")
        for c in range(planes):
            if c not in (qp, kp):
                assert np.array_equal(host_raw(outs[c][r]), plain[c][r]), f"{case} plane {c} rank {r}"


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("case", PACKED, ids=[f"pb{c[0][4]}" for c in PACKED])
def test_packed_backward_head_dims(oracle, case, engine):
    """The packed backward with each kernel: the q and k planes' dx within tolerance, the others
    byte-exact, a token's extra columns untouched, and dw."""
    from gpu_util import FILL
    g, planes, qp, kp, extra = case
    W, b, seq, heads, d = g
    N, S = sum(heads), sum(seq)
    xs, pitch = _packed_inputs(g, planes, extra, seed=sum(seq) + 7 * planes + d)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(planes + 100 + d)
    grads = [[torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).cuda() for n in heads]
             for _ in range(planes)]
    w = wl.rms_weights(d, seed=planes + 3 + d).cuda()
    plan = B.ulysses_plan(*g, "bfloat16")
    B.ulysses_plan_set_fused_engine(plan, ENGINES[engine])
    want = ENGINES[engine] if _fits_row_blocks(g) else B.ULY_ENGINE_TMA
    assert B.ulysses_plan_fused_backward_kernel(plan) == want
    dpk = GuardedOutputs([(b, s, pitch) for s in seq], torch.bfloat16)
    dwo = GuardedOutputs([(2, d)], torch.float32)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_packed_fused_backward(plan, planes, qp, kp, pitch * 2, dpk.tensors, xs, grads,
                                           w, dwo.tensors[0], EPS, THETA, ws)
    torch.cuda.synchronize()
    assert dpk.guards_intact() and dwo.guards_intact(), "a kernel wrote outside its output"
    wn = w.cpu().numpy().astype(np.float64)
    ref_dx, ref_dw = oracle.packed_fused_bwd([host_raw(x) for x in xs],
                                             [[host_raw(t) for t in gp] for gp in grads], seq,
                                             heads, d, planes, qp, kp, pitch, wn[0], wn[1], EPS,
                                             THETA)
    for q in range(W):
        got = host_raw(dpk.tensors[q])
        for c in range(planes):
            cols = slice(c * N * d, (c + 1) * N * d)
            if c in (qp, kp):
                _check_dx_pp(oracle, got[:, :, cols], ref_dx[q][:, :, cols], f"{case} plane {c} q={q}")
            else:
                want = oracle.double_to_bf16(ref_dx[q][:, :, cols])
                assert np.array_equal(got[:, :, cols], want), f"{case} plane {c} q={q}"
        fill = np.uint16(FILL | (FILL << 8))
        assert np.all(got[:, :, planes * N * d:] == fill), f"{case}: extra columns written"
    for t in range(2):
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw[t], b * S * N, f"{case} dw {t}")


def test_head_dim_72_chunked_equals_unchunked():
    """A chunk cap that splits the call into many launches gives the same bytes (forward, and the
    backward's dq and dk; dw within its bound), fp16 rotate-half."""
    g = (8, 2, [300, 310, 290, 305, 295, 300, 301, 299], [2] * 8, 72)
    W, b, seq, heads, d = g
    (q, k), w = _inputs(g, 1, seed=171)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(172)
    S = sum(seq)
    gq = [torch.randn((b, S, n, d), generator=gen).half().cuda() for n in heads]
    gk = [torch.randn((b, S, n, d), generator=gen).half().cuda() for n in heads]
    res = []
    for cap in (None, 64 << 10):
        plan = _plan(g, 1, 1, cap)
        assert B.ulysses_plan_num_chunks(plan, 0) == (1 if cap is None else 23)
        qo = [torch.empty((b, S, n, d), dtype=torch.float16, device="cuda") for n in heads]
        ko = [torch.empty_like(x) for x in qo]
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
        dq = [torch.empty_like(x) for x in q]
        dk = [torch.empty_like(x) for x in k]
        dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device="cuda")
        B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw, EPS, THETA, ws)
        torch.cuda.synchronize()
        res.append((qo + ko + dq + dk, dw))
    for x, y in zip(res[0][0], res[1][0]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    # dw is summed in another order: within the bound of its sum over b * S * N rows
    check_dw(res[1][1].cpu().numpy(), res[0][1].cpu().numpy().astype(np.float64),
             b * S * sum(heads), "chunked dw")


def test_dit_xl_shape_full(oracle):
    """A DiT-XL-shaped exchange at Wan-720p length: W=8, 75,600 tokens, 16 heads of d = 72 (2 per
    rank), bf16: every element of the forward and of the backward's dq, dk against the oracle,
    dw within its bound."""
    g = (8, 1, [9450] * 8, [2] * 8, 72)
    W, b, seq, heads, d = g
    S = sum(seq)
    threads = max(1, os.cpu_count() or 1)
    (q, k), w = _inputs(g, 0, seed=181)
    qo, ko = _forward(g, 0, 0, q, k, w)
    wn = w.cpu().numpy().astype(np.float64)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(182)
    gy = [[torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).cuda() for n in heads]
          for _ in range(2)]
    plan = _plan(g, 0, 0)
    dxs = [[torch.empty_like(x) for x in xs] for xs in (q, k)]
    dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dxs[0], dxs[1], q, k, gy[0], gy[1], w, dw, EPS, THETA,
                                       ws)
    torch.cuda.synchronize()
    for t, (x, out) in enumerate(((q, qo), (k, ko))):
        xh = [host_raw(v) for v in x]
        ref = oracle.qk_fused_A(xh, seq, heads, wn[t], EPS, THETA, threads=threads)
        for r in range(W):
            check_all(out[r], ref[r], 2.0 ** -8, 1e-5, f"forward t{t} r{r}")
        ref_dx, ref_dw = oracle.qk_fused_bwd(xh, [host_raw(v) for v in gy[t]], seq, heads, wn[t],
                                             EPS, THETA, threads=threads)
        for qq in range(W):
            check_all(dxs[t][qq], ref_dx[qq], 2.0 ** -8, 1e-4, f"dx t{t} q{qq}")
        check_dw(dw[t].cpu().numpy(), ref_dw, b * S * sum(heads), f"dw t{t}")


def test_head_dim_72_host_buffers_and_autograd():
    """The host-buffer form and the differentiable form at d = 72 (fp16, rotate-half pairs): the
    host-buffer call returns the device call's bytes, and the autograd gradients are the direct
    backward call's, bit for bit."""
    from ulysses_sequence_all_gb300 import autograd as A
    g = (4, 2, [40, 37, 0, 45], [3, 3, 3, 3], 72)
    W, b, seq, heads, d = g
    S = sum(seq)
    (q, k), w = _inputs(g, 1, seed=191)
    plan = _plan(g, 1, 1)
    qo = [torch.empty((b, S, n, d), dtype=torch.float16, device="cuda") for n in heads]
    ko = [torch.empty_like(x) for x in qo]
    B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
    torch.cuda.synchronize()
    hq = [x.cpu().pin_memory() for x in q]
    hk = [x.cpu().pin_memory() for x in k]
    hqo = [torch.empty(x.shape, dtype=torch.float16).pin_memory() for x in qo]
    hko = [torch.empty(x.shape, dtype=torch.float16).pin_memory() for x in ko]
    dq_in = [torch.empty_like(x) for x in q]
    dk_in = [torch.empty_like(x) for x in k]
    dqo = [torch.empty_like(x) for x in qo]
    dko = [torch.empty_like(x) for x in ko]
    B.ulysses_a2a_4d_qk_fused_host(plan, hq, hk, hqo, hko, dq_in, dk_in, dqo, dko, w, EPS, THETA)
    torch.cuda.synchronize()
    for x, y in zip(hqo + hko, qo + ko):
        assert torch.equal(x.view(torch.int16), y.cpu().view(torch.int16))

    gen = torch.Generator(device="cpu")
    gen.manual_seed(192)
    gq = [torch.randn(x.shape, generator=gen).half().cuda() for x in qo]
    gk = [torch.randn(x.shape, generator=gen).half().cuda() for x in ko]
    qr = [x.clone().requires_grad_() for x in q]
    kr = [x.clone().requires_grad_() for x in k]
    wr = w.clone().requires_grad_()
    ao, bo = A.qk_fused(plan, qr, kr, wr, EPS, THETA)
    torch.autograd.backward(ao + bo, gq + gk)
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dw = torch.empty_like(w)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    for x, y in zip(ao + bo + [t.grad for t in qr + kr], qo + ko + dq + dk):
        assert torch.equal(x.detach().view(torch.int16), y.view(torch.int16))
    assert torch.equal(wr.grad.view(torch.int32), dw.view(torch.int32))
