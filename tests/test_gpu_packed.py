"""GPU parity of the fused call on packed inputs (C planes per token, a token pitch: QKV, QKVG and
other packings) against the CPU oracle.

Tolerances as the other fused tests: |gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's
unrounded double, and one rounding of an fp32 result (2^-8 |ref| + 1e-5 for bf16, 2^-10 |ref| +
1e-5 for fp16); the planes other than q and k byte-exact.
"""
import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from test_gpu_fused import EPS, THETA, check_close
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


# (geometry, planes, q_plane, k_plane, extra elements per token beyond the planes)
CASES = [
    ((2, 1, [16, 16], [4, 4], 128), 4, 0, 1, 0),                   # QKVG
    ((3, 2, [5, 0, 7], [3, 2, 1], 64), 4, 2, 0, 8),                # k before q, not adjacent
    ((5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128), 5, 3, 4, 0),
    ((2, 1, [7, 2], [3, 1], 8), 2, 1, 0, 8),                       # two planes, k first
    ((1, 1, [50], [4], 256), 3, 0, 1, 0),                          # the QKV layout
    ((4, 2, [3, 1, 0, 2], [1, 0, 2, 1], 16), 6, 5, 2, 16),
    ((8, 1, [64] * 8, [5] * 8, 128), 8, 1, 2, 24),                 # eight planes
    ((2, 1, [75000, 600], [1, 1], 128), 4, 0, 1, 0),               # positions to 75,599
    ((2, 1, [3, 2], [64, 64], 128), 3, 1, 0, 0),                   # wide rows: fewer CTAs per SM
    # equal head groups: the shapes the row-block (tensor-map) kernel takes
    ((3, 2, [5, 0, 7], [2, 2, 2], 64), 4, 2, 0, 8),
    ((4, 2, [3, 1, 0, 2], [1, 1, 1, 1], 16), 6, 5, 2, 16),
    ((8, 1, [37, 41, 29, 33, 40, 35, 31, 38], [5] * 8, 128), 3, 0, 1, 0),
    ((4, 1, [300, 280, 310, 290], [4] * 4, 128), 5, 3, 1, 8),
]

ENGINES = {"tokens": B.ULY_ENGINE_TMA, "tensor": B.ULY_ENGINE_TENSOR}


def _packed_inputs(g, planes, extra, seed, dtype=torch.bfloat16):
    W, b, seq, heads, d = g
    N = sum(heads)
    pitch = planes * N * d + extra
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    xs = [torch.randn((b, s, pitch), generator=gen).to(dtype).cuda() for s in seq]
    return xs, pitch


def _plane(xs, c, N, d):
    """Plane c of every rank's packed input, as (b, s_q, N, d) host bit patterns."""
    return [np.ascontiguousarray(host_raw(x)[:, :, c * N * d:(c + 1) * N * d])
            .reshape(x.shape[0], x.shape[1], N, d) for x in xs]


def run_packed(g, planes, q_plane, k_plane, xs, pitch_elems, w, dtype=torch.bfloat16, cap=None,
               half=False, engine=B.ULY_ENGINE_AUTO):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "float16" if dtype == torch.float16 else "bfloat16")
    B.ulysses_plan_set_fused_engine(plan, engine)
    if half:
        B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    outs = [GuardedOutputs([(b, sum(seq), n, d) for n in heads], dtype) for _ in range(planes)]
    B.ulysses_a2a_4d_packed_fused(plan, planes, q_plane, k_plane, pitch_elems * 2, xs,
                                  [o.tensors for o in outs], w, EPS, THETA)
    torch.cuda.synchronize()
    assert all(o.guards_intact() for o in outs), "a kernel wrote outside its output"
    return [o.tensors for o in outs]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("case", CASES, ids=[f"p{i}" for i in range(len(CASES))])
def test_packed_full(oracle, case, engine):
    g, planes, qp, kp, extra = case
    W, b, seq, heads, d = g
    xs, pitch = _packed_inputs(g, planes, extra, seed=sum(seq) + planes)
    w = wl.rms_weights(d, seed=planes + 1).cuda()
    outs = run_packed(g, planes, qp, kp, xs, pitch, w, engine=ENGINES[engine])
    wn = w.cpu().numpy().astype(np.float64)
    qo, ko, plain = oracle.packed_fused([host_raw(x) for x in xs], seq, heads, d, planes, qp, kp,
                                        pitch, wn[0], wn[1], EPS, THETA)
    for r in range(W):
        check_close(oracle, host_raw(outs[qp][r]), qo[r], f"{case} q rank {r}")
        check_close(oracle, host_raw(outs[kp][r]), ko[r], f"{case} k rank {r}")
        for c in range(planes):
            if c not in (qp, kp):
                assert np.array_equal(host_raw(outs[c][r]), plain[c][r]), f"{case} plane {c} rank {r}"


@pytest.mark.parametrize("engine", list(ENGINES))
def test_packed_matches_separate_calls(engine):
    """QKVG packed in one tensor gives, byte for byte, what the separate fused call on its q and k
    planes and mode 0 of its v and g planes give, on either kernel."""
    g = (8, 1, [300] * 8, [5] * 8, 128)
    W, b, seq, heads, d = g
    N = sum(heads)
    xs, pitch = _packed_inputs(g, 4, 0, seed=41)
    w = wl.rms_weights(d, seed=42).cuda()
    outs = run_packed(g, 4, 0, 1, xs, pitch, w, engine=ENGINES[engine])
    plan = B.ulysses_plan(*g, "bfloat16")
    sl = lambda c: [x[:, :, c * N * d:(c + 1) * N * d].reshape(b, x.shape[1], N, d).contiguous()  # noqa: E731
                    for x in xs]
    ref = [[torch.empty((b, sum(seq), n, d), dtype=torch.bfloat16, device="cuda") for n in heads]
           for _ in range(4)]
    B.ulysses_a2a_4d_qk_fused(plan, sl(0), sl(1), ref[0], ref[1], w, EPS, THETA)
    B.ulysses_a2a_4d(plan, 0, sl(2), ref[2])
    B.ulysses_a2a_4d(plan, 0, sl(3), ref[3])
    torch.cuda.synchronize()
    for c in range(4):
        for a, b_ in zip(outs[c], ref[c]):
            assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), f"plane {c}"


def test_packed_qkv_equals_interleaved_call():
    g = (5, 2, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 64)
    W, b, seq, heads, d = g
    xs, pitch = _packed_inputs(g, 3, 0, seed=43)
    w = wl.rms_weights(d, seed=44).cuda()
    outs = run_packed(g, 3, 0, 1, xs, pitch, w)
    plan = B.ulysses_plan(*g, "bfloat16")
    qkv = [x.view(b, x.shape[1], 3, sum(heads), d) for x in xs]
    ref = [[torch.empty((b, sum(seq), n, d), dtype=torch.bfloat16, device="cuda") for n in heads]
           for _ in range(3)]
    B.ulysses_a2a_4d_qkv_fused(plan, qkv, ref[0], ref[1], ref[2], w, EPS, THETA)
    torch.cuda.synchronize()
    for c in range(3):
        for a, b_ in zip(outs[c], ref[c]):
            assert torch.equal(a.view(torch.int16), b_.view(torch.int16)), f"plane {c}"


@pytest.mark.parametrize("g", [(5, 2, [300, 310, 290, 305, 295], [9, 8, 8, 8, 7], 128),
                               (5, 2, [300, 310, 290, 305, 295], [8] * 5, 128)],
                         ids=["uneven_heads", "equal_heads"])
def test_packed_chunked_equals_unchunked(g):
    xs, pitch = _packed_inputs(g, 4, 16, seed=45)
    w = wl.rms_weights(g[4], seed=46).cuda()
    a = run_packed(g, 4, 2, 0, xs, pitch, w)
    c = run_packed(g, 4, 2, 0, xs, pitch, w, cap=1 << 20)
    for pa, pc in zip(a, c):
        for x, y in zip(pa, pc):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("g", [(3, 2, [5, 0, 7], [3, 2, 1], 64), (3, 2, [5, 0, 7], [2, 2, 2], 64)],
                         ids=["tokens", "row_blocks"])
@pytest.mark.parametrize("f16,half", [(1, 1), (0, 1), (1, 0)], ids=["f16-half", "bf16-half", "f16-adj"])
def test_packed_variants(oracle, f16, half, g):
    """fp16 elements and rotate-half pairs: the q and k planes against the oracle's variant of the
    fused call on each plane (the oracle's packed form is the planes' slices through it), the
    others byte-exact. Unequal head groups take the token units, equal ones the row blocks."""
    W, b, seq, heads, d = g
    N = sum(heads)
    dtype = torch.float16 if f16 else torch.bfloat16
    xs, pitch = _packed_inputs(g, 4, 8, seed=47, dtype=dtype)
    w = wl.rms_weights(d, seed=48).cuda()
    outs = run_packed(g, 4, 3, 1, xs, pitch, w, dtype=dtype, half=bool(half))
    wn = w.cpu().numpy().astype(np.float64)
    rel = 2.0 ** -10 if f16 else 2.0 ** -8
    for c, wrow in ((3, wn[0]), (1, wn[1])):
        ref = oracle.qk_fused_var(_plane(xs, c, N, d), seq, heads, wrow, EPS, THETA, f16, half)
        for r in range(W):
            got = oracle.decode(host_raw(outs[c][r]), f16)
            err = np.abs(got - ref[r])
            assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref[r])), f"plane {c} rank {r}"
            assert np.all(err <= rel * np.abs(ref[r]) + 1e-5), f"plane {c} rank {r}: one rounding"
    for c in (0, 2):
        want = oracle.a2a_4d(_plane(xs, c, N, d), seq, heads, 0)
        for r in range(W):
            assert np.array_equal(host_raw(outs[c][r]), want[r]), f"plane {c} rank {r}"


# ---- backward -----------------------------------------------------------------------------------
def _check_dx_pp(oracle, got_u16, ref, what):
    got = oracle.bf16_to_double(got_u16)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {np.nanmax(err):.3e}"
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-4), f"{what}: beyond one rounding"


@pytest.mark.parametrize("case", CASES[:7], ids=[f"pb{i}" for i in range(7)])
def test_packed_backward_full(oracle, case):
    """dpacked (q and k planes within tolerance, the other planes byte-exact, a token's extra
    columns untouched) and dw against the oracle's packed backward."""
    from gpu_util import FILL
    from test_gpu_fused_bwd import check_dw
    g, planes, qp, kp, extra = case
    W, b, seq, heads, d = g
    N, S = sum(heads), sum(seq)
    xs, pitch = _packed_inputs(g, planes, extra, seed=sum(seq) + 7 * planes)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(planes + 100)
    grads = [[torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).cuda() for n in heads]
             for _ in range(planes)]
    w = wl.rms_weights(d, seed=planes + 3).cuda()
    plan = B.ulysses_plan(*g, "bfloat16")
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
    n_rows = b * S * N
    for t in range(2):
        check_dw(dwo.tensors[0][t].cpu().numpy(), ref_dw[t], n_rows, f"{case} dw {t}")


def test_packed_backward_matches_qkv_backward():
    """The packed backward with the QKV packing gives the interleaved call's backward bytes."""
    g = (5, 2, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 64)
    W, b, seq, heads, d = g
    N, S = sum(heads), sum(seq)
    xs, pitch = _packed_inputs(g, 3, 0, seed=51)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(52)
    grads = [[torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).cuda() for n in heads]
             for _ in range(3)]
    w = wl.rms_weights(d, seed=53).cuda()
    plan = B.ulysses_plan(*g, "bfloat16")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    a = [torch.empty_like(x) for x in xs]
    c = [torch.empty_like(x) for x in xs]
    dwa = torch.empty((2, d), dtype=torch.float32, device="cuda")
    dwc = torch.empty_like(dwa)
    B.ulysses_a2a_4d_packed_fused_backward(plan, 3, 0, 1, pitch * 2, a, xs, grads, w, dwa, EPS,
                                           THETA, ws)
    qkv = [x.view(b, x.shape[1], 3, N, d) for x in xs]
    B.ulysses_a2a_4d_qkv_fused_backward(plan, [t.view(b, t.shape[1], 3, N, d) for t in c], qkv,
                                        grads[0], grads[1], grads[2], w, dwc, EPS, THETA, ws)
    torch.cuda.synchronize()
    for x, y in zip(a, c):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(dwa.view(torch.int32), dwc.view(torch.int32))
