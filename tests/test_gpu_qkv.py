"""GPU parity of the interleaved packed QKV call against the CPU oracle: q and k within the fused
tolerance (and one bf16 rounding of the exact result), v bit-exact."""
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


def run_qkv(g, qkv, w, cap=None):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    shapes = [(b, sum(seq), n, d) for n in heads]
    outs = [GuardedOutputs(shapes, torch.bfloat16) for _ in range(3)]
    B.ulysses_a2a_4d_qkv_fused(plan, qkv, outs[0].tensors, outs[1].tensors, outs[2].tensors, w,
                               EPS, THETA)
    torch.cuda.synchronize()
    assert all(o.guards_intact() for o in outs), "a kernel wrote outside its output"
    return [o.tensors for o in outs]


def make_qkv(g, seed):
    W, b, seq, heads, d = g
    N = sum(heads)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    qkv = [torch.randn((b, s, 3, N, d), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    return qkv, wl.rms_weights(d, seed=seed + 1).cuda()


GEOMS = [
    (2, 1, [16, 16], [4, 4], 128),
    (3, 2, [5, 0, 7], [3, 2, 1], 64),
    (8, 1, [64] * 8, [5] * 8, 128),
    (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128),
    (4, 1, [3, 4, 5, 6], [2, 2, 1, 3], 32),
    (1, 1, [9], [3], 256),
    (2, 1, [3, 2], [48, 48], 128),   # 72 KiB per token of q, k and v: fewer CTAs per SM
]


@pytest.mark.parametrize("g", GEOMS, ids=[f"qkv{i}" for i in range(len(GEOMS))])
def test_qkv_full(oracle, g):
    W, b, seq, heads, d = g
    qkv, w = make_qkv(g, seed=sum(seq) + d)
    qo, ko, vo = run_qkv(g, qkv, w)
    wn = w.cpu().numpy().astype(np.float64)
    rq, rk, rv = oracle.qkv_fused([host_raw(x) for x in qkv], seq, heads, wn[0], wn[1], EPS, THETA)
    for r in range(W):
        check_close(oracle, host_raw(qo[r]), rq[r], f"{g} q rank {r}")
        check_close(oracle, host_raw(ko[r]), rk[r], f"{g} k rank {r}")
        assert np.array_equal(host_raw(vo[r]), rv[r]), f"{g} v rank {r}"


def test_qkv_matches_separate_calls():
    """Interleaved in one launch == the separate fused q,k call plus mode 0 on v, byte for byte."""
    g = (8, 1, [300] * 8, [5] * 8, 128)
    W, b, seq, heads, d = g
    qkv, w = make_qkv(g, seed=5)
    qo, ko, vo = run_qkv(g, qkv, w)
    q = [x[:, :, 0].contiguous() for x in qkv]
    k = [x[:, :, 1].contiguous() for x in qkv]
    v = [x[:, :, 2].contiguous() for x in qkv]
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    q2 = [torch.empty_like(t) for t in qo]
    k2 = [torch.empty_like(t) for t in ko]
    v2 = [torch.empty_like(t) for t in vo]
    B.ulysses_a2a_4d_qk_fused(plan, q, k, q2, k2, w, EPS, THETA)
    B.ulysses_a2a_4d(plan, 0, v, v2)
    torch.cuda.synchronize()
    for a, b_ in zip(qo + ko + vo, q2 + k2 + v2):
        assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


def test_qkv_chunked_equals_unchunked():
    g = (5, 2, [100, 110, 90, 105, 95], [9, 8, 8, 8, 7], 128)
    qkv, w = make_qkv(g, seed=8)
    a = run_qkv(g, qkv, w)
    b = run_qkv(g, qkv, w, cap=1 << 20)
    for x, y in zip(sum(a, []), sum(b, [])):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_qkv_wan720p_sampled(oracle):
    """W=8, b=1, 75,600 tokens, 40 heads, d=128: 1,000 sampled rows per plane against the
    oracle's single-row rule (q, k) and single-element rule (v)."""
    cfg = wl.WAN
    g = (cfg.W, cfg.b, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(41)
    qkv = [torch.randn((1, s, 3, cfg.N, cfg.d), generator=gen, device="cuda").to(torch.bfloat16)
           for s in cfg.seq_splits]
    w = wl.rms_weights(cfg.d, seed=2).cuda()
    qo, ko, vo = run_qkv(g, qkv, w)
    wn = w.cpu().numpy().astype(np.float64)
    xh = [host_raw(x) for x in qkv]
    planes = [[np.ascontiguousarray(x[:, :, c]) for x in xh] for c in range(3)]
    oh = [[host_raw(o) for o in outs] for outs in (qo, ko, vo)]
    rng = np.random.default_rng(9)
    for _ in range(1000):
        r, s = int(rng.integers(0, cfg.W)), int(rng.integers(0, cfg.S))
        h = int(rng.integers(0, cfg.head_splits[r]))
        for c, wrow in ((0, wn[0]), (1, wn[1])):
            ref = oracle.qk_fused_row(planes[c], g[2], g[3], wrow, EPS, THETA, r, 0, s, h)
            check_close(oracle, oh[c][r][0, s, h], ref, f"plane {c} r={r} s={s} h={h}")
        flat = (s * cfg.head_splits[r] + h) * cfg.d
        q, idx = oracle.a2a_4d_source(cfg.W, 1, g[2], g[3], cfg.d, 0, r, flat)
        assert np.array_equal(oh[2][r].reshape(-1)[flat:flat + cfg.d],
                              planes[2][q].reshape(-1)[idx:idx + cfg.d])


# ---- backward of the interleaved call ------------------------------------------------------------
def _qkv_bwd(g, qkv, gq, gk, gv, w, f16=False, half=False, cap=None):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "float16" if f16 else "bfloat16")
    if half:
        B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    dt = torch.float16 if f16 else torch.bfloat16
    out = GuardedOutputs([(b, s, 3, sum(heads), d) for s in seq], dt)
    dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qkv_fused_backward(plan, out.tensors, qkv, gq, gk, gv, w, dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    assert out.guards_intact(), "a kernel wrote outside its output"
    return out.tensors, dw


def _grads3(g, seed, dt):
    W, b, seq, heads, d = g
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    S = sum(seq)
    return [[torch.randn((b, S, n, d), generator=gen).to(dt).cuda() for n in heads] for _ in range(3)]


BWD_GEOMS = [(2, 1, [16, 16], [4, 4], 128), (3, 2, [5, 0, 7], [3, 2, 1], 64),
             (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128), (4, 1, [3, 4, 5, 6], [2, 2, 1, 3], 32),
             (1, 1, [9], [3], 256)]


@pytest.mark.parametrize("variant", [(False, False), (True, True)], ids=["bf16-adjacent", "f16-half"])
@pytest.mark.parametrize("g", BWD_GEOMS, ids=[f"qkvbwd{i}" for i in range(len(BWD_GEOMS))])
def test_qkv_backward(oracle, g, variant):
    """Planes q, k against the oracle's backward of the fused call on those planes; plane v
    against mode 1 of the v gradient, bit for bit; dw within the summation bound."""
    from test_gpu_fused_bwd import check_dw
    f16, half = variant
    W, b, seq, heads, d = g
    dt = torch.float16 if f16 else torch.bfloat16
    gen = torch.Generator(device="cpu")
    gen.manual_seed(sum(seq) + d)
    qkv = [torch.randn((b, s, 3, sum(heads), d), generator=gen).to(dt).cuda() for s in seq]
    w = wl.rms_weights(d, seed=sum(heads)).cuda()
    gq, gk, gv = _grads3(g, seed=3 * d + 1, dt=dt)
    dqkv, dw = _qkv_bwd(g, qkv, gq, gk, gv, w, f16, half)
    wn = w.cpu().numpy().astype(np.float64)
    raw = [host_raw(x) for x in qkv]
    n_rows = b * sum(seq) * sum(heads)
    rel = 2.0 ** -10 if f16 else 2.0 ** -8
    for t, gy in enumerate((gq, gk)):
        planes = [np.ascontiguousarray(x[:, :, t]) for x in raw]
        ref_dx, ref_dw = oracle.qk_fused_bwd_var(planes, [host_raw(v) for v in gy], seq, heads,
                                                 wn[t], EPS, THETA, int(f16), int(half))
        for r in range(W):
            got = oracle.decode(np.ascontiguousarray(host_raw(dqkv[r])[:, :, t]), int(f16))
            err = np.abs(got - ref_dx[r])
            assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref_dx[r])), f"{g} plane {t} rank {r}"
            assert np.all(err <= rel * np.abs(ref_dx[r]) + 1e-4), f"{g} plane {t} rank {r} (tight)"
        check_dw(dw[t].cpu().numpy(), ref_dw, n_rows, f"{g} dw {t}")
    want_v = oracle.a2a_4d([host_raw(x) for x in gv], seq, heads, 1)
    for r in range(W):
        assert np.array_equal(np.ascontiguousarray(host_raw(dqkv[r])[:, :, 2]), want_v[r])


def test_qkv_backward_matches_separate_calls():
    """dq and dk planes equal the separate backward's bytes; dv equals mode 1 of the v gradient;
    chunked equals unchunked."""
    from test_gpu_fused_bwd import check_dw
    g = (8, 1, [300] * 8, [5] * 8, 128)
    W, b, seq, heads, d = g
    qkv, w = make_qkv(g, seed=15)
    gq, gk, gv = _grads3(g, seed=16, dt=torch.bfloat16)
    dqkv, dw = _qkv_bwd(g, qkv, gq, gk, gv, w)
    plan = B.ulysses_plan(*g, "bfloat16")
    q = [x[:, :, 0].contiguous() for x in qkv]
    k = [x[:, :, 1].contiguous() for x in qkv]
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dv = [torch.empty_like(x) for x in q]
    dw2 = torch.empty_like(dw)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw2, EPS, THETA, ws)
    B.ulysses_a2a_4d(plan, 1, gv, dv)
    torch.cuda.synchronize()
    for r in range(W):
        for t, ref in enumerate((dq[r], dk[r], dv[r])):
            assert torch.equal(dqkv[r][:, :, t].contiguous().view(torch.int16), ref.view(torch.int16))
    check_dw(dw.cpu().numpy(), dw2.cpu().numpy().astype(np.float64), sum(seq) * sum(heads), "dw")
    dqkv_c, dw_c = _qkv_bwd(g, qkv, gq, gk, gv, w, cap=1 << 20)
    for a, c in zip(dqkv, dqkv_c):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
