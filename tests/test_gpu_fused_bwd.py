"""GPU parity of the fused QK backward (RMSNorm + RoPE vector-Jacobian product inside the mode-1
gather) against the CPU oracle (double precision).

dx tolerance: |gpu - ref| <= 1e-2 + 1e-2 * |ref| (the forward's bound), and the tighter bound the
fp32 arithmetic and one bf16 rounding allow at these magnitudes (inputs and gradients of unit
scale): |gpu - ref| <= 2^-8 * |ref| + 1e-4.
dw tolerance (dw_bound): dw is a sum over n = b * S * N rows of terms of unit scale with mean
zero (independent N(0, 1) inputs and gradients), accumulated in fp32 in blocks: each lane adds the
terms of the m rows it handles in sequence, then lanes, warps and CTAs are added in a fixed tree.
The rounding of such a sum behaves like a random walk whose steps scale with the partial sums,
about 2^-24 sigma sqrt(n m / 6) in all (sigma the terms' rms, about 1): 1.5e-3 at the Wan shape
(n = 3,024,000, m about 1,250). The tests allow min(n 2^-20, 1e-4 sqrt(n)) + 1e-4: at the Wan
shape 0.17, over 100 times that, and it stays above it for chains up to about 10^6 rows; while one
row dropped or counted twice moves some element of dw by that row's largest term, u_j xh_j, which
for a row of 128 unit-scale products exceeds 0.17 with overwhelming probability (the full-size
tests check it on sampled rows).
"""
import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from test_gpu_fused import EPS, SMALL, THETA, make_inputs
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def check_dx(oracle, got_bf16_u16, ref, what):
    got = oracle.bf16_to_double(got_bf16_u16)
    assert got.shape == ref.shape, what
    if ref.size == 0:
        return
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {err.max():.3e}"
    tight = err <= 2.0 ** -8 * np.abs(ref) + 1e-4
    assert tight.all(), f"{what}: {int((~tight).sum())} elements beyond the fp32 + bf16 bound"


def dw_bound(n_rows):
    """Allowed |gpu - oracle| for each element of dw, a sum over n_rows rows (module docstring)."""
    return min(n_rows * 2.0 ** -20, 1e-4 * float(np.sqrt(n_rows))) + 1e-4


def check_dw(got, ref, n_rows, what):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    bound = dw_bound(n_rows)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e} > {bound:.3e}"


def make_grads(g, seed, device="cuda"):
    W, b, seq, heads, d = g
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    S = sum(seq)
    return ([torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).to(device) for n in heads],
            [torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).to(device) for n in heads])


# the backward's units follow the plan's fused-kernel setting: token units, or row blocks
# grouped by head group (plans with equal head groups)
ENGINES = {"tokens": B.ULY_ENGINE_TMA, "row_blocks": B.ULY_ENGINE_TENSOR}


def run_bwd(g, q, k, dq, dk, w, cap=None, workspace=None, engine=B.ULY_ENGINE_AUTO):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    B.ulysses_plan_set_fused_engine(plan, engine)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    shapes = [(b, s, sum(heads), d) for s in seq]
    dqo = GuardedOutputs(shapes, torch.bfloat16)
    dko = GuardedOutputs(shapes, torch.bfloat16)
    dwo = GuardedOutputs([(2, d)], torch.float32)
    if workspace is None:
        nbytes = B.ulysses_qk_fused_backward_workspace(plan)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dqo.tensors, dko.tensors, q, k, dq, dk, w,
                                       dwo.tensors[0], EPS, THETA, workspace)
    torch.cuda.synchronize()
    assert dqo.guards_intact() and dko.guards_intact() and dwo.guards_intact(), \
        "a kernel wrote outside its output"
    return dqo.tensors, dko.tensors, dwo.tensors[0]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("g", SMALL, ids=[f"bwd{i}" for i in range(len(SMALL))])
def test_backward_small(oracle, g, engine):
    """Every element of dq, dk and dw against the oracle, over several tiles and ragged tails
    (token blocks of up to 160 tokens at small N * d), empty shards and head groups, d 8..256,
    and positions up to 75,599."""
    W, b, seq, heads, d = g
    q, k, w = make_inputs(g, seed=sum(seq) + 3 * d)
    dq, dk = make_grads(g, seed=7 * sum(heads) + d)
    dqo, dko, dwo = run_bwd(g, q, k, dq, dk, w, engine=ENGINES[engine])
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = b * sum(seq) * sum(heads)
    for t, (x, gy, got) in enumerate(((q, dq, dqo), (k, dk, dko))):
        ref_dx, ref_dw = oracle.qk_fused_bwd([host_raw(v) for v in x], [host_raw(v) for v in gy],
                                             seq, heads, wn[t], EPS, THETA)
        for r in range(W):
            check_dx(oracle, host_raw(got[r]), ref_dx[r], f"{g} tensor {t} rank {r}")
        check_dw(dwo[t].cpu().numpy(), ref_dw, n_rows, f"{g} dw {t}")


@pytest.mark.parametrize("g", [(5, 2, [100, 110, 90, 105, 95], [9, 8, 8, 8, 7], 128),
                               (5, 2, [100, 110, 90, 105, 95], [8] * 5, 128)],
                         ids=["uneven_heads", "equal_heads"])
def test_backward_chunked_matches_unchunked(oracle, g):
    """Chunking changes no dx byte; dw (summed in another order) stays within the bound."""
    q, k, w = make_inputs(g, seed=11)
    dq, dk = make_grads(g, seed=12)
    a = run_bwd(g, q, k, dq, dk, w)
    c = run_bwd(g, q, k, dq, dk, w, cap=1 << 20)
    t = run_bwd(g, q, k, dq, dk, w, engine=B.ULY_ENGINE_TMA)  # token units: dx the same bytes
    for x, y in zip(a[0] + a[1], t[0] + t[1]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for x, y in zip(a[0] + a[1], c[0] + c[1]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    n_rows = 2 * sum(g[2]) * sum(g[3])
    check_dw(c[2].cpu().numpy(), a[2].cpu().numpy().astype(np.float64), n_rows, "chunked dw")


def test_backward_deterministic():
    """Two calls in a row (the second reusing the first's workspace) give identical bytes,
    dw included: its sums do not depend on timing."""
    g = (8, 1, [300] * 8, [5] * 8, 128)
    q, k, w = make_inputs(g, seed=21)
    dq, dk = make_grads(g, seed=22)
    plan = B.ulysses_plan(*g, "bfloat16")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    a = run_bwd(g, q, k, dq, dk, w, workspace=ws)
    c = run_bwd(g, q, k, dq, dk, w, workspace=ws)
    for x, y in zip(a[0] + a[1], c[0] + c[1]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(a[2].view(torch.int32), c[2].view(torch.int32))


def test_backward_workspace_and_argument_checks():
    g = (2, 1, [16, 16], [4, 4], 128)
    W, b, seq, heads, d = g
    q, k, w = make_inputs(g, seed=31)
    dq, dk = make_grads(g, seed=32)
    plan = B.ulysses_plan(*g, "bfloat16")
    need = B.ulysses_qk_fused_backward_workspace(plan)
    assert need >= 2 * d * 4
    dqo = [torch.empty_like(x) for x in q]
    dko = [torch.empty_like(x) for x in k]
    dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
    short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.UlyssesError):
        B.ulysses_a2a_4d_qk_fused_backward(plan, dqo, dko, q, k, dq, dk, w, dw, EPS, THETA, short)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.UlyssesError):  # dq output on top of the forward input
        B.ulysses_a2a_4d_qk_fused_backward(plan, q, dko, q, k, dq, dk, w, dw, EPS, THETA, ws)
    with pytest.raises(B.UlyssesError):  # dw inside the workspace
        B.ulysses_a2a_4d_qk_fused_backward(plan, dqo, dko, q, k, dq, dk, w,
                                           ws[:2 * d * 4].view(torch.float32), EPS, THETA, ws)
    fp32 = B.ulysses_plan(*g, "float32")
    with pytest.raises(B.UlyssesError):
        B.ulysses_qk_fused_backward_workspace(fp32)


def _wan_inputs(seed):
    cfg = wl.WAN
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = [[torch.randn((1, s, cfg.N, cfg.d), generator=gen, device="cuda").to(torch.bfloat16)
          for s in cfg.seq_splits] for _ in range(2)]
    return cfg, x, wl.rms_weights(cfg.d, seed=seed + 1).cuda()


def test_backward_wan720p_sampled(oracle):
    """W=8, b=1, 75,600 tokens, 40 heads, d=128, in the launch configuration the bench times:
    1,000 sampled rows of dq and of dk against the oracle's single-row backward."""
    cfg, (q, k), w = _wan_inputs(51)
    g = (cfg.W, 1, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    dq, dk = make_grads(g, seed=52)
    dqo, dko, _ = run_bwd(g, q, k, dq, dk, w)
    wn = w.cpu().numpy().astype(np.float64)
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(53)
    for t, (x, gy, got) in enumerate(((q, dq, dqo), (k, dk, dko))):
        for _ in range(500):
            qr = int(rng.integers(0, cfg.W))
            i = int(rng.integers(0, cfg.seq_splits[qr]))
            hg = int(rng.integers(0, cfg.N))
            r = int(np.searchsorted(head_off, hg, side="right") - 1)
            xrow = oracle.bf16_to_double(host_raw(x[qr][0, i, hg]))
            grow = oracle.bf16_to_double(host_raw(gy[r][0, seq_off[qr] + i, hg - head_off[r]]))
            ref, _ = oracle.fused_row_bwd(xrow, grow, wn[t], EPS, seq_off[qr] + i, THETA)
            check_dx(oracle, host_raw(got[qr][0, i, hg]), ref, f"tensor {t} q={qr} i={i} h={hg}")


def test_backward_long_sequence_sampled(oracle):
    """The long packed-QKV geometry (W=4, 250,000 tokens, 56 heads, d=128), positions up to
    249,999: 600 sampled rows of dq and of dk against the oracle's single-row backward."""
    cfg = wl.LONG_QKV
    g = (cfg.W, 1, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(71)
    bf = lambda shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)  # noqa: E731
    q = [bf((1, s, cfg.N, cfg.d)) for s in cfg.seq_splits]
    k = [bf((1, s, cfg.N, cfg.d)) for s in cfg.seq_splits]
    dq = [bf((1, cfg.S, n, cfg.d)) for n in cfg.head_splits]
    dk = [bf((1, cfg.S, n, cfg.d)) for n in cfg.head_splits]
    w = wl.rms_weights(cfg.d, seed=72).cuda()
    dqo, dko, _ = run_bwd(g, q, k, dq, dk, w)
    wn = w.cpu().numpy().astype(np.float64)
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(73)
    for t, (x, gy, got) in enumerate(((q, dq, dqo), (k, dk, dko))):
        for _ in range(300):
            p = int(rng.integers(cfg.S - 2000, cfg.S)) if rng.random() < 0.5 else int(rng.integers(0, cfg.S))
            hg = int(rng.integers(0, cfg.N))
            qr = int(np.searchsorted(seq_off, p, side="right") - 1)
            r = int(np.searchsorted(head_off, hg, side="right") - 1)
            i = p - seq_off[qr]
            xrow = oracle.bf16_to_double(host_raw(x[qr][0, i, hg]))
            grow = oracle.bf16_to_double(host_raw(gy[r][0, p, hg - head_off[r]]))
            ref, _ = oracle.fused_row_bwd(xrow, grow, wn[t], EPS, p, THETA)
            check_dx(oracle, host_raw(got[qr][0, i, hg]), ref, f"tensor {t} p={p} h={hg}")


def test_backward_wan720p_sparse_gradient(oracle):
    """Full size with the output gradient zero except on 2,000 random rows: every dx row without
    a gradient is exactly zero, the others match the oracle's row backward, and dw equals the
    oracle's sum over those rows alone (a property that holds at any size)."""
    cfg, (q, k), w = _wan_inputs(61)
    g = (cfg.W, 1, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(62)
    dq = [torch.zeros((1, cfg.S, n, cfg.d), dtype=torch.bfloat16, device="cuda")
          for n in cfg.head_splits]
    dk = [torch.zeros_like(t) for t in dq]
    picks = set()
    while len(picks) < 2000:
        picks.add((int(rng.integers(0, 2)), int(rng.integers(0, cfg.S)), int(rng.integers(0, cfg.N))))
    picks = sorted(picks)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(63)
    rows = torch.randn((len(picks), cfg.d), generator=gen).to(torch.bfloat16)
    for (t, s, hg), row in zip(picks, rows):
        r = int(np.searchsorted(head_off, hg, side="right") - 1)
        (dq, dk)[t][r][0, s, hg - head_off[r]] = row.cuda()
    dqo, dko, dwo = run_bwd(g, q, k, dq, dk, w)
    wn = w.cpu().numpy().astype(np.float64)
    dw_ref = np.zeros((2, cfg.d))
    hit = [np.zeros((cfg.S, cfg.N), dtype=bool) for _ in range(2)]
    for (t, s, hg), row in zip(picks, rows):
        qr = int(np.searchsorted(seq_off, s, side="right") - 1)
        i = s - seq_off[qr]
        x = (q, k)[t][qr][0, i, hg]
        ref_dx, ref_dw = oracle.fused_row_bwd(oracle.bf16_to_double(host_raw(x)),
                                              oracle.bf16_to_double(host_raw(row)), wn[t], EPS, s,
                                              THETA)
        dw_ref[t] += ref_dw
        hit[t][s, hg] = True
        check_dx(oracle, host_raw((dqo, dko)[t][qr][0, i, hg]), ref_dx, f"tensor {t} s={s} h={hg}")
    for t, got in enumerate((dqo, dko)):
        whole = torch.cat([x[0] for x in got], dim=0).float()       # (S, N, d)
        mask = torch.from_numpy(~hit[t]).cuda()
        assert bool((whole[mask] == 0).all()), f"tensor {t}: a row without gradient is not zero"
    check_dw(dwo.cpu().numpy(), dw_ref, len(picks), "sparse dw")
