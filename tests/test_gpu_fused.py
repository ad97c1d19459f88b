"""GPU parity of the fused QK RMSNorm + RoPE scatter against the CPU oracle (double precision).

Tolerance: elementwise |gpu - ref| <= 1e-2 + 1e-2 * |ref| against the oracle's unrounded double
result (max abs and max rel error 1e-2 read as one allclose bound, since the bf16 output alone
carries up to 2^-8 relative rounding). The tests also hold the result to a tighter bound that the
fp32 arithmetic and one bf16 rounding allow: |gpu - ref| <= 2^-8 * |ref| + 1e-5.
"""
import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, host_raw
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def check_close(oracle, got_bf16_u16: np.ndarray, ref: np.ndarray, what: str):
    got = oracle.bf16_to_double(got_bf16_u16)
    assert got.shape == ref.shape, what
    if ref.size == 0:
        return 0.0
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {err.max():.3e}"
    tight = err <= 2.0 ** -8 * np.abs(ref) + 1e-5
    assert tight.all(), f"{what}: {int((~tight).sum())} elements beyond one bf16 rounding"
    return float(err.max())


# the fused forward's kernels: token units and row blocks per head group (tensor maps)
ENGINES = {"tokens": B.ULY_ENGINE_TMA, "tensor": B.ULY_ENGINE_TENSOR}


def run_fused(g, q_in, k_in, w, cap=None, engine=B.ULY_ENGINE_AUTO):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    B.ulysses_plan_set_fused_engine(plan, engine)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    shapes = [(b, sum(seq), n, d) for n in heads]
    qo = GuardedOutputs(shapes, torch.bfloat16)
    ko = GuardedOutputs(shapes, torch.bfloat16)
    B.ulysses_a2a_4d_qk_fused(plan, q_in, k_in, qo.tensors, ko.tensors, w, EPS, THETA)
    torch.cuda.synchronize()
    assert qo.guards_intact() and ko.guards_intact(), "a kernel wrote outside its output"
    return qo.tensors, ko.tensors


def make_inputs(g, seed):
    W, b, seq, heads, d = g
    N = sum(heads)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = [torch.randn((b, s, N, d), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    k = [torch.randn((b, s, N, d), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    w = wl.rms_weights(d, seed=seed + 1).cuda()
    return q, k, w


SMALL = [
    (2, 1, [16, 16], [4, 4], 128),
    (3, 2, [5, 0, 7], [3, 2, 1], 64),
    (8, 1, [64] * 8, [5] * 8, 128),
    (5, 1, [30, 31, 29, 30, 30], [9, 8, 8, 8, 7], 128),
    (1, 1, [50], [4], 256),
    (4, 2, [3, 1, 0, 2], [1, 0, 2, 1], 16),
    (4, 1, [3, 4, 5, 6], [2, 2, 1, 3], 32),
    (2, 1, [7, 2], [3, 1], 8),
    (2, 1, [75000, 600], [1, 1], 128),   # positions up to 75,599 on every pair
    (2, 1, [3, 2], [64, 64], 128),       # 64 KiB per token of q and k: fewer CTAs per SM
    (1, 1, [4], [100], 256),             # 100 KiB per token: one CTA per SM
    # equal head groups: the shapes the row-block (tensor-map) kernel takes; others fall back
    (3, 2, [5, 0, 7], [2, 2, 2], 64),
    (4, 1, [3, 4, 5, 6], [2, 2, 2, 2], 32),
    (2, 1, [7, 2], [3, 3], 8),
    (4, 2, [3, 1, 0, 2], [1, 1, 1, 1], 16),
    (5, 2, [300, 310, 290, 305, 295], [8] * 5, 128),
    (8, 1, [1000, 999, 1001, 998, 1002, 997, 1003, 1000], [5] * 8, 128),
    (4, 2, [20, 25, 0, 30], [3, 0, 5, 2], 128),  # unequal head groups with an empty one
]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("g", SMALL, ids=[f"f{i}" for i in range(len(SMALL))])
def test_fused_full(oracle, g, engine):
    W, b, seq, heads, d = g
    q, k, w = make_inputs(g, seed=sum(seq) + d)
    qo, ko = run_fused(g, q, k, w, engine=ENGINES[engine])
    wn = w.cpu().numpy().astype(np.float64)
    for name, xin, out, wrow in (("q", q, qo, wn[0]), ("k", k, ko, wn[1])):
        ref = oracle.qk_fused_A([host_raw(x) for x in xin], seq, heads, wrow, EPS, THETA)
        for r in range(W):
            check_close(oracle, host_raw(out[r]), ref[r], f"{g} {name} rank {r}")


def test_fused_wan720p_sampled(oracle):
    """W=8, b=1, 75,600 tokens, 40 heads, d=128, bf16 q (seed 3) and k (seed 4), weights
    N(1, 0.1) (seed 2), eps 1e-6, theta 1e4, in the launch configuration the benchmark times:
    4,000 sampled output rows per tensor against the oracle's single-row rule, plus every row of
    rank 7's first and last 64 positions."""
    cfg = wl.FUSED
    g = (cfg.W, cfg.b, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    q = wl.seq_side_inputs(cfg, "cuda", seed=cfg.seed)
    k = wl.seq_side_inputs(cfg, "cuda", seed=cfg.extra["k_seed"])
    w = wl.rms_weights(cfg.d, seed=cfg.extra["w_seed"]).cuda()
    qo, ko = run_fused(g, q, k, w)
    wn = w.cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(5)
    for name, xin, out, wrow in (("q", q, qo, wn[0]), ("k", k, ko, wn[1])):
        xh = [host_raw(x) for x in xin]
        oh = [host_raw(o) for o in out]
        rows = [(int(rng.integers(0, cfg.W)), int(rng.integers(0, cfg.S))) for _ in range(4000)]
        rows += [(7, s) for s in list(range(64)) + list(range(cfg.S - 64, cfg.S))]
        for r, s in rows:
            h = int(rng.integers(0, cfg.head_splits[r]))
            ref = oracle.qk_fused_row(xh, g[2], g[3], wrow, EPS, THETA, r, 0, s, h)
            check_close(oracle, oh[r][0, s, h], ref, f"{name} r={r} s={s} h={h}")


def test_fused_long_sequence_sampled(oracle):
    """The long packed-QKV geometry (W=4, 250,000 tokens, 56 heads, d=128: 896,000,000 bytes per
    rank and tensor), positions up to 249,999: 1,000 sampled rows per tensor plus every head of
    the last 16 positions, each against the oracle's single-row rule."""
    cfg = wl.LONG_QKV
    g = (cfg.W, cfg.b, list(cfg.seq_splits), list(cfg.head_splits), cfg.d)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(13)
    q = [torch.randn((1, s, cfg.N, cfg.d), generator=gen, device="cuda").to(torch.bfloat16)
         for s in cfg.seq_splits]
    k = [torch.randn((1, s, cfg.N, cfg.d), generator=gen, device="cuda").to(torch.bfloat16)
         for s in cfg.seq_splits]
    w = wl.rms_weights(cfg.d, seed=14).cuda()
    qo, ko = run_fused(g, q, k, w)
    wn = w.cpu().numpy().astype(np.float64)
    seq_off = np.cumsum([0] + list(cfg.seq_splits))
    head_off = np.cumsum([0] + list(cfg.head_splits))
    rng = np.random.default_rng(15)
    picks = [(int(rng.integers(0, cfg.S)), int(rng.integers(0, cfg.N))) for _ in range(1000)]
    picks += [(p, h) for p in range(cfg.S - 16, cfg.S) for h in range(cfg.N)]
    for t, (xin, out) in enumerate(((q, qo), (k, ko))):
        for p, hg in picks:
            qr = int(np.searchsorted(seq_off, p, side="right") - 1)
            r = int(np.searchsorted(head_off, hg, side="right") - 1)
            raw = host_raw(xin[qr][0, p - seq_off[qr], hg])
            ref = oracle.fused_row_var(raw, 0, 0, wn[t], EPS, p, THETA)
            check_close(oracle, host_raw(out[r][0, p, hg - head_off[r]]), ref, f"t{t} p={p} h={hg}")


@pytest.mark.parametrize("g", [(5, 2, [300, 310, 290, 305, 295], [9, 8, 8, 8, 7], 128),
                               (5, 2, [300, 310, 290, 305, 295], [8] * 5, 128)],
                         ids=["uneven_heads", "equal_heads"])
@pytest.mark.parametrize("engine", list(ENGINES))
def test_fused_chunked_equals_unchunked(engine, g):
    q, k, w = make_inputs(g, seed=9)
    qa, ka = run_fused(g, q, k, w, engine=ENGINES[engine])
    qb, kb = run_fused(g, q, k, w, cap=1 << 20, engine=ENGINES[engine])
    for a, b in zip(qa + ka, qb + kb):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("g", [SMALL[2], SMALL[8], SMALL[-1], (3, 2, [37, 0, 41], [2, 2, 2], 64),
                               (1, 1, [50], [4], 256)],
                         ids=["wan_like", "long_positions", "w8_1000", "zero_split_b2", "run_2048"])
def test_fused_engines_give_the_same_bytes(g):
    """The token-unit and tensor-map kernels compute the same fp32 arithmetic per head row, so
    their outputs are equal bit for bit."""
    q, k, w = make_inputs(g, seed=21)
    qa, ka = run_fused(g, q, k, w, engine=B.ULY_ENGINE_TMA)
    qb, kb = run_fused(g, q, k, w, engine=B.ULY_ENGINE_TENSOR)
    for a, b in zip(qa + ka, qb + kb):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("g", [(5, 2, [300, 310, 290, 305, 295], [9, 8, 8, 8, 7], 128),
                               (3, 1, [4, 0, 3], [2, 1, 1], 64),
                               (5, 2, [300, 310, 290, 305, 295], [8] * 5, 128),
                               (3, 1, [4, 0, 3], [2, 2, 2], 64)],
                         ids=["uneven_b2", "zero_split", "equal_b2", "equal_zero_split"])
def test_fused_host_buffers_match_device_path(oracle, g):
    """The chunked host-buffer fused call gives the device call's bytes exactly (twice in a row),
    on either kernel."""
    W, b, seq, heads, d = g
    q, k, w = make_inputs(g, seed=11)
    qa, ka = run_fused(g, q, k, w, engine=B.ULY_ENGINE_TMA)
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    B.ulysses_plan_set_fused_engine(plan, B.ULY_ENGINE_TENSOR)
    hq = [x.cpu().pin_memory() for x in q]
    hk = [x.cpu().pin_memory() for x in k]
    hqo = [torch.zeros(t.shape, dtype=torch.bfloat16).pin_memory() for t in qa]
    hko = [torch.zeros(t.shape, dtype=torch.bfloat16).pin_memory() for t in ka]
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dqo = [torch.empty_like(t) for t in qa]
    dko = [torch.empty_like(t) for t in ka]
    for _ in range(2):
        B.ulysses_a2a_4d_qk_fused_host(plan, hq, hk, hqo, hko, dq, dk, dqo, dko, w, EPS, THETA)
        torch.cuda.synchronize()
        for h, dev in zip(hqo + hko, qa + ka):
            assert torch.equal(h.view(torch.int16), dev.cpu().view(torch.int16))


def test_fused_zero_rows_stay_zero():
    """All-zero head rows normalise to zero (eps > 0) and stay zero under rotation."""
    g = (2, 1, [5, 3], [2, 2], 128)
    q = [torch.zeros((1, s, 4, 128), dtype=torch.bfloat16, device="cuda") for s in g[2]]
    k = [torch.zeros_like(x) for x in q]
    w = wl.rms_weights(128).cuda()
    for engine in ENGINES.values():
        qo, ko = run_fused(g, q, k, w, engine=engine)
        for t in qo + ko:
            assert torch.count_nonzero(t.float()) == 0
