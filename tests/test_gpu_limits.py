"""GPU parity at the library's size limits, through the C ABI against the CPU oracle.

Two limits of the plan are exercised here, each in the launch configurations the library picks
for it (every relayout engine, both fused kernels, one launch per call and the default 1 GiB
chunking):
* tensors past 4 GiB per rank (b = 2, so batch strides alone pass 2^31 bytes): byte offsets that
  need 64-bit arithmetic in every kernel and in the tensor maps;
* the largest sequence the fused calls accept, S = 2^24 - 1 (positions are carried exactly in
  fp32 below 2^24), so RoPE angles p theta^(-2j/d) reach p = 16,777,214 radians at j = 0.

At these sizes the oracle computes sampled outputs one by one (its single-element source rule for
the relayout, its single-row forward and backward for the fused calls), and properties that hold
at any size cover the rest: the mode-1 round trip returns the input bit for bit, and a backward
whose output gradient is zero except on sampled rows must give exactly zero elsewhere and a dw
equal to the sum of those rows' terms. Tolerances are those of the other fused tests: within
1e-2 + 1e-2 |ref| of the oracle's unrounded double, and one rounding of an fp32 result to the
element type (2^-8 |ref| for bf16, 2^-10 |ref| for fp16, plus 1e-5 forward and 1e-4 for dx).
"""
import os

import numpy as np
import pytest
import torch

from test_gpu_fullsize import check_all
from test_gpu_fused_bwd import check_dw
from ulysses_sequence_all_gb300 import binding as B

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4
FOUR_GIB = 1 << 32
ONE_LAUNCH = 1 << 40  # a chunk cap no rank reaches: each call is one launch

RELAYOUT_ENGINES = {"auto": B.ULY_ENGINE_AUTO, "tma": B.ULY_ENGINE_TMA, "vec": B.ULY_ENGINE_VEC,
                    "ce": B.ULY_ENGINE_CE, "tensor": B.ULY_ENGINE_TENSOR}
FUSED_ENGINES = {"tokens": B.ULY_ENGINE_TMA, "row_blocks": B.ULY_ENGINE_TENSOR}
CAPS = {"one_launch": ONE_LAUNCH, "chunked_1GiB": None}

# W, b, seq_splits, head_splits, d (bf16): rank 0 holds 4,505,600,000 bytes on the sequence side
# and 5,376,007,680 on the head side; unequal head groups (runs of 1,280 and 768 bytes)
RELAYOUT_BIG = (2, 2, [1_100_000, 1_000_003], [5, 3], 128)
# equal head groups (the row-block kernel's plans): 4,505,600,000 / 4,505,604,096 bytes per rank
# and tensor on the sequence side, 4,505,601,024 on the head side
FUSED_BIG = (2, 2, [1_100_000, 1_100_001], [4, 4], 128)
S_MAX = (1 << 24) - 1


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"
    torch.cuda.empty_cache()


def _flat16(t: torch.Tensor) -> torch.Tensor:
    return t.reshape(-1).view(torch.int16)


def _side_shapes(g, mode):
    W, b, seq, heads, d = g
    if mode == 0:
        return [(b, sum(seq), n, d) for n in heads]
    return [(b, s, sum(heads), d) for s in seq]


def _plan(g, dtype="bfloat16", cap=None, fused_engine=None, half=False):
    plan = B.ulysses_plan(*g, dtype)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    if fused_engine is not None:
        B.ulysses_plan_set_fused_engine(plan, fused_engine)
    if half:
        B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    return plan


def _sample_indices(rng, n, k_random, k_tail):
    """k_random uniform indices below n plus the last k_tail ones (the far end of the buffer)."""
    idx = np.concatenate([rng.integers(0, n, size=k_random), np.arange(n - k_tail, n)])
    return np.unique(idx)


# ---- relayout -----------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def relayout_big(oracle):
    """Uniform random bytes on the sequence side (NaN patterns included; compared as raw bytes)
    and, per head-side rank, sampled element positions with the values the oracle's
    single-element rule assigns them."""
    W, b, seq, heads, d = RELAYOUT_BIG
    gen = torch.Generator(device="cuda")
    gen.manual_seed(71)
    ins = []
    for sh in _side_shapes(RELAYOUT_BIG, 1):
        n = int(np.prod(sh)) * 2
        ins.append(torch.randint(0, 256, (n,), dtype=torch.uint8, generator=gen,
                                 device="cuda").view(torch.bfloat16).view(sh))
    assert ins[0].numel() * 2 > FOUR_GIB
    flat_in = [_flat16(x) for x in ins]
    rng = np.random.default_rng(72)
    samples = []
    for r, sh in enumerate(_side_shapes(RELAYOUT_BIG, 0)):
        n = int(np.prod(sh))
        ks = _sample_indices(rng, n, 3000, 2000)
        src = [oracle.a2a_4d_source(W, b, seq, heads, d, 0, r, int(k)) for k in ks]
        want = torch.empty(len(ks), dtype=torch.int16, device="cuda")
        for q in range(W):
            sel = [j for j, (sq, _) in enumerate(src) if sq == q]
            if sel:
                idx = torch.as_tensor([src[j][1] for j in sel], device="cuda")
                want[torch.as_tensor(sel, device="cuda")] = flat_in[q][idx]
        samples.append((torch.as_tensor(ks, device="cuda"), want))
    yield ins, samples
    del ins, flat_in, samples
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cap", list(CAPS))
@pytest.mark.parametrize("engine", list(RELAYOUT_ENGINES))
def test_relayout_past_4gib(relayout_big, engine, cap):
    """Mode 0 on ranks of more than 4 GiB: 5,000 sampled elements per head-side rank (among them
    the last 2,000) equal the oracle's; mode 1 of the result returns every input byte."""
    ins, samples = relayout_big
    plan = _plan(RELAYOUT_BIG, cap=CAPS[cap])
    if CAPS[cap] is None:
        assert B.ulysses_plan_num_chunks(plan, 0) >= 5
    else:
        assert B.ulysses_plan_num_chunks(plan, 0) == 1
    outs = [torch.empty(sh, dtype=torch.bfloat16, device="cuda")
            for sh in _side_shapes(RELAYOUT_BIG, 0)]
    for o in outs:
        o.view(torch.int16).fill_(-23131)  # 0xA5A5: an unwritten element fails the compare
    B.ulysses_a2a_4d_engine(plan, 0, RELAYOUT_ENGINES[engine], ins, outs)
    torch.cuda.synchronize()
    for r, (ks, want) in enumerate(samples):
        got = _flat16(outs[r])[ks]
        bad = int((got != want).sum())
        assert bad == 0, f"mode 0 rank {r}: {bad} of {len(ks)} sampled elements differ"
    back = [torch.empty_like(x) for x in ins]
    B.ulysses_a2a_4d_engine(plan, 1, RELAYOUT_ENGINES[engine], outs, back)
    torch.cuda.synchronize()
    del outs
    for q, (a, x) in enumerate(zip(back, ins)):
        assert torch.equal(_flat16(a), _flat16(x)), f"round trip rank {q} differs"


# ---- fused forward ------------------------------------------------------------------------------

def _dtype(f16):
    return torch.float16 if f16 else torch.bfloat16


def _fused_inputs(g, f16, seed):
    """q and k N(0, 1) on the device (per rank, seeded) and RMSNorm weights N(1, 0.1)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    xs = [[torch.randn(sh, dtype=_dtype(f16), generator=gen, device="cuda")
           for sh in _side_shapes(g, 1)] for _ in range(2)]
    wgen = torch.Generator(device="cpu")
    wgen.manual_seed(seed + 1)
    w = (1.0 + 0.1 * torch.randn((2, g[4]), generator=wgen)).float()
    return xs, w.cuda(), w.numpy().astype(np.float64)


def _close(oracle, got_raw, ref, f16, atol, what):
    got = oracle.decode(got_raw, f16)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"{what}: max err {err.max():.3e}"
    rel = 2.0 ** -10 if f16 else 2.0 ** -8
    tight = err <= rel * np.abs(ref) + atol
    assert tight.all(), f"{what}: {int((~tight).sum())} elements beyond one rounding"


def _sample_rows(g, rng, k_random, k_tail):
    """Head-side rows (r, bb, s, h): k_random uniform ones and every row of the last k_tail
    positions of the last batch index."""
    W, b, seq, heads, d = g
    S = sum(seq)
    live = [r for r in range(W) if heads[r] > 0]
    rows = set()
    while len(rows) < k_random:
        r = live[int(rng.integers(0, len(live)))]
        rows.add((r, int(rng.integers(0, b)), int(rng.integers(0, S)), int(rng.integers(0, heads[r]))))
    for r in live:
        for s in range(S - k_tail, S):
            for h in range(heads[r]):
                rows.add((r, b - 1, s, h))
    return sorted(rows)


def _source_rows(oracle, g, rows):
    """For each head-side row (r, bb, s, h), the sequence-side (rank, row index) the oracle's
    single-element rule takes its first element from, and the head-side row index."""
    W, b, seq, heads, d = g
    S = sum(seq)
    out = []
    for r, bb, s, h in rows:
        head_row = (bb * S + s) * heads[r] + h
        q, elem = oracle.a2a_4d_source(W, b, seq, heads, d, 0, r, head_row * d)
        assert elem % d == 0
        out.append((q, elem // d, head_row))
    return out


def _gather_rows(tensors, picks, d):
    """Rows picks[j] = (rank, row index) of per-rank tensors, as one host array (len, d) of raw
    16-bit words."""
    res = torch.empty((len(picks), d), dtype=torch.int16, device="cuda")
    for k, t in enumerate(tensors):
        sel = [j for j, (kk, _) in enumerate(picks) if kk == k]
        if sel:
            idx = torch.as_tensor([picks[j][1] for j in sel], device="cuda")
            res[torch.as_tensor(sel, device="cuda")] = t.reshape(-1, d).view(torch.int16)[idx]
    return res.cpu().numpy().view(np.uint16)


def _check_fused_rows(oracle, g, xs, outs, wn, f16, half, rows, what):
    d = g[4]
    src = _source_rows(oracle, g, rows)
    for t in range(2):
        x_rows = _gather_rows(xs[t], [(q, i) for q, i, _ in src], d)
        got_rows = _gather_rows(outs[t], [(r, hr) for (r, _, _, _), (_, _, hr) in zip(rows, src)], d)
        for j, (r, bb, s, h) in enumerate(rows):
            ref = oracle.fused_row_var(x_rows[j], int(f16), int(half), wn[t], EPS, s, THETA)
            _close(oracle, got_rows[j], ref, f16, 1e-5, f"{what} tensor {t} r={r} bb={bb} s={s} h={h}")


def _run_fused(g, xs, w, f16=False, half=False, engine=B.ULY_ENGINE_AUTO, cap=None, outs=None):
    plan = _plan(g, "float16" if f16 else "bfloat16", cap=cap, fused_engine=engine, half=half)
    if outs is None:
        outs = [[torch.empty(sh, dtype=_dtype(f16), device="cuda") for sh in _side_shapes(g, 0)]
                for _ in range(2)]
    for t in outs:
        for o in t:
            o.view(torch.int16).fill_(-23131)
    B.ulysses_a2a_4d_qk_fused(plan, xs[0], xs[1], outs[0], outs[1], w, EPS, THETA)
    torch.cuda.synchronize()
    return plan, outs


@pytest.mark.parametrize("engine", list(FUSED_ENGINES))
def test_fused_past_4gib(oracle, engine):
    """The fused forward (bf16, adjacent pairs) on ranks of more than 4 GiB per tensor, in one
    launch and chunked: 1,500 sampled rows per tensor plus every row of the last 16 positions of
    batch 1, each against the oracle's single-row rule at the row's global position."""
    g = FUSED_BIG
    xs, w, wn = _fused_inputs(g, False, 81)
    assert xs[0][0].numel() * 2 > FOUR_GIB
    rows = _sample_rows(g, np.random.default_rng(82), 1500, 16)
    outs = None
    for cap in CAPS.values():
        plan, outs = _run_fused(g, xs, w, engine=FUSED_ENGINES[engine], cap=cap, outs=outs)
        assert B.ulysses_plan_fused_kernel(plan) == FUSED_ENGINES[engine]
        _check_fused_rows(oracle, g, xs, outs, wn, False, False, rows, f"cap {cap}")
    del xs, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", list(FUSED_ENGINES))
@pytest.mark.parametrize("f16,half", [(False, False), (True, True)], ids=["bf16-adjacent", "f16-half"])
def test_fused_max_positions_full(oracle, engine, f16, half):
    """S = 2^24 - 1 tokens, the largest the fused calls accept (W=2, one head per rank, d=8):
    every element of both tensors against the oracle, positions 0 .. 16,777,214."""
    g = (2, 1, [1 << 23, (1 << 23) - 1], [1, 1], 8)
    assert sum(g[2]) == S_MAX
    xs, w, wn = _fused_inputs(g, f16, 91)
    plan, outs = _run_fused(g, xs, w, f16=f16, half=half, engine=FUSED_ENGINES[engine])
    assert B.ulysses_plan_fused_kernel(plan) == FUSED_ENGINES[engine]
    threads = max(1, os.cpu_count() or 1)
    for t in range(2):
        xh = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs[t]]
        ref = oracle.qk_fused_var(xh, g[2], g[3], wn[t], EPS, THETA, int(f16), int(half),
                                  threads=threads)
        for r in range(2):
            check_all(outs[t][r], ref[r], 2.0 ** -10 if f16 else 2.0 ** -8, 1e-5,
                      f"tensor {t} rank {r}")
    del xs, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", list(FUSED_ENGINES))
@pytest.mark.parametrize("f16,half", [(False, False), (True, True)], ids=["bf16-adjacent", "f16-half"])
def test_fused_max_positions_sampled(oracle, engine, f16, half):
    """S = 2^24 - 1 tokens at d = 128 (W=2, one head per rank: 4 GiB per rank and tensor on both
    sides): 1,500 sampled rows per tensor plus the last 64 positions, against the oracle's
    single-row rule."""
    g = (2, 1, [1 << 23, (1 << 23) - 1], [1, 1], 128)
    xs, w, wn = _fused_inputs(g, f16, 93)
    assert xs[0][0].numel() * 2 == FOUR_GIB
    plan, outs = _run_fused(g, xs, w, f16=f16, half=half, engine=FUSED_ENGINES[engine])
    assert B.ulysses_plan_fused_kernel(plan) == FUSED_ENGINES[engine]
    rows = _sample_rows(g, np.random.default_rng(94), 1500, 64)
    _check_fused_rows(oracle, g, xs, outs, wn, f16, half, rows, "max positions")
    del xs, outs
    torch.cuda.empty_cache()


# ---- fused backward -----------------------------------------------------------------------------

def _check_sparse_backward(oracle, g, xs, w, wn, f16, half, rows, engine, cap, seed, what):
    """Output gradients zero except on `rows` (N(0, 1) there, both tensors): each picked row's
    dx against the oracle's row backward at its global position, every other dx row exactly
    zero, and dw against the sum of the picked rows' dw terms."""
    d = g[4]
    grads = [[torch.zeros(sh, dtype=_dtype(f16), device="cuda") for sh in _side_shapes(g, 0)]
             for _ in range(2)]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    vals = [torch.randn((len(rows), d), generator=gen).to(_dtype(f16)) for _ in range(2)]
    src = _source_rows(oracle, g, rows)
    for t in range(2):
        for r in range(g[0]):
            sel = [j for j, row in enumerate(rows) if row[0] == r]
            if sel:
                idx = torch.as_tensor([src[j][2] for j in sel], device="cuda")
                grads[t][r].reshape(-1, d)[idx] = vals[t][sel].cuda()
    plan = _plan(g, "float16" if f16 else "bfloat16", cap=cap, fused_engine=engine, half=half)
    assert B.ulysses_plan_fused_backward_kernel(plan) == engine
    dxs = [[torch.empty_like(x) for x in xs[t]] for t in range(2)]
    for t in dxs:
        for o in t:
            o.view(torch.int16).fill_(-23131)
    dw = torch.full((2, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dxs[0], dxs[1], xs[0], xs[1], grads[0], grads[1], w,
                                       dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    del grads
    picks = [(q, i) for q, i, _ in src]
    dw_ref = np.zeros((2, d))
    for t in range(2):
        x_rows = _gather_rows(xs[t], picks, d)
        got_rows = _gather_rows(dxs[t], picks, d)
        g_rows = vals[t].view(torch.int16).numpy().view(np.uint16)
        for j, (r, bb, s, h) in enumerate(rows):
            ref_dx, ref_dw = oracle.fused_row_bwd_var(oracle.decode(x_rows[j], int(f16)),
                                                      oracle.decode(g_rows[j], int(f16)), int(half),
                                                      wn[t], EPS, s, THETA)
            dw_ref[t] += ref_dw
            _close(oracle, got_rows[j], ref_dx, f16, 1e-4, f"{what} dx {t} r={r} bb={bb} s={s} h={h}")
        # every row without a gradient is +0 or -0: clear the picked rows, then no bit but the
        # sign may remain anywhere
        for q in range(g[0]):
            sel = [i for qq, i in picks if qq == q]
            flat = dxs[t][q].reshape(-1, d).view(torch.int16)
            if sel:
                flat[torch.as_tensor(sel, device="cuda")] = 0
            nonzero = int(((flat & 0x7FFF) != 0).sum())
            assert nonzero == 0, f"{what} dx {t} rank {q}: {nonzero} elements without gradient are not 0"
    check_dw(dw.cpu().numpy(), dw_ref, len(rows), f"{what} dw")
    del dxs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", list(FUSED_ENGINES))
def test_backward_past_4gib(oracle, engine):
    """The fused backward (bf16, adjacent pairs) on ranks of more than 4 GiB per tensor, in one
    launch and chunked, with the output gradient zero except on 1,200 sampled rows per tensor and
    every row of the last 8 positions of batch 1."""
    g = FUSED_BIG
    xs, w, wn = _fused_inputs(g, False, 101)
    rows = _sample_rows(g, np.random.default_rng(102), 1200, 8)
    for name, cap in CAPS.items():
        _check_sparse_backward(oracle, g, xs, w, wn, False, False, rows, FUSED_ENGINES[engine], cap,
                               103, f"cap {name}")
    del xs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("engine", list(FUSED_ENGINES))
@pytest.mark.parametrize("f16,half", [(False, False), (True, True)], ids=["bf16-adjacent", "f16-half"])
def test_backward_max_positions(oracle, engine, f16, half):
    """The fused backward at S = 2^24 - 1 tokens, d = 128 (W=2, one head per rank), with the
    output gradient zero except on 1,200 sampled rows and the last 64 positions."""
    g = (2, 1, [1 << 23, (1 << 23) - 1], [1, 1], 128)
    xs, w, wn = _fused_inputs(g, f16, 111)
    rows = _sample_rows(g, np.random.default_rng(112), 1200, 64)
    _check_sparse_backward(oracle, g, xs, w, wn, f16, half, rows, FUSED_ENGINES[engine], None, 113,
                           "max positions")
    del xs
    torch.cuda.empty_cache()
