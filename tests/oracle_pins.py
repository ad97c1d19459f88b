"""Checks that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle
disagrees with an independent fact: a library formulation of the same mapping (torch ``split`` +
``cat``; the pages' own baseline of permute + all_to_all + permute, emulated in one process), an
identity or invariant (W=1, round trip, byte conservation), the shapes the pages print, a library
routine (``torch.nn.functional.rms_norm``, complex multiplication, torch's float32->bf16
rounding) or a closed form (one-hot rows, unit-weight RMS).

``test_oracle.py`` runs every pin against the oracle; ``test_oracle_mutants.py`` plants plausible
mistakes in a copy of the oracle's C source and checks that some pin catches each one.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

UINT = {1: np.uint8, 2: np.uint16, 4: np.uint32}
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------------------------
# independent formulations of the relayout
# --------------------------------------------------------------------------------------------
def split_cat_mode0(xs, head_splits):
    """out[r] = concatenation over ranks q (along the sequence) of rank q's r-th head group."""
    W = len(xs)
    pieces = [torch.split(torch.from_numpy(x), list(head_splits), dim=2) for x in xs]
    return [torch.cat([pieces[q][r] for q in range(W)], dim=1).numpy() for r in range(W)]


def split_cat_mode1(ys, seq_splits):
    """out[q] = concatenation over ranks r (along heads) of rank r's q-th sequence piece."""
    W = len(ys)
    pieces = [torch.split(torch.from_numpy(y), list(seq_splits), dim=1) for y in ys]
    return [torch.cat([pieces[r][q] for r in range(W)], dim=2).numpy() for q in range(W)]


def pages_base_mode0(xs):
    """Even splits only: the baseline the pages measure against, permute + all_to_all_single +
    permute, with the all-to-all of W ranks emulated as a swap of the (sender, receiver) axes."""
    W = len(xs)
    b, s, N, d = xs[0].shape
    n = N // W
    send = [torch.from_numpy(x).reshape(b, s, W, n, d).permute(2, 0, 1, 3, 4) for x in xs]
    recv = [torch.stack([send[q][r] for q in range(W)], dim=0) for r in range(W)]
    return [t.permute(1, 0, 2, 3, 4).reshape(b, W * s, n, d).numpy() for t in recv]


def pages_base_mode1(ys):
    W = len(ys)
    b, S, n, d = ys[0].shape
    s = S // W
    send = [torch.from_numpy(y).reshape(b, W, s, n, d).permute(1, 0, 2, 3, 4) for y in ys]
    recv = [torch.stack([send[r][q] for r in range(W)], dim=0) for q in range(W)]
    return [t.permute(1, 2, 0, 3, 4).reshape(b, s, W * n, d).numpy() for t in recv]


# --------------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------------
def _rand_inputs(rng, W, b, seq_splits, head_splits, d, e, mode):
    N, S = sum(head_splits), sum(seq_splits)
    if mode == 0:
        shapes = [(b, s, N, d) for s in seq_splits]
    else:
        shapes = [(b, S, n, d) for n in head_splits]
    info = np.iinfo(UINT[e])
    return [rng.integers(0, info.max, size=sh, dtype=UINT[e], endpoint=True) for sh in shapes]


def _same(a_list, b_list, what):
    assert len(a_list) == len(b_list), what
    for k, (a, b) in enumerate(zip(a_list, b_list)):
        assert a.shape == b.shape, f"{what}: rank {k} shape {a.shape} != {b.shape}"
        assert np.array_equal(a, b), f"{what}: rank {k} differs"


def _random_geometries(rng, count, max_W=4, allow_zero=True):
    out = []
    while len(out) < count:
        W = int(rng.integers(1, max_W + 1))
        lo = 0 if allow_zero else 1
        seq = [int(v) for v in rng.integers(lo, 5, size=W)]
        heads = [int(v) for v in rng.integers(lo, 4, size=W)]
        if sum(seq) == 0 or sum(heads) == 0:
            continue
        out.append((W, int(rng.integers(1, 3)), seq, heads, int(rng.choice([2, 4, 8])),
                    int(rng.choice([1, 2, 4]))))
    return out


# --------------------------------------------------------------------------------------------
# relayout pins
# --------------------------------------------------------------------------------------------
def pin_relayout_vs_split_cat(orc, quick=False):
    rng = np.random.default_rng(11)
    for W, b, seq, heads, d, e in _random_geometries(rng, 40 if quick else 200):
        xs = _rand_inputs(rng, W, b, seq, heads, d, e, 0)
        _same(orc.a2a_4d(xs, seq, heads, 0), split_cat_mode0(xs, heads), f"mode0 {W,b,seq,heads,d,e}")
        ys = _rand_inputs(rng, W, b, seq, heads, d, e, 1)
        _same(orc.a2a_4d(ys, seq, heads, 1), split_cat_mode1(ys, seq), f"mode1 {W,b,seq,heads,d,e}")


def pin_relayout_enumeration(orc, quick=False):
    """Every split combination with shares in {0, 1, 2} for W <= 3 (W <= 2 when quick), b in
    {1, 2}, against the split/cat formulation."""
    rng = np.random.default_rng(12)
    max_W = 2 if quick else 3
    for W in range(1, max_W + 1):
        for seq in itertools.product(range(3), repeat=W):
            if sum(seq) == 0:
                continue
            for heads in itertools.product(range(3), repeat=W):
                if sum(heads) == 0:
                    continue
                for b in (1, 2):
                    xs = _rand_inputs(rng, W, b, seq, heads, 4, 2, 0)
                    _same(orc.a2a_4d(xs, seq, heads, 0), split_cat_mode0(xs, heads), "enum mode0")
                    ys = _rand_inputs(rng, W, b, seq, heads, 4, 2, 1)
                    _same(orc.a2a_4d(ys, seq, heads, 1), split_cat_mode1(ys, seq), "enum mode1")


def pin_relayout_vs_pages_base(orc, quick=False):
    rng = np.random.default_rng(13)
    for W in (1, 2, 3, 4, 8):
        for b, s, n, d, e in ((1, 3, 2, 8, 2), (2, 5, 1, 4, 4), (1, 2, 3, 16, 1)):
            seq, heads = [s] * W, [n] * W
            xs = _rand_inputs(rng, W, b, seq, heads, d, e, 0)
            _same(orc.a2a_4d(xs, seq, heads, 0), pages_base_mode0(xs), f"base mode0 W={W}")
            ys = _rand_inputs(rng, W, b, seq, heads, d, e, 1)
            _same(orc.a2a_4d(ys, seq, heads, 1), pages_base_mode1(ys), f"base mode1 W={W}")


def pin_identity_w1(orc, quick=False):
    rng = np.random.default_rng(14)
    for b, s, n, d, e in ((1, 7, 3, 8, 2), (2, 1, 5, 4, 4), (3, 4, 1, 16, 1)):
        x = _rand_inputs(rng, 1, b, [s], [n], d, e, 0)
        _same(orc.a2a_4d(x, [s], [n], 0), x, "W=1 mode 0 identity")
        _same(orc.a2a_4d(x, [s], [n], 1), x, "W=1 mode 1 identity")


def pin_round_trip(orc, quick=False):
    rng = np.random.default_rng(15)
    for W, b, seq, heads, d, e in _random_geometries(rng, 30 if quick else 120):
        xs = _rand_inputs(rng, W, b, seq, heads, d, e, 0)
        _same(orc.a2a_4d(orc.a2a_4d(xs, seq, heads, 0), seq, heads, 1), xs, "mode1(mode0(x))")
        ys = _rand_inputs(rng, W, b, seq, heads, d, e, 1)
        _same(orc.a2a_4d(orc.a2a_4d(ys, seq, heads, 1), seq, heads, 0), ys, "mode0(mode1(y))")


def pin_conservation_and_coverage(orc, quick=False):
    """Unique 32-bit tags in, every output slot written exactly once with some input's tag."""
    rng = np.random.default_rng(16)
    for W, b, seq, heads, d, _ in _random_geometries(rng, 20 if quick else 80):
        N, S = sum(heads), sum(seq)
        for mode in (0, 1):
            in_shapes = ([(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads])
            out_shapes = orc.out_shapes(b, seq, heads, d, mode)
            base = 0
            xs = []
            for sh in in_shapes:
                cnt = int(np.prod(sh))
                xs.append((np.arange(cnt, dtype=np.uint32) + base + 1).reshape(sh))
                base += cnt
            outs = [np.zeros(sh, dtype=np.uint32) for sh in out_shapes]  # 0 = never written
            orc.a2a_4d_raw(W, b, seq, heads, d, 4, mode, [x.ctypes.data for x in xs],
                           [o.ctypes.data for o in outs])
            # the sizes the definition implies: sum of splits equals the global extents
            assert sum(int(np.prod(s)) for s in out_shapes) == base
            got = np.sort(np.concatenate([o.ravel() for o in outs])) if outs else np.array([])
            want = np.arange(1, base + 1, dtype=np.uint32)
            assert np.array_equal(got, want), f"not a permutation of the input (mode {mode})"


def pin_source_query(orc, quick=False):
    """The single-element query names the input element the bulk relayout put there."""
    rng = np.random.default_rng(17)
    for W, b, seq, heads, d, e in _random_geometries(rng, 20 if quick else 60):
        for mode in (0, 1):
            xs = _rand_inputs(rng, W, b, seq, heads, d, e, mode)
            outs = orc.a2a_4d(xs, seq, heads, mode)
            for r, o in enumerate(outs):
                flat = o.ravel()
                for k in rng.integers(0, max(flat.size, 1), size=min(8, flat.size)):
                    q, idx = orc.a2a_4d_source(W, b, seq, heads, d, mode, r, int(k))
                    assert xs[q].ravel()[idx] == flat[k], "source query disagrees with relayout"


def _golden_lines():
    with open(os.path.join(GOLDEN, "page_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


def _kv(text):
    return dict(item.split("=", 1) for item in text.split())


def pin_page_shapes(orc, quick=False):
    """The shapes the two Quick start sections print, computed by actually running the oracle."""
    rng = np.random.default_rng(18)
    lines = {name: (_kv(inp), _kv(exp)) for name, inp, exp in _golden_lines()}
    inp, exp = lines["quickstart_v010"]
    for ws in ((2,) if quick else (1, 2, 8)):
        b, s, hpr, d = int(inp["b"]), int(inp["s_local"]), int(inp["heads_per_rank"]), int(inp["d"])
        xs = _rand_inputs(rng, ws, b, [s] * ws, [hpr] * ws, d, 2, 0)
        assert xs[0].shape == (b, s, hpr * ws, d)
        outs = orc.a2a_4d(xs, [s] * ws, [hpr] * ws, 0)
        want = eval(exp["out_shape"], {"ws": ws})  # noqa: S307  (fixture arithmetic like 16*ws)
        assert all(o.shape == want for o in outs)
    inp, exp = lines["quickstart_v021"]
    for ws in ((2,) if quick else (2, 4)):
        b, s, hpr, d = int(inp["b"]), int(inp["s_local"]), int(inp["heads_per_rank"]), int(inp["d"])
        xs = _rand_inputs(rng, ws, b, [s] * ws, [hpr] * ws, d, 2, 0)
        ys = orc.a2a_4d(xs, [s] * ws, [hpr] * ws, 0)
        assert all(y.shape == eval(exp["out_shape"], {"ws": ws}) for y in ys)  # noqa: S307
        zs = orc.a2a_4d(ys, [s] * ws, [hpr] * ws, 1)
        assert all(z.shape == eval(exp["back"], {"ws": ws}) for z in zs)  # noqa: S307
        _same(zs, xs, "quick start round trip")


# --------------------------------------------------------------------------------------------
# fused QK RMSNorm + RoPE pins
# --------------------------------------------------------------------------------------------
def _freq(theta, j, d):
    return theta ** (-2.0 * j / d)


def pin_rmsnorm_vs_torch(orc, quick=False):
    rng = np.random.default_rng(21)
    for d in (2, 8, 24, 64, 72, 128):
        for eps in (1e-6, 1e-2, 0.0):
            x = rng.standard_normal(d) * rng.uniform(0.01, 10)
            w = 1.0 + 0.1 * rng.standard_normal(d)
            want = F.rms_norm(torch.from_numpy(x)[None], (d,), weight=torch.from_numpy(w),
                              eps=eps)[0].numpy()
            np.testing.assert_allclose(orc.rmsnorm(x, w, eps), want, rtol=1e-13, atol=1e-15)


def pin_rope_vs_complex(orc, quick=False):
    """Adjacent pairs as complex numbers, multiplied by exp(i * p * theta^(-2j/d))."""
    rng = np.random.default_rng(22)
    for d in (2, 8, 24, 72, 128):
        for p in (0, 1, 7, 9450, 75599, 249999):
            y = rng.standard_normal(d)
            z = torch.view_as_complex(torch.from_numpy(y.copy()).view(d // 2, 2))
            ang = torch.tensor([p * _freq(1e4, j, d) for j in range(d // 2)], dtype=torch.float64)
            rot = z * torch.polar(torch.ones_like(ang), ang)
            want = torch.view_as_real(rot).reshape(d).numpy()
            np.testing.assert_allclose(orc.rope(y, p, 1e4), want, rtol=1e-12, atol=1e-12)


def pin_rope_identities(orc, quick=False):
    rng = np.random.default_rng(23)
    d = 128
    y = rng.standard_normal(d)
    np.testing.assert_array_equal(orc.rope(y, 0, 1e4), y)           # p = 0 is the identity
    for p1, p2 in ((3, 5), (9450, -9450), (75599, 1), (12345, 678)):
        a = orc.rope(y, p1, 1e4)
        pairs_in = np.hypot(y[0::2], y[1::2])
        pairs_out = np.hypot(a[0::2], a[1::2])
        np.testing.assert_allclose(pairs_out, pairs_in, rtol=1e-12)  # rotation keeps pair norms
        np.testing.assert_allclose(orc.rope(a, p2, 1e4), orc.rope(y, p1 + p2, 1e4),
                                   rtol=1e-9, atol=1e-9)             # rotations compose


def pin_one_hot_rows(orc, quick=False):
    """x = e_(2j): the normalised row is c * e_(2j) with c = w_(2j) / sqrt(1/d + eps), and RoPE
    turns it into c * (cos(p theta_j), sin(p theta_j)) in pair j, zero elsewhere."""
    d, eps, theta = 16, 1e-6, 1e4
    w = np.linspace(0.5, 1.5, d)
    for j in range(d // 2):
        for p in (0, 1, 4, 100):
            x = np.zeros(d)
            x[2 * j] = 1.0
            got = orc.rope(orc.rmsnorm(x, w, eps), p, theta)
            c = w[2 * j] / math.sqrt(1.0 / d + eps)
            want = np.zeros(d)
            want[2 * j] = c * math.cos(p * _freq(theta, j, d))
            want[2 * j + 1] = c * math.sin(p * _freq(theta, j, d))
            np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def pin_unit_weight_rms(orc, quick=False):
    """With unit weights the output's RMS is sqrt(ms / (ms + eps)) at any position."""
    rng = np.random.default_rng(24)
    d = 128
    for eps in (1e-6, 0.5):
        x = rng.standard_normal(d) * 0.05
        ms = float(np.mean(x * x))
        y = orc.rope(orc.rmsnorm(x, np.ones(d), eps), 777, 1e4)
        assert abs(math.sqrt(float(np.mean(y * y))) - math.sqrt(ms / (ms + eps))) < 1e-12


def _bf16_inputs(rng, W, b, seq, heads, d):
    N = sum(heads)
    out = []
    for s in seq:
        v = torch.from_numpy(rng.standard_normal((b, s, N, d)).astype(np.float32)).to(torch.bfloat16)
        out.append(v.view(torch.int16).numpy().view(np.uint16))
    return out


def pin_fused_formulations_agree(orc, quick=False):
    """Transform-then-place equals place-then-transform, exactly (same double operations)."""
    rng = np.random.default_rng(25)
    cases = [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16), (1, 1, [5], [2], 4),
             (4, 1, [1, 2, 1, 3], [1, 1, 1, 1], 8)]
    for W, b, seq, heads, d in cases:
        xs = _bf16_inputs(rng, W, b, seq, heads, d)
        w = 1.0 + 0.1 * rng.standard_normal(d)
        A = orc.qk_fused_A(xs, seq, heads, w, 1e-6, 1e4)
        B = orc.qk_fused_B(xs, seq, heads, w, 1e-6, 1e4)
        _same(A, B, "fused A vs B")
        for r in range(W):
            for bb in range(b):
                for s in range(sum(seq)):
                    for h in range(heads[r]):
                        row = orc.qk_fused_row(xs, seq, heads, w, 1e-6, 1e4, r, bb, s, h)
                        assert np.array_equal(row, A[r][bb, s, h]), "fused row query disagrees"


def pin_fused_placement_decode(orc, quick=False):
    """One-hot source rows whose hot pair index encodes (source rank, global head): each output
    row's hot pair and rotation angle must decode to the rank/head/position mode 0 names."""
    theta = 1e4
    W, seq, heads = 3, [2, 1, 2], [1, 2, 1]
    N, S = sum(heads), sum(seq)
    d = 2 * W * N                      # one pair per (q, g)
    xs = []
    for q in range(W):
        x = np.zeros((1, seq[q], N, d), dtype=np.float32)
        for g in range(N):
            x[0, :, g, 2 * (q * N + g)] = 1.0
        xs.append(torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    outs = orc.qk_fused_A(xs, seq, heads, np.ones(d), 0.0, theta)
    head_owner = [r for r in range(W) for _ in range(heads[r])]
    seq_owner = [q for q in range(W) for _ in range(seq[q])]
    for r in range(W):
        for s in range(S):
            for h in range(heads[r]):
                row = outs[r][0, s, h]
                mags = np.hypot(row[0::2], row[1::2])
                j = int(np.argmax(mags))
                q, g = divmod(j, N)
                assert q == seq_owner[s], "row came from the wrong source rank"
                assert head_owner[g] == r and g - sum(heads[:r]) == h, "wrong head"
                ang = math.atan2(row[2 * j + 1], row[2 * j]) % (2 * math.pi)
                p = ang / _freq(theta, j, d)
                assert abs(p - s) < 1e-6, f"rotation angle decodes to p={p}, expected {s}"


def pin_qkv_interleaved(orc, quick=False):
    """Interleaved (b, s, 3, N, d) QKV: torch.unbind of the plane axis gives q, k, v; the result
    must equal the separately pinned fused transform on q and k and the mode-0 relayout of v."""
    rng = np.random.default_rng(27)
    cases = [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16), (1, 1, [4], [3], 8),
             (4, 1, [1, 2, 1, 2], [2, 0, 1, 1], 8)]
    for W, b, seq, heads, d in cases:
        N = sum(heads)
        qkv = []
        for s in seq:
            v = torch.from_numpy(rng.standard_normal((b, s, 3, N, d)).astype(np.float32))
            qkv.append(v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
        wq = 1.0 + 0.1 * rng.standard_normal(d)
        wk = 1.0 + 0.1 * rng.standard_normal(d)
        planes = [[t.contiguous().numpy().view(np.uint16)
                   for t in torch.unbind(torch.from_numpy(x.view(np.int16)), dim=2)] for x in qkv]
        q_in = [p[0] for p in planes]
        k_in = [p[1] for p in planes]
        v_in = [p[2] for p in planes]
        qo, ko, vo = orc.qkv_fused(qkv, seq, heads, wq, wk, 1e-6, 1e4)
        _same(qo, orc.qk_fused_A(q_in, seq, heads, wq, 1e-6, 1e4), "qkv: q plane")
        _same(ko, orc.qk_fused_A(k_in, seq, heads, wk, 1e-6, 1e4), "qkv: k plane")
        _same(vo, split_cat_mode0(v_in, heads), "qkv: v plane")


def pin_packed_planes(orc, quick=False):
    """Packed inputs with C planes per token and a token pitch: slicing each token's row into its
    planes (plane c = columns c*N*d .. (c+1)*N*d of the (b, s, pitch) view, a numpy view) gives the
    plane tensors; the q and k planes must equal the pinned fused transform (with their own
    weights), every other plane the pinned split/cat relayout, whatever the extra columns of a
    token hold. With 3 planes (q, k, v) and no extra columns it is the interleaved QKV form."""
    rng = np.random.default_rng(48)
    cases = [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16), (1, 1, [4], [3], 8),
             (4, 1, [1, 2, 1, 2], [2, 0, 1, 1], 8)]
    bf16 = lambda shape: (torch.from_numpy(rng.standard_normal(shape).astype(np.float32))  # noqa: E731
                          .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    for W, b, seq, heads, d in cases:
        N = sum(heads)
        wq = 1.0 + 0.1 * rng.standard_normal(d)
        wk = 1.0 + 0.1 * rng.standard_normal(d)
        # the interleaved QKV form as a special case
        qkv = [bf16((b, s, 3, N, d)) for s in seq]
        got = orc.packed_fused(qkv, seq, heads, d, 3, 0, 1, 3 * N * d, wq, wk, 1e-6, 1e4)
        want = orc.qkv_fused(qkv, seq, heads, wq, wk, 1e-6, 1e4)
        _same(got[0], want[0], "packed 3 planes: q")
        _same(got[1], want[1], "packed 3 planes: k")
        _same(got[2][2], want[2], "packed 3 planes: v")
        for C, qp, kp, extra in [(4, 0, 1, 0), (4, 2, 0, 24), (2, 1, 0, 8), (6, 3, 5, 16)]:
            pitch = C * N * d + extra
            packed = [bf16((b, s, pitch)) for s in seq]
            qo, ko, plain = orc.packed_fused(packed, seq, heads, d, C, qp, kp, pitch, wq, wk, 1e-6,
                                             1e4)
            plane = lambda c: [np.ascontiguousarray(x[:, :, c * N * d:(c + 1) * N * d])  # noqa: E731
                               .reshape(b, x.shape[1], N, d) for x in packed]
            _same(qo, orc.qk_fused_A(plane(qp), seq, heads, wq, 1e-6, 1e4), f"packed C={C}: q")
            _same(ko, orc.qk_fused_A(plane(kp), seq, heads, wk, 1e-6, 1e4), f"packed C={C}: k")
            for c in range(C):
                if c in (qp, kp):
                    assert plain[c] is None
                else:
                    _same(plain[c], split_cat_mode0(plane(c), heads), f"packed C={C}: plane {c}")
            if extra:  # the extra columns are never read
                other = [x.copy() for x in packed]
                for x in other:
                    x[:, :, C * N * d:] = rng.integers(0, 1 << 16, x[:, :, C * N * d:].shape)
                again = orc.packed_fused(other, seq, heads, d, C, qp, kp, pitch, wq, wk, 1e-6, 1e4)
                _same(again[0], qo, "extra columns: q")
                _same(again[1], ko, "extra columns: k")


def pin_packed_planes_backward(orc, quick=False):
    """Backward of the packed form: slicing the planes as in pin_packed_planes, the q and k planes'
    gradients must equal the pinned backward of the fused call on those slices (bit for bit, dw
    too: the rows are visited in the same order), every other plane's the pinned mode 1 of its
    output gradient; the extra columns of a token are never written."""
    rng = np.random.default_rng(49)
    bf16 = lambda shape: (torch.from_numpy(rng.standard_normal(shape).astype(np.float32))  # noqa: E731
                          .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    for W, b, seq, heads, d in [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16),
                                (4, 1, [1, 2, 1, 2], [2, 0, 1, 1], 8)]:
        N, S = sum(heads), sum(seq)
        wq = 1.0 + 0.1 * rng.standard_normal(d)
        wk = 1.0 + 0.1 * rng.standard_normal(d)
        for C, qp, kp, extra in [(3, 0, 1, 0), (4, 2, 0, 24), (2, 1, 0, 8)]:
            pitch = C * N * d + extra
            packed = [bf16((b, s, pitch)) for s in seq]
            grads = [[bf16((b, S, n, d)) for n in heads] for _ in range(C)]
            dx, dw = orc.packed_fused_bwd(packed, grads, seq, heads, d, C, qp, kp, pitch, wq, wk,
                                          1e-6, 1e4)
            plane = lambda arrs, c: [arr[:, :, c * N * d:(c + 1) * N * d].reshape(b, arr.shape[1], N, d)  # noqa: E731
                                     for arr in arrs]
            for c, w, row in ((qp, wq, 0), (kp, wk, 1)):
                want_dx, want_dw = orc.qk_fused_bwd(plane(packed, c), grads[c], seq, heads, w, 1e-6,
                                                    1e4)
                _same(plane(dx, c), want_dx, f"packed bwd C={C}: plane {c}")
                assert np.array_equal(dw[row], want_dw), f"packed bwd C={C}: dw {row}"
            for c in range(C):
                if c not in (qp, kp):
                    want = orc.a2a_4d(grads[c], seq, heads, 1)
                    got = [orc.double_to_bf16(x) for x in plane(dx, c)]
                    _same(got, want, f"packed bwd C={C}: plane {c}")
            for x in dx:
                assert np.all(np.isnan(x[:, :, C * N * d:])), "extra columns written"


def _torch_row_forward(x, w, eps, p, theta):
    """The fused row transform built from library pieces (F.rms_norm, complex multiplication),
    differentiable by torch.autograd."""
    d = x.shape[-1]
    y = F.rms_norm(x[None], (d,), weight=w, eps=eps)[0]
    ang = torch.tensor([p * _freq(theta, j, d) for j in range(d // 2)], dtype=torch.float64)
    z = torch.view_as_complex(y.reshape(d // 2, 2)) * torch.polar(torch.ones_like(ang), ang)
    return torch.view_as_real(z).reshape(d)


def pin_fused_bwd_vs_autograd(orc, quick=False):
    """The row backward equals torch.autograd's gradients of the library-built forward."""
    rng = np.random.default_rng(28)
    for d in (2, 8, 72, 128):
        for p in (0, 3, 9450, 75599):
            for eps in (1e-6, 0.3):
                x = torch.tensor(rng.standard_normal(d), dtype=torch.float64, requires_grad=True)
                w = torch.tensor(1.0 + 0.1 * rng.standard_normal(d), dtype=torch.float64,
                                 requires_grad=True)
                g = torch.tensor(rng.standard_normal(d), dtype=torch.float64)
                _torch_row_forward(x, w, eps, p, 1e4).backward(g)
                dx, dw = orc.fused_row_bwd(x.detach().numpy(), g.numpy(), w.detach().numpy(), eps,
                                           p, 1e4)
                np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-9, atol=1e-11)
                np.testing.assert_allclose(dw, w.grad.numpy(), rtol=1e-9, atol=1e-11)


def pin_fused_bwd_finite_differences(orc, quick=False):
    """Adjoint identity against the forward oracle: <g, (f(x + h v) - f(x - h v)) / 2h>
    equals <dL/dx, v> (and the same for w)."""
    rng = np.random.default_rng(29)
    d, eps, theta, h = 16, 1e-3, 1e4, 1e-5
    for p in (0, 5, 1234):
        x, w, g, v = (rng.standard_normal(d) for _ in range(4))
        w = 1.0 + 0.1 * w
        f = lambda xx, ww: orc.rope(orc.rmsnorm(xx, ww, eps), p, theta)  # noqa: E731
        dx, dw = orc.fused_row_bwd(x, g, w, eps, p, theta)
        num_x = np.dot(g, (f(x + h * v, w) - f(x - h * v, w)) / (2 * h))
        num_w = np.dot(g, (f(x, w + h * v) - f(x, w - h * v)) / (2 * h))
        assert abs(num_x - np.dot(dx, v)) < 1e-6 * (1 + abs(num_x))
        assert abs(num_w - np.dot(dw, v)) < 1e-6 * (1 + abs(num_w))


def pin_fused_bwd_placement(orc, quick=False):
    """The whole-call backward equals: mode 1 (pinned above) brings the output gradients back to
    the sequence side, then the row backward at each row's global position; dw is the sum."""
    rng = np.random.default_rng(30)
    for W, b, seq, heads, d in [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16)]:
        N, S = sum(heads), sum(seq)
        bf = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(  # noqa: E731
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xs = [bf((b, s, N, d)) for s in seq]
        gs = [bf((b, S, n, d)) for n in heads]
        w = 1.0 + 0.1 * rng.standard_normal(d)
        dx, dw = orc.qk_fused_bwd(xs, gs, seq, heads, w, 1e-6, 1e4)
        g_seq = orc.a2a_4d(gs, seq, heads, 1)
        dw_want = np.zeros(d)
        seq_off = np.cumsum([0] + list(seq))
        for q in range(W):
            for bb in range(b):
                for i in range(seq[q]):
                    for hh in range(N):
                        x = orc.bf16_to_double(xs[q][bb, i, hh])
                        g = orc.bf16_to_double(g_seq[q][bb, i, hh])
                        want, dwr = orc.fused_row_bwd(x, g, w, 1e-6, seq_off[q] + i, 1e4)
                        dw_want += dwr
                        np.testing.assert_allclose(dx[q][bb, i, hh], want, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dw, dw_want, rtol=1e-12, atol=1e-12)


def pin_relayout_adjoint(orc, quick=False):
    """Mode 1 is the adjoint of mode 0 (the backward pairing): <mode0(x), y> = <x, mode1(y)>."""
    rng = np.random.default_rng(31)
    for W, b, seq, heads, d, _ in _random_geometries(rng, 20):
        N, S = sum(heads), sum(seq)
        xs = [rng.standard_normal((b, s, N, d)).astype(np.float32) for s in seq]
        ys = [rng.standard_normal((b, S, n, d)).astype(np.float32) for n in heads]
        dot = lambda a, c: float(np.sum(a.astype(np.float64) * c))  # noqa: E731
        lhs = sum(dot(a, c) for a, c in zip(orc.a2a_4d(xs, seq, heads, 0), ys))
        rhs = sum(dot(a, c) for a, c in zip(xs, orc.a2a_4d(ys, seq, heads, 1)))
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(lhs))


# ---- variants: fp16 elements, rotate-half pairs ------------------------------------------------
def pin_f16_decode(orc, quick=False):
    """Every binary16 bit pattern decodes as numpy's float16 does (NaNs as NaNs)."""
    h = np.arange(65536, dtype=np.uint16)
    got = orc.f16_to_double(h)
    want = h.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def pin_f16_encode(orc, quick=False):
    """double -> binary16 against numpy's correctly rounded conversion on random values over the
    whole range, exact ties, the subnormal range and the overflow edge, plus closed forms."""
    rng = np.random.default_rng(40)
    vals = [rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000)),
            (rng.integers(0, 2048, 4000) + 0.5) * np.exp2(rng.integers(-24, 6, 4000)),  # ties
            rng.uniform(-2.0 ** -14, 2.0 ** -14, 4000),                                # subnormal
            np.array([65504.0, 65519.99, 65520.0, 65535.0, 1e6, 2.0 ** -25, 3 * 2.0 ** -25,
                      2.0 ** -26, -0.0, 0.0, np.inf, -np.inf])]
    x = np.concatenate(vals)
    got = orc.double_to_f16(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want), int((got != want).sum())
    closed = {1.0 + 2.0 ** -11: 0x3C00, 1.0 + 3 * 2.0 ** -11: 0x3C02, 65519.0: 0x7BFF,
              65520.0: 0x7C00, 2.0 ** -25: 0x0000, 3 * 2.0 ** -25: 0x0002, -2.0: 0xC000}
    for v, bits in closed.items():
        assert int(orc.double_to_f16(np.array([v]))[0]) == bits, v


def pin_rope_half_vs_complex(orc, quick=False):
    """Rotate-half pairs (y_j, y_(j+d/2)) as complex numbers times exp(i p theta^(-2j/d))."""
    rng = np.random.default_rng(41)
    for d in (2, 8, 24, 72, 128):
        for p in (0, 1, 9450, 75599):
            y = rng.standard_normal(d)
            h = d // 2
            z = torch.complex(torch.from_numpy(y[:h].copy()), torch.from_numpy(y[h:].copy()))
            ang = torch.tensor([p * _freq(1e4, j, d) for j in range(h)], dtype=torch.float64)
            rot = z * torch.polar(torch.ones_like(ang), ang)
            want = np.concatenate([rot.real.numpy(), rot.imag.numpy()])
            np.testing.assert_allclose(orc.rope_half(y, p, 1e4), want, rtol=1e-12, atol=1e-12)


def pin_rope_half_is_permuted_adjacent(orc, quick=False):
    """Rotate-half equals adjacent pairs on the interleaved row: (P y)_(2j) = y_j,
    (P y)_(2j+1) = y_(j+d/2), rope_half(y) = P^-1 rope(P y)."""
    rng = np.random.default_rng(42)
    for d in (4, 24, 64, 72, 256):
        h = d // 2
        perm = np.empty(d, dtype=np.int64)
        perm[0::2] = np.arange(h)
        perm[1::2] = np.arange(h, d)
        for p in (3, 1000, 75599):
            y = rng.standard_normal(d)
            adj = orc.rope(y[perm], p, 1e4)
            back = np.empty(d)
            back[perm] = adj
            np.testing.assert_array_equal(orc.rope_half(y, p, 1e4), back)


def _torch_row_half(x, w, eps, p, theta):
    """RMSNorm then the usual rotate-half formula y*cos + rotate_half(y)*sin, with cos and sin of
    pair j repeated in both halves; differentiable."""
    d = x.shape[-1]
    y = F.rms_norm(x[None], (d,), weight=w, eps=eps)[0]
    ang = torch.tensor([p * _freq(theta, j, d) for j in range(d // 2)], dtype=torch.float64)
    cos, sin = torch.cat([ang.cos(), ang.cos()]), torch.cat([ang.sin(), ang.sin()])
    rot = torch.cat([-y[d // 2:], y[:d // 2]])
    return y * cos + rot * sin


def pin_fused_row_variants(orc, quick=False):
    """A variant row equals the library-built forward on the decoded values: adjacent pairs via
    the pinned complex formulation, rotate-half via the rotate_half formula; bf16 and fp16
    decoding via torch's own bf16 and numpy's float16."""
    rng = np.random.default_rng(43)
    for d in (8, 72, 128):
        for f16 in (0, 1):
            for half in (0, 1):
                for p in (0, 5, 75599):
                    xf = rng.standard_normal(d).astype(np.float32)
                    if f16:
                        raw = xf.astype(np.float16).view(np.uint16)
                        x = raw.view(np.float16).astype(np.float64)
                    else:
                        t = torch.from_numpy(xf).to(torch.bfloat16)
                        raw = t.view(torch.int16).numpy().view(np.uint16)
                        x = t.double().numpy()
                    w = 1.0 + 0.1 * rng.standard_normal(d)
                    xt, wt = torch.from_numpy(x), torch.from_numpy(w)
                    if half:
                        want = _torch_row_half(xt, wt, 1e-6, p, 1e4).numpy()
                    else:
                        want = _torch_row_forward(xt, wt, 1e-6, p, 1e4).detach().numpy()
                    got = orc.fused_row_var(raw, f16, half, w, 1e-6, p, 1e4)
                    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_fused_var_whole_call(orc, quick=False):
    """The whole call of a variant: (bf16, adjacent) is bit-identical to the pinned formulation
    A; every variant equals mode 0 of the raw elements (pinned above) followed by the variant row
    at the destination row's sequence index."""
    rng = np.random.default_rng(44)
    for W, b, seq, heads, d in [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16),
                                (2, 1, [2, 3], [1, 2], 24)]:
        N, S = sum(heads), sum(seq)
        raw = [rng.integers(0, 1 << 16, (b, s, N, d)).astype(np.uint16) for s in seq]
        # keep the elements finite and moderate for both decodings
        raw = [(r & 0x3FFF) | 0x3000 for r in raw]
        w = 1.0 + 0.1 * rng.standard_normal(d)
        a = orc.qk_fused_var(raw, seq, heads, w, 1e-6, 1e4, 0, 0)
        ref = orc.qk_fused_A(raw, seq, heads, w, 1e-6, 1e4)
        for x, y in zip(a, ref):
            assert np.array_equal(x, y)
        placed = orc.a2a_4d(raw, seq, heads, 0)
        for f16 in (0, 1):
            for half in (0, 1):
                got = orc.qk_fused_var(raw, seq, heads, w, 1e-6, 1e4, f16, half)
                for r in range(W):
                    for bb in range(b):
                        for t in range(S):
                            for h in range(heads[r]):
                                want = orc.fused_row_var(placed[r][bb, t, h], f16, half, w, 1e-6,
                                                         t, 1e4)
                                np.testing.assert_array_equal(got[r][bb, t, h], want)


def pin_fused_bwd_variants(orc, quick=False):
    """Row backward of a variant: adjacent pairs bit-identical to the pinned row backward;
    rotate-half against torch.autograd of the rotate_half formula (fp64), x.grad and w.grad."""
    rng = np.random.default_rng(45)
    for d in (2, 8, 72, 128):
        for p in (0, 3, 75599):
            x, g = rng.standard_normal(d), rng.standard_normal(d)
            w = 1.0 + 0.1 * rng.standard_normal(d)
            a = orc.fused_row_bwd_var(x, g, 0, w, 1e-6, p, 1e4)
            b_ = orc.fused_row_bwd(x, g, w, 1e-6, p, 1e4)
            assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])
            xt = torch.tensor(x, requires_grad=True)
            wt = torch.tensor(w, requires_grad=True)
            _torch_row_half(xt, wt, 1e-6, p, 1e4).backward(torch.from_numpy(g))
            dx, dw = orc.fused_row_bwd_var(x, g, 1, w, 1e-6, p, 1e4)
            np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-9, atol=1e-11)


def pin_fused_bwd_var_whole_call(orc, quick=False):
    """Whole-call backward of a variant: (bf16, adjacent) dx bit-identical to the pinned one (dw up
    to the order of its sum); every
    variant equals mode 1 (pinned) of the output gradients, then the variant row backward at
    each row's global position, dw the sum over rows."""
    rng = np.random.default_rng(46)
    for W, b, seq, heads, d in [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16)]:
        N, S = sum(heads), sum(seq)
        mk = lambda shape: ((rng.integers(0, 1 << 16, shape).astype(np.uint16) & 0x3FFF)  # noqa: E731
                            | 0x3000).astype(np.uint16)
        xs = [mk((b, s, N, d)) for s in seq]
        gs = [mk((b, S, n, d)) for n in heads]
        w = 1.0 + 0.1 * rng.standard_normal(d)
        a = orc.qk_fused_bwd_var(xs, gs, seq, heads, w, 1e-6, 1e4, 0, 0)
        ref = orc.qk_fused_bwd(xs, gs, seq, heads, w, 1e-6, 1e4)
        for x, y in zip(a[0], ref[0]):
            assert np.array_equal(x, y)
        np.testing.assert_allclose(a[1], ref[1], rtol=1e-13, atol=1e-13)  # rows summed in another order
        g_seq = orc.a2a_4d(gs, seq, heads, 1)
        seq_off = np.cumsum([0] + list(seq))
        for f16 in (0, 1):
            for half in (0, 1):
                dx, dw = orc.qk_fused_bwd_var(xs, gs, seq, heads, w, 1e-6, 1e4, f16, half)
                dw_want = np.zeros(d)
                for q in range(W):
                    for bb in range(b):
                        for i in range(seq[q]):
                            for hh in range(N):
                                want, dwr = orc.fused_row_bwd_var(
                                    orc.decode(xs[q][bb, i, hh], f16),
                                    orc.decode(g_seq[q][bb, i, hh], f16), half, w, 1e-6,
                                    seq_off[q] + i, 1e4)
                                dw_want += dwr
                                np.testing.assert_allclose(dx[q][bb, i, hh], want, rtol=1e-13,
                                                           atol=1e-15)
                np.testing.assert_allclose(dw, dw_want, rtol=1e-12, atol=1e-12)


def pin_parts_cover_the_call(orc, quick=False):
    """A call split into parts on host threads (ranges of shards and rows, the form the full-size
    GPU checks use) covers every row once: outputs prefilled with NaN come back bit-identical to
    the whole call, and dw, summed part by part, equals the whole call's dw up to the order of its
    double sum (a row computed twice or skipped moves it by a whole term)."""
    rng = np.random.default_rng(47)
    mk = lambda shape: ((rng.integers(0, 1 << 16, shape).astype(np.uint16) & 0x3FFF)  # noqa: E731
                        | 0x3000).astype(np.uint16)
    for W, b, seq, heads, d in [(3, 2, [5, 0, 7], [2, 1, 2], 16), (4, 1, [9, 3, 1, 6], [1, 2, 1, 1], 8)]:
        N, S = sum(heads), sum(seq)
        xs = [mk((b, s, N, d)) for s in seq]
        gs = [mk((b, S, n, d)) for n in heads]
        qkv = [mk((b, s, 3, N, d)) for s in seq]
        w = 1.0 + 0.1 * rng.standard_normal(d)
        w2 = 1.0 + 0.1 * rng.standard_normal(d)
        for threads in (2, 3, 5):
            for got, want in zip(orc.qk_fused_A(xs, seq, heads, w, 1e-6, 1e4, threads=threads),
                                 orc.qk_fused_A(xs, seq, heads, w, 1e-6, 1e4)):
                assert np.array_equal(got, want)
            a = orc.qkv_fused(qkv, seq, heads, w, w2, 1e-6, 1e4, threads=threads)
            c = orc.qkv_fused(qkv, seq, heads, w, w2, 1e-6, 1e4)
            for got, want in zip(a[0] + a[1] + a[2], c[0] + c[1] + c[2]):
                assert np.array_equal(got, want)
            dx, dw = orc.qk_fused_bwd(xs, gs, seq, heads, w, 1e-6, 1e4, threads=threads)
            dx1, dw1 = orc.qk_fused_bwd(xs, gs, seq, heads, w, 1e-6, 1e4)
            for got, want in zip(dx, dx1):
                assert np.array_equal(got, want)
            np.testing.assert_allclose(dw, dw1, rtol=1e-12, atol=1e-12)
            for f16 in (0, 1):
                for half in (0, 1):
                    for got, want in zip(
                            orc.qk_fused_var(xs, seq, heads, w, 1e-6, 1e4, f16, half, threads=threads),
                            orc.qk_fused_var(xs, seq, heads, w, 1e-6, 1e4, f16, half)):
                        assert np.array_equal(got, want)
                    dx, dw = orc.qk_fused_bwd_var(xs, gs, seq, heads, w, 1e-6, 1e4, f16, half,
                                                  threads=threads)
                    dx1, dw1 = orc.qk_fused_bwd_var(xs, gs, seq, heads, w, 1e-6, 1e4, f16, half)
                    for got, want in zip(dx, dx1):
                        assert np.array_equal(got, want)
                    np.testing.assert_allclose(dw, dw1, rtol=1e-12, atol=1e-12)


def pin_bf16_rounding(orc, quick=False):
    """double -> bf16 on float32-representable values equals torch's float32 -> bf16 (one
    round-to-nearest-even); bf16 -> double equals torch's widening."""
    rng = np.random.default_rng(26)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = np.concatenate([ties - 1, ties + 1])
    special = np.array([0x00000001, 0x00008000, 0x00018000, 0x007F8000, 0x7F7F8000, 0x7F7FFFFF,
                        0x80008000, 0x3F808000, 0x3F818000], dtype=np.uint32)
    allbits = np.concatenate([bits, ties, near, special])
    f = allbits.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.double_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, want), "bf16 rounding differs from torch float32->bf16"
    h = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    wide = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    mine = orc.bf16_to_double(h)
    finite = np.isfinite(wide)
    assert np.array_equal(mine[finite], wide[finite])


PINS = [
    pin_relayout_vs_split_cat,
    pin_relayout_enumeration,
    pin_relayout_vs_pages_base,
    pin_identity_w1,
    pin_round_trip,
    pin_conservation_and_coverage,
    pin_source_query,
    pin_page_shapes,
    pin_rmsnorm_vs_torch,
    pin_rope_vs_complex,
    pin_rope_identities,
    pin_one_hot_rows,
    pin_unit_weight_rms,
    pin_fused_formulations_agree,
    pin_fused_placement_decode,
    pin_qkv_interleaved,
    pin_packed_planes,
    pin_packed_planes_backward,
    pin_fused_bwd_vs_autograd,
    pin_fused_bwd_finite_differences,
    pin_fused_bwd_placement,
    pin_relayout_adjoint,
    pin_f16_decode,
    pin_f16_encode,
    pin_rope_half_vs_complex,
    pin_rope_half_is_permuted_adjacent,
    pin_fused_row_variants,
    pin_fused_var_whole_call,
    pin_fused_bwd_variants,
    pin_fused_bwd_var_whole_call,
    pin_parts_cover_the_call,
    pin_bf16_rounding,
]


def run_all(orc, quick=True):
    """Run every pin; return the names of those that failed (a crash counts as a failure)."""
    failed = []
    for pin in PINS:
        try:
            pin(orc, quick=quick)
        except Exception as exc:  # noqa: BLE001  (any failure is a caught mistake)
            failed.append(f"{pin.__name__}: {type(exc).__name__}")
    return failed
