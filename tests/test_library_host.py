"""Host-only checks of libulysses.so (no GPU): the library loads and exports every symbol that
include/ulysses.h declares; the host plan validates, sizes and chunks as documented; argument
errors are reported before any CUDA call is made."""
import ctypes
import os
import re

import pytest

from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from ulysses_sequence_all_gb300 import build
    if not os.path.exists(B.LIBRARY) or any(
            os.path.getmtime(os.path.join(build.CSRC, s)) > os.path.getmtime(B.LIBRARY)
            for s in os.listdir(build.CSRC)):
        build.build_library()
    return B.library()


def header_functions():
    with open(os.path.join(ROOT, "include", "ulysses.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(ulysses_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol():
    declared = header_functions()
    assert len(declared) >= 14
    lib = ctypes.CDLL(B.LIBRARY)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in ulysses.h but not exported"
    assert sorted(B.EXPORTS) == declared


def test_version_and_strerror():
    assert B.ulysses_version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert B.ulysses_strerror(code) != "unknown status"


def test_plan_bytes_match_shapes():
    for cfg in [wl.TINY, wl.WAN, wl.LONG_QKV] + wl.UNEVEN:
        plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
        for k in range(cfg.W):
            seq_b = cfg.b * cfg.seq_splits[k] * cfg.N * cfg.d * cfg.elem_size
            head_b = cfg.b * cfg.S * cfg.head_splits[k] * cfg.d * cfg.elem_size
            assert B.ulysses_plan_bytes(plan, 0, k) == (seq_b, head_b)
            assert B.ulysses_plan_bytes(plan, 1, k) == (head_b, seq_b)


def test_fastvideo_plane_is_one_chunk():
    """FastVideo, "Ulysses performance on GB200": 896,000,000 bytes per plane fit the 1 GiB
    window, so a plane is one launch."""
    cfg = wl.LONG_QKV
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    assert B.ulysses_plan_bytes(plan, 0, 0)[0] == 896_000_000
    assert B.ulysses_plan_num_chunks(plan, 0) == 1
    assert B.ulysses_plan_num_chunks(plan, 1) == 1


@pytest.mark.parametrize("cap", [1 << 20, 3 << 20, 64 << 20, 300 << 20])
@pytest.mark.parametrize("cfg", [wl.WAN, wl.uneven(7, "float32"), wl.uneven(3, "float8_e4m3fn")],
                         ids=lambda c: getattr(c, "name", c))
def test_chunks_cover_rows_and_respect_cap(cfg, cap):
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    B.ulysses_plan_set_chunk_bytes(plan, cap)
    C = B.ulysses_plan_num_chunks(plan, 0)
    row = cfg.d * cfg.elem_size
    nxt = [0] * cfg.W
    for c in range(C):
        lo, cnt = B.ulysses_plan_chunk_rows(plan, 0, c)
        assert lo == nxt, "chunks must tile each shard in order, without gaps"
        nxt = [a + b for a, b in zip(lo, cnt)]
        for q in range(cfg.W):
            assert cfg.b * cnt[q] * cfg.N * row <= cap          # rank q's seq-side bytes
        for r in range(cfg.W):
            assert cfg.b * sum(cnt) * cfg.head_splits[r] * row <= cap  # rank r's head side
    assert nxt == list(cfg.seq_splits)
    if C > 1:  # minimality under the per-shard ceil bound
        assert cap < max(cfg.b * -(-s // (C - 1)) * cfg.N * row for s in cfg.seq_splits) or \
            cap < max(cfg.b * sum(-(-s // (C - 1)) for s in cfg.seq_splits) * n * row
                      for n in cfg.head_splits)


def test_chunk_cap_below_one_row_is_rejected():
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    B.ulysses_plan_set_chunk_bytes(plan, 100)   # one row is 4 heads * 128 bytes
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_plan_num_chunks(plan, 0)
    assert ei.value.status == B.ULY_ECHUNK


@pytest.mark.parametrize("args,status", [
    ((0, 1, [], [], 128, "bfloat16"), B.ULY_EINVAL),              # W = 0
    ((9, 1, [1] * 9, [1] * 9, 128, "bfloat16"), B.ULY_EINVAL),    # W > 8
    ((2, 0, [1, 1], [1, 1], 128, "bfloat16"), B.ULY_EINVAL),      # b = 0
    ((2, 1, [0, 0], [1, 1], 128, "bfloat16"), B.ULY_EINVAL),      # S = 0
    ((2, 1, [1, 1], [0, 0], 128, "bfloat16"), B.ULY_EINVAL),      # N = 0
    ((2, 1, [-1, 2], [1, 1], 128, "bfloat16"), B.ULY_EINVAL),     # negative split
    ((2, 1, [1, 1], [1, 1], 12, "bfloat16"), B.ULY_EALIGN),       # d * 2 = 24 bytes
    ((2, 1, [1, 1], [1, 1], 8, "float8_e4m3fn"), B.ULY_EALIGN),   # d * 1 = 8 bytes
    ((2, 1, [1, 1], [1, 1], 128, 99), B.ULY_EINVAL),              # unknown dtype
])
def test_plan_rejects(args, status):
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_plan(*args)
    assert ei.value.status == status


def test_plan_accepts_pages_limits():
    """World sizes 1..8 including odd ones, every listed dtype with d * elem 16-byte aligned."""
    for W in range(1, 9):
        B.ulysses_plan(W, 1, [3] * W, [2] * W, 128, "bfloat16")
    for dt, d in (("float16", 8), ("bfloat16", 8), ("float32", 4), ("float8_e4m3fn", 16),
                  ("float8_e5m2", 16), ("int8", 16), ("uint8", 16)):
        B.ulysses_plan(2, 1, [1, 1], [1, 1], d, dt)


def _fake_ptrs(base, sizes, align=256):
    out, cur = [], base
    for s in sizes:
        out.append(cur)
        cur += (s + align - 1) // align * align + align
    return out


def test_launch_argument_errors_before_cuda():
    """Misaligned, missing and overlapping pointers are refused on the host (no GPU needed:
    these checks run before the first CUDA call)."""
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    in_b = [B.ulysses_plan_bytes(plan, 0, k)[0] for k in range(2)]
    out_b = [B.ulysses_plan_bytes(plan, 0, k)[1] for k in range(2)]
    ins = _fake_ptrs(1 << 40, in_b)
    outs = _fake_ptrs(1 << 41, out_b)
    cases = [
        (0, [ins[0] + 8, ins[1]], outs, B.ULY_EALIGN),
        (0, ins, [outs[0], outs[1] + 4], B.ULY_EALIGN),
        (0, [0, ins[1]], outs, B.ULY_EINVAL),
        (0, ins, [ins[0], outs[1]], B.ULY_EOVERLAP),             # output aliases an input
        (0, ins, [outs[0], outs[0] + 256], B.ULY_EOVERLAP),      # outputs overlap
        (2, ins, outs, B.ULY_EINVAL),                            # bad mode
    ]
    for mode, i, o, status in cases:
        with pytest.raises(B.UlyssesError) as ei:
            B.ulysses_a2a_4d(plan, mode, i, o, stream=0)
        assert ei.value.status == status, (mode, status)
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_a2a_4d_engine(plan, 0, 7, ins, outs, stream=0)
    assert ei.value.status == B.ULY_EINVAL


def test_rope_pairs_setter():
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_HALF)
    B.ulysses_plan_set_rope_pairs(plan, B.ULY_ROPE_ADJACENT)
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_plan_set_rope_pairs(plan, 2)
    assert ei.value.status == B.ULY_EINVAL


def test_max_ctas_setter():
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    B.ulysses_plan_set_max_ctas(plan, 0)
    B.ulysses_plan_set_max_ctas(plan, 17)
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_plan_set_max_ctas(plan, -1)
    assert ei.value.status == B.ULY_EINVAL


def test_fused_engine_setter():
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    for engine in (B.ULY_ENGINE_AUTO, B.ULY_ENGINE_TMA, B.ULY_ENGINE_TENSOR):
        B.ulysses_plan_set_fused_engine(plan, engine)
    for engine in (B.ULY_ENGINE_VEC, B.ULY_ENGINE_CE, 9, -1):
        with pytest.raises(B.UlyssesError) as ei:
            B.ulysses_plan_set_fused_engine(plan, engine)
        assert ei.value.status == B.ULY_EINVAL


def test_fused_kernel_choice():
    """The fused forward's kernel, decided on the host: the row-block kernel for equal head groups
    with runs of at most 2,048 bytes, rows of at most 10,240 bytes and a power-of-two d, else the
    token units."""
    def kernel(W, heads, d, dtype="bfloat16", engine=None):
        plan = B.ulysses_plan(W, 1, [8] * W, heads, d, dtype)
        if engine is not None:
            B.ulysses_plan_set_fused_engine(plan, engine)
        return B.ulysses_plan_fused_kernel(plan)

    T, K = B.ULY_ENGINE_TENSOR, B.ULY_ENGINE_TMA
    assert kernel(8, [5] * 8, 128) == T                    # Wan-720p: rows of 10,240 bytes
    assert kernel(4, [4] * 4, 128) == T
    assert kernel(8, [8] * 8, 64, "float16") == T
    assert kernel(8, [4] * 8, 256) == K                    # rows of 16,384 bytes
    assert kernel(8, [4] * 8, 256, engine=T) == T          # forced: it fits (runs of 2,048)
    assert kernel(5, [9, 8, 8, 8, 7], 128) == K            # unequal head groups
    assert kernel(5, [9, 8, 8, 8, 7], 128, engine=T) == K  # does not fit: token units
    assert kernel(2, [9, 9], 128) == K                     # runs of 2,304 bytes
    assert kernel(8, [5] * 8, 128, engine=K) == K
    assert kernel(2, [64, 64], 128, engine=T) == K         # runs of 16 KiB: token units
    assert kernel(8, [5] * 8, 72) == K                     # d not a power of two: token units
    assert kernel(8, [5] * 8, 72, engine=T) == T           # forced: it fits
    assert kernel(5, [9, 8, 8, 8, 7], 72, engine=T) == K
    assert kernel(8, [5] * 8, 96, engine=K) == K
    lib = B.library()
    engine = ctypes.c_int()
    assert lib.ulysses_plan_fused_kernel(None, ctypes.byref(engine)) == B.ULY_EINVAL


def test_fused_backward_kernel_choice():
    """The backward's kernel: row blocks for equal head groups with runs of at most 2,048 bytes
    and rows of at least 6,144 bytes, else token units; the plan's setting overrides."""
    def kernel(W, heads, d, dtype="bfloat16", engine=None):
        plan = B.ulysses_plan(W, 1, [8] * W, heads, d, dtype)
        if engine is not None:
            B.ulysses_plan_set_fused_engine(plan, engine)
        return B.ulysses_plan_fused_backward_kernel(plan)

    T, K = B.ULY_ENGINE_TENSOR, B.ULY_ENGINE_TMA
    assert kernel(8, [5] * 8, 128) == T                    # Wan-720p: rows of 10,240 bytes
    assert kernel(8, [4] * 8, 256) == T                    # rows of 16,384 bytes
    assert kernel(4, [14] * 4, 64) == T                    # rows of 7,168 bytes
    assert kernel(4, [4] * 4, 128) == K                    # rows of 4,096 bytes
    assert kernel(4, [4] * 4, 128, engine=T) == T          # forced: it fits
    assert kernel(5, [9, 8, 8, 8, 7], 128, engine=T) == K  # unequal head groups
    assert kernel(8, [5] * 8, 128, engine=K) == K
    assert kernel(8, [8] * 8, 120) == T                    # d = 120: rows of 15,360 bytes
    assert kernel(8, [5] * 8, 72) == K                     # rows of 5,760 bytes
    assert kernel(8, [5] * 8, 72, engine=T) == T
    engine = ctypes.c_int()
    assert B.library().ulysses_plan_fused_backward_kernel(None, ctypes.byref(engine)) == B.ULY_EINVAL


def test_auto_engine_argument_errors():
    lib = B.library()
    engine = ctypes.c_int()
    assert lib.ulysses_plan_auto_engine(None, ctypes.byref(engine)) == B.ULY_EINVAL
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    assert lib.ulysses_plan_auto_engine(plan, None) == B.ULY_EINVAL


def test_fused_argument_errors_before_cuda():
    plan32 = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "float32")
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    plan_d = B.ulysses_plan(2, 1, [4, 4], [2, 2], 264, "bfloat16")  # d above the fused calls' 256
    in_b = [B.ulysses_plan_bytes(plan, 0, k)[0] for k in range(2)]
    out_b = [B.ulysses_plan_bytes(plan, 0, k)[1] for k in range(2)]
    q, k = _fake_ptrs(1 << 40, in_b), _fake_ptrs(1 << 39, in_b)
    qo, ko = _fake_ptrs(1 << 41, out_b), _fake_ptrs(1 << 42, out_b)
    w = 1 << 43
    for p, args, status in [
        (plan32, (q, k, qo, ko, w, 1e-6, 1e4), B.ULY_EINVAL),   # neither bf16 nor fp16
        (plan_d, (q, k, qo, ko, w, 1e-6, 1e4), B.ULY_EINVAL),   # unsupported d
        (plan, (q, k, qo, ko, w + 4, 1e-6, 1e4), B.ULY_EALIGN), # weights misaligned
        (plan, (q, k, qo, ko, 0, 1e-6, 1e4), B.ULY_EINVAL),     # no weights
        (plan, (q, k, qo, ko, w, -1.0, 1e4), B.ULY_EINVAL),     # eps < 0
        (plan, (q, k, qo, ko, w, 1e-6, 0.0), B.ULY_EINVAL),     # theta <= 0
        (plan, (q, k, q, ko, w, 1e-6, 1e4), B.ULY_EOVERLAP),    # q_out aliases q_in
        (plan, (q, k, qo, qo, w, 1e-6, 1e4), B.ULY_EOVERLAP),   # k_out aliases q_out
    ]:
        with pytest.raises(B.UlyssesError) as ei:
            B.ulysses_a2a_4d_qk_fused(p, *args, stream=0)
        assert ei.value.status == status


def test_fused_sequence_limit_before_cuda():
    """Positions travel as exact fp32 integers, so the fused calls take S < 2^24: a plan of
    exactly 2^24 tokens is refused on the host (the relayout itself has no such limit)."""
    plan = B.ulysses_plan(2, 1, [1 << 23, 1 << 23], [1, 1], 8, "bfloat16")
    in_b = [B.ulysses_plan_bytes(plan, 0, k)[0] for k in range(2)]
    out_b = [B.ulysses_plan_bytes(plan, 0, k)[1] for k in range(2)]
    q, k = _fake_ptrs(1 << 40, in_b), _fake_ptrs(1 << 39, in_b)
    qo, ko = _fake_ptrs(1 << 41, out_b), _fake_ptrs(1 << 42, out_b)
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, 1 << 43, 1e-6, 1e4, stream=0)
    assert ei.value.status == B.ULY_EINVAL
    packed = _fake_ptrs(1 << 44, [2 * x for x in in_b])
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_a2a_4d_packed_fused(plan, 2, 0, 1, 2 * 8 * 2 * 2, packed, [qo, ko], 1 << 43,
                                      1e-6, 1e4, stream=0)
    assert ei.value.status == B.ULY_EINVAL


def test_packed_argument_errors_before_cuda():
    """The packed fused call refuses bad plane counts and roles, a short or unaligned token pitch,
    and overlapping outputs on the host."""
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    row = 4 * 64 * 2                                  # one plane of one token: N * d * e bytes
    out_b = [B.ulysses_plan_bytes(plan, 0, k)[1] for k in range(2)]
    w = 1 << 43

    def call(planes, qp, kp, pitch, outs=None):
        ins = _fake_ptrs(1 << 40, [4 * pitch] * 2)
        outs = outs or [_fake_ptrs((1 << 41) + (c << 30), out_b) for c in range(planes)]
        B.ulysses_a2a_4d_packed_fused(plan, planes, qp, kp, pitch, ins, outs, w, 1e-6, 1e4,
                                      stream=0)

    for args, status in [
        ((1, 0, 1, row), B.ULY_EINVAL),          # fewer than two planes
        ((9, 0, 1, 9 * row), B.ULY_EINVAL),      # more than eight
        ((3, 1, 1, 3 * row), B.ULY_EINVAL),      # q and k the same plane
        ((3, 0, 3, 3 * row), B.ULY_EINVAL),      # k plane out of range
        ((3, -1, 1, 3 * row), B.ULY_EINVAL),     # q plane out of range
        ((3, 0, 1, 3 * row - 16), B.ULY_EINVAL), # pitch shorter than the planes
        ((3, 0, 1, 3 * row + 8), B.ULY_EALIGN),  # pitch not a multiple of 16 bytes
        ((3, 0, 1, 1 << 31), B.ULY_EINVAL),      # pitch of 2 GiB or more
    ]:
        with pytest.raises(B.UlyssesError) as ei:
            call(*args)
        assert ei.value.status == status, args
    same = _fake_ptrs(1 << 41, out_b)
    with pytest.raises(B.UlyssesError) as ei:        # two planes' outputs on the same buffers
        call(3, 0, 1, 3 * row, outs=[same, same, _fake_ptrs(1 << 42, out_b)])
    assert ei.value.status == B.ULY_EOVERLAP
