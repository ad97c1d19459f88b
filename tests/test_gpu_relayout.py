"""GPU parity of the relayout (modes 0 and 1) through the C ABI against the CPU oracle.

The relayout is a byte move, so every comparison is bit-exact on raw bytes. Outputs sit between
guard bands that must stay untouched, and are prefilled with a sentinel so an unwritten byte
fails the exact compare.
"""
import zlib

import numpy as np
import pytest
import torch

from gpu_util import GuardedOutputs, assert_same_bytes, host_raw, random_bytes_tensor
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ENGINES = {"tma": B.ULY_ENGINE_TMA, "vec": B.ULY_ENGINE_VEC, "ce": B.ULY_ENGINE_CE,
           "tensor": B.ULY_ENGINE_TENSOR}


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()  # raises if the library was not built
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def run(cfg_like, mode, ins, engine=None, cap=None):
    W, b, seq, heads, d, dtype = cfg_like
    plan = B.ulysses_plan(W, b, seq, heads, d, dtype)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    N, S = sum(heads), sum(seq)
    shapes = [(b, S, n, d) for n in heads] if mode == 0 else [(b, s, N, d) for s in seq]
    outs = GuardedOutputs(shapes, wl.torch_dtype(dtype))
    if engine is None:
        B.ulysses_a2a_4d(plan, mode, ins, outs.tensors)
    else:
        B.ulysses_a2a_4d_engine(plan, mode, engine, ins, outs.tensors)
    torch.cuda.synchronize()
    assert outs.guards_intact(), "a kernel wrote outside its output"
    return outs.tensors


def oracle_of(oracle, cfg_like, mode, ins):
    W, b, seq, heads, d, dtype = cfg_like
    return oracle.a2a_4d([host_raw(x) for x in ins], seq, heads, mode)


def geom(cfg):
    return (cfg.W, cfg.b, list(cfg.seq_splits), list(cfg.head_splits), cfg.d, cfg.dtype)


@pytest.mark.parametrize("engine", list(ENGINES))
def test_tiny_round_trip(oracle, engine):
    """W=2, b=1, s_local=16, 8 heads, d=128, bf16 N(0,1) from seed 0: mode 0 matches the oracle
    and mode 1 returns the input bit-exactly."""
    cfg = wl.TINY
    x = [t.cuda() for t in wl.seq_side_inputs(cfg, "cpu")]
    y = run(geom(cfg), 0, x, ENGINES[engine])
    assert_same_bytes(y, oracle_of(oracle, geom(cfg), 0, x), "tiny mode 0")
    z = run(geom(cfg), 1, y, ENGINES[engine])
    for a, b in zip(z, x):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _random_geometries(rng, count):
    dts = {1: ["uint8", "float8_e4m3fn", "int8", "float8_e5m2"], 2: ["bfloat16", "float16"],
           4: ["float32"]}
    out = []
    for _ in range(count):
        W = int(rng.integers(1, 9))
        e = int(rng.choice([1, 2, 4]))
        d = int(rng.choice([16, 32, 64, 128, 256, 512])) // e  # d * e bytes per head
        seq = [int(v) for v in rng.integers(0, 40, size=W)]
        heads = [int(v) for v in rng.integers(0, 7, size=W)]
        if rng.random() < 0.3:  # ranks with nothing to send or receive
            seq[int(rng.integers(0, W))] = 0
            heads[int(rng.integers(0, W))] = 0
        if sum(seq) == 0:
            seq[0] = 3
        if sum(heads) == 0:
            heads[-1] = 2
        out.append((W, int(rng.integers(1, 4)), seq, heads, d, str(rng.choice(dts[e]))))
    return out


GEOMS = _random_geometries(np.random.default_rng(2024), 40) + [
    (1, 2, [37], [5], 128, "bfloat16"),                          # W=1: identity
    (8, 1, [1] * 8, [1] * 8, 8, "float16"),                      # 16-byte runs
    (3, 2, [5, 0, 7], [40, 0, 20], 256, "float32"),              # runs of 40 KiB and 20 KiB
    (2, 1, [3, 2], [70, 1], 128, "float32"),                     # one run of 35 KiB
    (4, 3, [0, 0, 9, 0], [0, 3, 0, 0], 64, "bfloat16"),          # one live segment
    (5, 1, [2, 3, 2, 3, 2], [9, 8, 8, 8, 7], 16, "uint8"),       # d * e = 16
]


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("g", GEOMS, ids=[f"g{i}" for i in range(len(GEOMS))])
def test_random_geometries(oracle, g, engine):
    W, b, seq, heads, d, dtype = g
    gen = torch.Generator(device="cuda")
    gen.manual_seed(zlib.crc32(str(g).encode()))
    td = wl.torch_dtype(dtype)
    N, S = sum(heads), sum(seq)
    for mode in (0, 1):
        shapes = [(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads]
        ins = [random_bytes_tensor(sh, td, gen) for sh in shapes]
        got = run(g, mode, ins, ENGINES[engine])
        assert_same_bytes(got, oracle_of(oracle, g, mode, ins), f"{g} mode {mode}")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("engine", list(ENGINES))
def test_wan720p_full(oracle, engine, mode):
    """W=8, b=1, s_global=75,600 (9,450 per rank), 40 heads (5 per rank), d=128, bf16: every byte
    of every rank against the oracle."""
    cfg = wl.WAN
    ins = (wl.seq_side_inputs(cfg, "cuda") if mode == 0 else wl.head_side_inputs(cfg, "cuda"))
    got = run(geom(cfg), mode, ins, ENGINES[engine])
    assert_same_bytes(got, oracle_of(oracle, geom(cfg), mode, ins), f"wan mode {mode}")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cfg", wl.UNEVEN, ids=lambda c: c.name)
def test_uneven_full(oracle, cfg, mode):
    """W in {3,5,7,8}, b=2, 75,000 tokens split unevenly, 40 heads split unevenly, d=128, fp16 /
    fp32 / fp8 e4m3: every byte against the oracle."""
    ins = (wl.seq_side_inputs(cfg, "cuda") if mode == 0 else wl.head_side_inputs(cfg, "cuda"))
    got = run(geom(cfg), mode, ins)
    assert_same_bytes(got, oracle_of(oracle, geom(cfg), mode, ins), f"{cfg.name} mode {mode}")


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("cap", [1 << 20, 5 << 20, 16 << 20])
def test_chunked_matches_oracle(oracle, cap, engine):
    """A chunk cap far below the tensor sizes splits the call into many launches along the
    sequence shards; the bytes are those of the definition all the same."""
    cfg = wl.uneven(5, "float16")
    g = geom(cfg)
    plan = B.ulysses_plan(*g)
    B.ulysses_plan_set_chunk_bytes(plan, cap)
    assert B.ulysses_plan_num_chunks(plan, 0) > 1
    for mode in (0, 1):
        ins = (wl.seq_side_inputs(cfg, "cuda") if mode == 0 else wl.head_side_inputs(cfg, "cuda"))
        got = run(g, mode, ins, ENGINES[engine], cap=cap)
        assert_same_bytes(got, oracle_of(oracle, g, mode, ins), f"chunked cap={cap} mode {mode}")


def test_long_packed_qkv(oracle):
    """W=4, b=1, 250,000 tokens, 56 heads, d=128, bf16, three planes (Q, K, V) of 896,000,000
    bytes per rank in one packed (3, b, s_local, N, d) buffer per rank, moved one plane at a time
    (one launch each under the 1 GiB cap). Checked per plane: sampled elements against the
    oracle's single-element rule, the mode-1 round trip, and a 64 MiB chunking equal to the
    unchunked result."""
    cfg = wl.LONG_QKV
    g = geom(cfg)
    plan = B.ulysses_plan(*g)
    assert B.ulysses_plan_num_chunks(plan, 0) == 1
    plane_in = B.ulysses_plan_bytes(plan, 0, 0)[0]
    assert plane_in == 896_000_000
    packed_in = [torch.empty((3,) + cfg.seq_side_shape(q), dtype=torch.bfloat16, device="cuda")
                 for q in range(cfg.W)]
    for p in range(3):
        for q, x in enumerate(wl.seq_side_inputs(cfg, "cuda", plane=p)):
            packed_in[q][p].copy_(x)
            del x
    packed_out = [torch.empty((3,) + cfg.head_side_shape(r), dtype=torch.bfloat16, device="cuda")
                  for r in range(cfg.W)]
    rng = np.random.default_rng(7)
    for p in range(3):
        B.ulysses_a2a_4d(plan, 0, [t[p] for t in packed_in], [t[p] for t in packed_out])
    torch.cuda.synchronize()
    for p in range(3):
        ins = [t[p].reshape(-1).view(torch.int16) for t in packed_in]
        for r in range(cfg.W):
            flat_out = packed_out[r][p].reshape(-1).view(torch.int16)
            ks = rng.integers(0, flat_out.numel(), size=4000)
            src = [oracle.a2a_4d_source(cfg.W, cfg.b, g[2], g[3], cfg.d, 0, r, int(k)) for k in ks]
            got = flat_out[torch.as_tensor(ks, device="cuda")].cpu()
            want = torch.stack([ins[q][idx] for q, idx in src]).cpu()
            assert torch.equal(got, want), f"plane {p} rank {r}: sampled elements differ"
    # round trip of plane 1 and chunked == unchunked for plane 2
    back = [torch.empty_like(t[1]) for t in packed_in]
    B.ulysses_a2a_4d(plan, 1, [t[1] for t in packed_out], back)
    torch.cuda.synchronize()
    for a, b in zip(back, packed_in):
        assert torch.equal(a.view(torch.int16), b[1].view(torch.int16))
    del back
    plan_small = B.ulysses_plan(*g)
    B.ulysses_plan_set_chunk_bytes(plan_small, 64 << 20)
    assert B.ulysses_plan_num_chunks(plan_small, 0) >= 14
    chunked = [torch.empty_like(t[2]) for t in packed_out]
    B.ulysses_a2a_4d(plan_small, 0, [t[2] for t in packed_in], chunked)
    torch.cuda.synchronize()
    for a, b in zip(chunked, packed_out):
        assert torch.equal(a.view(torch.int16), b[2].view(torch.int16))


def test_end_to_end_host_buffers(oracle):
    """The host-buffer entry point: pinned host inputs -> device -> relayout -> pinned host outputs."""
    cfg = wl.uneven(3, "float16")
    g = geom(cfg)
    plan = B.ulysses_plan(*g)
    for mode in (0, 1):
        src = (wl.seq_side_inputs(cfg, "cpu") if mode == 0 else wl.head_side_inputs(cfg, "cpu"))
        host_in = [x.pin_memory() for x in src]
        shapes = ([cfg.head_side_shape(r) for r in range(cfg.W)] if mode == 0 else
                  [cfg.seq_side_shape(q) for q in range(cfg.W)])
        host_out = [torch.empty(sh, dtype=torch.float16).pin_memory() for sh in shapes]
        dev_in = [torch.empty_like(x, device="cuda") for x in src]
        dev_out = [torch.empty(sh, dtype=torch.float16, device="cuda") for sh in shapes]
        B.ulysses_a2a_4d_host(plan, mode, host_in, host_out, dev_in, dev_out)
        torch.cuda.synchronize()
        want = oracle.a2a_4d([x.view(torch.int16).numpy().view(np.uint16) for x in src],
                             g[2], g[3], mode)
        for h, w in zip(host_out, want):
            assert np.array_equal(h.view(torch.int16).numpy().view(np.uint16), w)


@pytest.mark.parametrize("g", [(4, 2, [3, 0, 5, 1], [2, 3, 0, 1], 64, "bfloat16"),
                               (3, 1, [7, 2, 9], [1, 1, 2], 16, "float32"),
                               (8, 1, [1] * 8, [5] * 8, 128, "bfloat16")],
                         ids=["zero_splits_b2", "fp32", "one_row_per_rank"])
def test_end_to_end_host_buffers_edges(oracle, g):
    """The chunked host-buffer path on zero splits, b > 1, shards shorter than the chunk count:
    identical to the oracle, and twice in a row on the same buffers."""
    W, b, seq, heads, d, dtype = g
    plan = B.ulysses_plan(*g)
    td = wl.torch_dtype(dtype)
    N, S = sum(heads), sum(seq)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(zlib.crc32(str(g).encode()))
    for mode in (0, 1):
        in_shapes = [(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads]
        out_shapes = [(b, S, n, d) for n in heads] if mode == 0 else [(b, s, N, d) for s in seq]
        src = [torch.randn(sh, generator=gen).to(td) for sh in in_shapes]
        host_in = [x.pin_memory() for x in src]
        host_out = [torch.full(sh, 7, dtype=td).pin_memory() for sh in out_shapes]
        dev_in = [torch.empty(sh, dtype=td, device="cuda") for sh in in_shapes]
        dev_out = [torch.empty(sh, dtype=td, device="cuda") for sh in out_shapes]
        want = oracle.a2a_4d([host_raw(x) for x in src], seq, heads, mode)
        for _ in range(2):
            B.ulysses_a2a_4d_host(plan, mode, host_in, host_out, dev_in, dev_out)
            torch.cuda.synchronize()
            for h, w in zip(host_out, want):
                assert np.array_equal(host_raw(h), w)


@pytest.mark.parametrize("cap", [None, 96 * 1024], ids=["default_ranges", "capped_ranges"])
def test_end_to_end_host_buffers_ranges(oracle, cap):
    """The host pipeline's ranges of the global sequence (a few hundred rows, ranges that cross
    shards of unequal length, b = 2), also when the chunk cap forces many short ranges: identical
    to the oracle in both modes, twice in a row on the same buffers."""
    W, b, seq, heads, d, dtype = 4, 2, [301, 257, 0, 410], [3, 1, 4, 2], 64, "bfloat16"
    plan = B.ulysses_plan(W, b, seq, heads, d, dtype)
    if cap is not None:
        B.ulysses_plan_set_chunk_bytes(plan, cap)
    N, S = sum(heads), sum(seq)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(97)
    for mode in (0, 1):
        in_shapes = [(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads]
        out_shapes = [(b, S, n, d) for n in heads] if mode == 0 else [(b, s, N, d) for s in seq]
        src = [random_bytes_tensor(sh, torch.bfloat16, gen, "cpu") for sh in in_shapes]
        host_in = [x.pin_memory() for x in src]
        host_out = [torch.full(sh, 7, dtype=torch.bfloat16).pin_memory() for sh in out_shapes]
        dev_in = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in in_shapes]
        dev_out = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in out_shapes]
        want = oracle.a2a_4d([host_raw(x) for x in src], seq, heads, mode)
        for _ in range(2):
            B.ulysses_a2a_4d_host(plan, mode, host_in, host_out, dev_in, dev_out)
            torch.cuda.synchronize()
            for h, w in zip(host_out, want):
                assert np.array_equal(host_raw(h), w)


def test_end_to_end_host_copies_wait_for_the_stream(oracle):
    """The host call's copies in run on a stream of their own, but only after the work already
    queued on the caller's stream: a fill of the device inputs queued behind a long wait on that
    stream must not land after the copies in (the result would then be the fill's bytes)."""
    W, b, seq, heads, d = 2, 1, [640, 512], [2, 2], 128
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    N, S = sum(heads), sum(seq)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(98)
    src = [random_bytes_tensor((b, s, N, d), torch.bfloat16, gen, "cpu") for s in seq]
    host_in = [x.pin_memory() for x in src]
    host_out = [torch.zeros((b, S, n, d), dtype=torch.bfloat16).pin_memory() for n in heads]
    dev_in = [torch.empty((b, s, N, d), dtype=torch.bfloat16, device="cuda") for s in seq]
    dev_out = [torch.empty((b, S, n, d), dtype=torch.bfloat16, device="cuda") for n in heads]
    want = oracle.a2a_4d([host_raw(x) for x in src], seq, heads, 0)
    stream = torch.cuda.current_stream()
    torch.cuda._sleep(20_000_000)  # roughly 10 ms of spinning on the caller's stream
    for t in dev_in:
        t.view(torch.int16).fill_(0x7F7F)
    B.ulysses_a2a_4d_host(plan, 0, host_in, host_out, dev_in, dev_out, stream)
    torch.cuda.synchronize()
    for h, w in zip(host_out, want):
        assert np.array_equal(host_raw(h), w)


def test_misaligned_and_overlapping_on_device():
    plan = B.ulysses_plan(2, 1, [4, 4], [2, 2], 64, "bfloat16")
    x = [torch.zeros(1, 4, 4, 64, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    big = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    y = [torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_a2a_4d(plan, 0, x, [big.data_ptr() + 2, y[1]])
    assert ei.value.status == B.ULY_EALIGN
    with pytest.raises(B.UlyssesError) as ei:
        B.ulysses_a2a_4d(plan, 0, x, [x[0], y[1]])
    assert ei.value.status == B.ULY_EOVERLAP


def test_auto_engine_choice():
    """AUTO takes the tensor engine where every run has one length of at most 2048 bytes, or
    under a CTA cap below the SM count when every run fits; the TMA kernel otherwise."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def auto(cfg, cap=0):
        plan = B.ulysses_plan(*geom(cfg))
        B.ulysses_plan_set_max_ctas(plan, cap)
        return B.ulysses_plan_auto_engine(plan)

    by_name = {c.name: c for c in wl.UNEVEN}
    w8_f16, w3_f16 = by_name["uneven_W8_float16"], by_name["uneven_W3_float16"]
    assert auto(wl.WAN) == B.ULY_ENGINE_TENSOR  # runs of 1,280 bytes
    assert auto(wl.TINY) == B.ULY_ENGINE_TENSOR
    assert auto(w8_f16) == B.ULY_ENGINE_TMA  # runs 1,024 to 1,536 bytes
    assert auto(w8_f16, cap=sms // 2) == B.ULY_ENGINE_TENSOR
    assert auto(w8_f16, cap=sms) == B.ULY_ENGINE_TMA  # a cap at the SM count caps nothing
    assert auto(w3_f16, cap=sms // 2) == B.ULY_ENGINE_TMA  # runs above 2,048 bytes
    assert auto(wl.LONG_QKV) == B.ULY_ENGINE_TMA  # 3,584-byte runs
