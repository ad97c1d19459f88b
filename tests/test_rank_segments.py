"""The plan's per-rank share of the exchange (ulysses_plan_rank_segments), the description a
transport running the ranks on separate GPUs would move bytes by (no GPU here: the plan is host
only, and the ranks are processes exchanging over gloo on the CPU).

* Single process: applying every rank's segments with numpy strided copies reproduces the oracle's
  relayout byte for byte, and writes every output byte exactly once.
* Several processes (gloo, world sizes 2 and 3): each process is one rank holding only its own
  tensor; it packs its segments, the ranks exchange them with one all-to-all, and each unpacks what
  it received with the senders' descriptors. Every rank's result equals the oracle's for that rank.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from ulysses_sequence_all_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rows(seg, b):
    """(source byte index, destination byte index) arrays of one segment, row by row."""
    src, dst = [], []
    for bb in range(b):
        for i in range(seg["rows"]):
            s0 = seg["src_offset"] + bb * seg["src_batch_pitch"] + i * seg["src_row_pitch"]
            d0 = seg["dst_offset"] + bb * seg["dst_batch_pitch"] + i * seg["dst_row_pitch"]
            src.append(np.arange(s0, s0 + seg["row_bytes"]))
            dst.append(np.arange(d0, d0 + seg["row_bytes"]))
    if not src:
        return np.zeros(0, dtype=np.int64), np.zeros(0, dtype=np.int64)
    return np.concatenate(src), np.concatenate(dst)


def _inputs(W, b, seq, heads, d, mode, seed):
    rng = np.random.default_rng(seed)
    N, S = sum(heads), sum(seq)
    shapes = [(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads]
    return [rng.integers(0, 1 << 16, sh, dtype=np.uint16) for sh in shapes]


GEOMS = [(2, 1, [3, 2], [2, 1], 8), (3, 2, [2, 0, 3], [1, 2, 1], 16), (4, 1, [1, 2, 1, 2], [2, 0, 1, 1], 8),
         (5, 2, [3, 1, 4, 1, 5], [2, 1, 1, 3, 1], 8), (1, 1, [4], [3], 8)]


@pytest.mark.parametrize("g", GEOMS, ids=[f"g{i}" for i in range(len(GEOMS))])
@pytest.mark.parametrize("mode", [0, 1])
def test_segments_reproduce_the_relayout(oracle, g, mode):
    W, b, seq, heads, d = g
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    xs = _inputs(W, b, seq, heads, d, mode, seed=7 * W + mode)
    want = oracle.a2a_4d(xs, seq, heads, mode)
    outs = [np.zeros(w.nbytes, dtype=np.uint8) for w in want]
    writes = [np.zeros(w.nbytes, dtype=np.int64) for w in want]
    for rank in range(W):
        src_bytes = xs[rank].view(np.uint8).reshape(-1)
        for seg in B.ulysses_plan_rank_segments(plan, mode, rank):
            si, di = _rows(seg, b)
            outs[seg["peer"]][di] = src_bytes[si]
            np.add.at(writes[seg["peer"]], di, 1)
    for r in range(W):
        assert np.array_equal(outs[r], want[r].view(np.uint8).reshape(-1)), f"rank {r}"
        assert np.all(writes[r] == 1), f"rank {r}: a byte written {writes[r].max()} times or never"


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, g, mode, results):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import oracle as oracle_pkg
    from ulysses_sequence_all_gb300 import binding as Bw
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        W, b, seq, heads, d = g
        plan = Bw.ulysses_plan(W, b, seq, heads, d, "bfloat16")
        xs = _inputs(W, b, seq, heads, d, mode, seed=11 * W + mode)  # every rank's, seeded
        mine = xs[rank].view(np.uint8).reshape(-1)                 # this rank keeps only its own
        # pack: the segments for ranks 0 .. W-1, back to back
        segs = Bw.ulysses_plan_rank_segments(plan, mode, rank)
        parts = [mine[_rows(s, b)[0]] for s in segs]
        send = torch.from_numpy(np.concatenate(parts).copy())
        # what this rank receives from each sender: that sender's segment addressed to it
        incoming = [Bw.ulysses_plan_rank_segments(plan, mode, src)[rank] for src in range(W)]
        recv_sizes = [b * s["rows"] * s["row_bytes"] for s in incoming]
        recv = torch.empty(sum(recv_sizes), dtype=torch.uint8)
        dist.all_to_all_single(recv, send, output_split_sizes=recv_sizes,
                               input_split_sizes=[p.numel() for p in map(torch.from_numpy, parts)])
        want = oracle_pkg.get().a2a_4d(xs, seq, heads, mode)[rank].view(np.uint8).reshape(-1)
        out = np.zeros(want.size, dtype=np.uint8)
        at = 0
        got = recv.numpy()
        for s, n in zip(incoming, recv_sizes):
            out[_rows(s, b)[1]] = got[at:at + n]
            at += n
        results[rank] = bool(np.array_equal(out, want))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("g", [(2, 2, [5, 3], [3, 1], 8), (3, 1, [2, 0, 4], [1, 2, 2], 16)],
                         ids=["world2", "world3"])
@pytest.mark.parametrize("mode", [0, 1])
def test_segments_exchanged_between_processes(g, mode):
    world = g[0]
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, port, g, mode, results), nprocs=world, join=True)
    assert all(results[r] for r in range(world)), dict(results)
