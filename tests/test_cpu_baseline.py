"""The benchmark's multi-threaded CPU baseline relayout (oracle/segment_memcpy.c) gives the
oracle's bytes exactly, in both modes, for any thread count (no GPU)."""
import numpy as np

import oracle as oracle_pkg


def test_segment_memcpy_matches_oracle(oracle):
    seg = oracle_pkg.SegmentMemcpy()
    assert seg.max_threads() >= 1
    rng = np.random.default_rng(3)
    for trial in range(120):
        W = int(rng.integers(1, 9))
        b = int(rng.integers(1, 3))
        e = int(rng.choice([1, 2, 4]))
        d = int(rng.choice([1, 2, 8, 16]))
        seq = [int(x) for x in rng.integers(0, 600 if trial % 10 == 0 else 5, W)]
        heads = [int(x) for x in rng.integers(0, 4, W)]
        seq[0] += sum(seq) == 0
        heads[-1] += sum(heads) == 0
        dt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[e]
        xs = [rng.integers(0, 2 ** (8 * e), (b, s, sum(heads), d)).astype(dt) for s in seq]
        for mode in (0, 1):
            src = xs if mode == 0 else oracle.a2a_4d(xs, seq, heads, 0)
            want = oracle.a2a_4d(src, seq, heads, mode)
            got = seg.a2a_4d(src, seq, heads, mode, threads=int(rng.integers(0, 5)))
            for r, (g, w) in enumerate(zip(got, want)):
                assert np.array_equal(g, w), (W, b, seq, heads, d, e, mode, r)
