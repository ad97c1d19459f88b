"""The CPU oracle against its pins (no GPU). Each pin is described in ``oracle_pins.py``."""
import numpy as np
import pytest

import oracle_pins
from oracle_pins import _golden_lines, _kv
from ulysses_sequence_all_gb300 import workloads as wl


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle, pin):
    pin(oracle, quick=False)


def test_fastvideo_plane_bytes_golden():
    """FastVideo "Ulysses performance on GB200": 250,000 tokens, 56 heads, d=128, bf16, SP=4 is
    896,000,000 bytes per plane per rank, under the 1 GiB window."""
    lines = {name: (_kv(inp), _kv(exp)) for name, inp, exp in _golden_lines()}
    inp, exp = lines["fastvideo_plane"]
    cfg = wl.LONG_QKV
    assert cfg.S == int(inp["tokens"]) and cfg.N == int(inp["heads"]) and cfg.d == int(inp["d"])
    assert cfg.W == int(inp["sp"]) and cfg.elem_size == int(inp["elem_bytes"])
    per_rank = int(np.prod(cfg.seq_side_shape(0))) * cfg.elem_size
    assert per_rank == int(exp["plane_bytes_per_rank"]) == 896_000_000
    assert per_rank <= int(exp["window_bytes"]) == 1 << 30


def test_uneven_split_readings():
    assert wl.uneven_head_splits(8) == [6, 5, 5, 5, 5, 5, 5, 4]
    assert wl.uneven_head_splits(3) == [15, 13, 12]
    assert wl.uneven_head_splits(5) == [9, 8, 8, 8, 7]
    assert wl.uneven_head_splits(7) == [7, 6, 6, 6, 6, 5, 4]
    for W in (3, 5, 7, 8):
        s = wl.uneven_seq_splits(W)
        assert sum(s) == 75000 and len(s) == W
        assert all(abs(v - 75000 / W) <= 0.1 * 75000 / W for v in s)
        assert s == wl.uneven_seq_splits(W)  # seeded: the same every time


def test_oracle_rejects_bad_geometry(oracle):
    x = [np.zeros((1, 2, 2, 4), dtype=np.uint16)]
    with pytest.raises(ValueError):
        oracle.a2a_4d(x, [0], [2], 0)          # S = 0
    with pytest.raises(ValueError):
        oracle.a2a_4d(x * 9, [2] * 9, [2] * 9, 0)  # W > 8
