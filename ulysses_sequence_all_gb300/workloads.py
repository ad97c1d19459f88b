"""Seeded synthetic workloads: geometries and input tensors, nothing of the relayout itself.

Both the CUDA path's tests/benchmark and the CPU oracle draw their inputs from here; this module
holds none of the method's arithmetic (no offsets, no index mapping, no normalisation).

Geometries follow the video-DiT shapes the fast-ulysses pages benchmark ("Performance": Wan 720p,
bf16, 8 GPUs) and the FastVideo page ("Ulysses performance on GB200": 250,000 tokens, 56 heads,
head dim 128, sequence parallelism 4, one plane of 896,000,000 bytes per rank). The pages give no
tensor shape for "Wan 720p"; the one used here is 75,600 latent tokens (21 x 45 x 80), 40 heads,
head dim 128.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ELEM_SIZE = {"uint8": 1, "int8": 1, "float8_e4m3fn": 1, "float8_e5m2": 1,
             "float16": 2, "bfloat16": 2, "float32": 4}


def torch_dtype(name: str) -> torch.dtype:
    return getattr(torch, name)


def uneven_head_splits(W: int, N: int = 40) -> list[int]:
    """Heads per rank for the uneven configs: the even split floor(N/W) with the remainder on the
    lowest ranks, then one head moved from the last rank to rank 0. For W=8, N=40 this gives
    [6, 5, 5, 5, 5, 5, 5, 4]."""
    base, rem = divmod(N, W)
    splits = [base + (1 if r < rem else 0) for r in range(W)]
    if W > 1:
        splits[0] += 1
        splits[-1] -= 1
    return splits


def uneven_seq_splits(W: int, S: int = 75000, spread: float = 0.1) -> list[int]:
    """Tokens per rank drawn within +-spread of the even share (numpy default_rng(1000 + W));
    the last rank takes the remainder, redrawn until it is also within the spread."""
    rng = np.random.default_rng(1000 + W)
    even = S / W
    while True:
        head = [int(round(even * (1.0 + rng.uniform(-spread, spread)))) for _ in range(W - 1)]
        last = S - sum(head)
        if abs(last - even) <= spread * even:
            return head + [last]


@dataclass(frozen=True)
class Workload:
    name: str
    W: int
    b: int
    seq_splits: tuple
    head_splits: tuple
    d: int
    dtype: str
    seed: int
    planes: int = 1
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def S(self) -> int:
        return int(sum(self.seq_splits))

    @property
    def N(self) -> int:
        return int(sum(self.head_splits))

    @property
    def elem_size(self) -> int:
        return ELEM_SIZE[self.dtype]

    def seq_side_shape(self, q: int) -> tuple:
        """Rank q's (b, s_q, N, d) tensor: mode 0's input, mode 1's output."""
        return (self.b, int(self.seq_splits[q]), self.N, self.d)

    def head_side_shape(self, r: int) -> tuple:
        """Rank r's (b, S, n_r, d) tensor: mode 0's output, mode 1's input."""
        return (self.b, self.S, int(self.head_splits[r]), self.d)

    def plane_bytes(self) -> int:
        """Bytes of all W ranks' tensors on one side, for one plane."""
        return self.b * self.S * self.N * self.d * self.elem_size

    def relayout_bytes(self) -> int:
        """Algorithmic bytes of one relayout of one plane: every byte read once, written once."""
        return 2 * self.plane_bytes()


TINY = Workload("tiny", 2, 1, (16, 16), (4, 4), 128, "bfloat16", seed=0)
WAN = Workload("wan720p", 8, 1, (9450,) * 8, (5,) * 8, 128, "bfloat16", seed=1)
LONG_QKV = Workload("long_qkv", 4, 1, (62500,) * 4, (14,) * 4, 128, "bfloat16", seed=20, planes=3)
FUSED = Workload("fused_qk", 8, 1, (9450,) * 8, (5,) * 8, 128, "bfloat16", seed=3,
                 extra={"k_seed": 4, "w_seed": 2, "eps": 1e-6, "theta": 1e4})


def uneven(W: int, dtype: str) -> Workload:
    return Workload(f"uneven_W{W}_{dtype}", W, 2, tuple(uneven_seq_splits(W)),
                    tuple(uneven_head_splits(W)), 128, dtype, seed=10 + W)


UNEVEN = [uneven(W, dt) for W in (3, 5, 7, 8) for dt in ("float16", "float32", "float8_e4m3fn")]


def _randn(shape, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(torch_dtype(dtype))


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def seq_side_inputs(wl: Workload, device="cpu", seed: int | None = None, plane: int = 0):
    """W tensors shaped (b, s_q, N, d), values ~N(0, 1) cast to the workload's dtype; rank q of
    plane p uses the sub-seed 100 * seed + 10 * p + q."""
    seed = wl.seed if seed is None else seed
    return [_randn(wl.seq_side_shape(q), wl.dtype, make_generator(100 * seed + 10 * plane + q, device),
                   device) for q in range(wl.W)]


def head_side_inputs(wl: Workload, device="cpu", seed: int | None = None, plane: int = 0):
    """W tensors shaped (b, S, n_r, d) for mode 1, values ~N(0, 1); rank r uses the sub-seed
    100 * seed + 50 + 10 * p + r."""
    seed = wl.seed if seed is None else seed
    return [_randn(wl.head_side_shape(r), wl.dtype,
                   make_generator(100 * seed + 50 + 10 * plane + r, device), device)
            for r in range(wl.W)]


def rms_weights(d: int, seed: int = 2) -> torch.Tensor:
    """fp32 weights of shape (2, d): row 0 for q, row 1 for k, each ~N(1, 0.1)."""
    g = make_generator(seed, "cpu")
    return 1.0 + 0.1 * torch.randn((2, d), generator=g, dtype=torch.float32)


def split_sizes_note(wl: Workload) -> dict:
    return {"seq_splits": list(wl.seq_splits), "head_splits": list(wl.head_splits)}
