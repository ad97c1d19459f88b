"""Shared helpers of the GPU parity tests: raw-byte host views, guarded output buffers, and the
comparison of device results with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

_TVIEW = {1: torch.uint8, 2: torch.int16, 4: torch.int32}
_NVIEW = {1: np.uint8, 2: np.uint16, 4: np.uint32}
GUARD = 4096
FILL = 0xA5


def host_raw(t: torch.Tensor) -> np.ndarray:
    """The tensor's bytes on the host, as unsigned integers of its element size."""
    e = t.element_size()
    return t.contiguous().view(_TVIEW[e]).cpu().numpy().view(_NVIEW[e])


class GuardedOutputs:
    """Output tensors carved out of larger buffers: GUARD bytes of FILL on each side (checked
    after the kernel ran) and FILL inside, so an unwritten byte shows up in the exact compare."""

    def __init__(self, shapes, dtype: torch.dtype, device="cuda"):
        self.bufs, self.tensors, self.nbytes = [], [], []
        esize = torch.empty((), dtype=dtype).element_size()
        for sh in shapes:
            nb = int(np.prod(sh)) * esize
            buf = torch.full((2 * GUARD + nb,), FILL, dtype=torch.uint8, device=device)
            view = buf[GUARD:GUARD + nb].view(dtype).view(sh)
            self.bufs.append(buf)
            self.tensors.append(view)
            self.nbytes.append(nb)

    def guards_intact(self) -> bool:
        for buf, nb in zip(self.bufs, self.nbytes):
            head = buf[:GUARD]
            tail = buf[GUARD + nb:]
            if not bool((head == FILL).all()) or not bool((tail == FILL).all()):
                return False
        return True


def random_bytes_tensor(shape, dtype: torch.dtype, gen: torch.Generator, device="cuda"):
    """Uniform random bytes of the given shape viewed as `dtype` (NaN patterns included, which
    is why every relayout compare is on raw bytes)."""
    esize = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) * esize
    raw = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=gen, device=device)
    return raw.view(dtype).view(shape)


def assert_same_bytes(got_tensors, want_arrays, what=""):
    assert len(got_tensors) == len(want_arrays)
    for k, (g, w) in enumerate(zip(got_tensors, want_arrays)):
        gh = host_raw(g)
        assert gh.shape == w.shape, f"{what} rank {k}: shape {gh.shape} vs {w.shape}"
        if not np.array_equal(gh, w):
            bad = np.argwhere(gh != w)
            raise AssertionError(f"{what} rank {k}: {len(bad)} elements differ, first at "
                                 f"{tuple(bad[0])}: got {gh[tuple(bad[0])]:#x} want {w[tuple(bad[0])]:#x}")
