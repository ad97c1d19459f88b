"""Plain CPU oracle for the Ulysses 4D sequence/head relayout and its fused QK variant.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and has no CPU fallback.

The arithmetic lives in ``ulysses_oracle.c`` (six nested loops for the relayout, double precision
for RMSNorm + RoPE); this module only compiles it with gcc and marshals numpy arrays through
ctypes. What is computed, and the passages it follows:

* fast-ulysses 0.1.0 (PyPI page), opening paragraph and "Quick start": mode 0 maps
  ``(b, s_local, n_global, d) -> (b, s_global, n_local, d)``.
* fast-ulysses 0.2.1 (README), "Quick start": mode 1 returns to x's shape.
* fast-ulysses 0.1.0, "What it does": uneven per-rank ``seq_splits`` / ``head_splits``.
* fast-ulysses 0.1.0, "Fusion examples": QK RMSNorm + RoPE inside the scatter.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "ulysses_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")
SEGMENT_SOURCE = os.path.join(HERE, "segment_memcpy.c")
SEGMENT_LIBRARY = os.path.join(HERE, "libsegment_memcpy.so")

_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_pi64 = ctypes.POINTER(ctypes.c_int64)


def build(out: str = LIBRARY, source: str = SOURCE) -> str:
    """Compile the oracle with gcc into a shared library and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", out, source, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build_segment(out: str = SEGMENT_LIBRARY, source: str = SEGMENT_SOURCE) -> str:
    """Compile the multi-threaded CPU baseline relayout (segment_memcpy.c, OpenMP)."""
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fopenmp", "-shared", "-fPIC", "-o", out, source]
    subprocess.run(cmd, check=True)
    return out


def build_all() -> None:
    """Everything in this directory that compiles: the oracle and the CPU baseline relayout."""
    build()
    build_segment()


def _needs_build(lib: str, source: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(source)


def _i64_array(values: Sequence[int]):
    return (ctypes.c_int64 * len(values))(*[int(v) for v in values])


def _ptr_array(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


_PART = [ctypes.c_int, ctypes.c_int, _i64, _i64]  # q_lo, q_hi, i_lo, i_hi
_WHOLE = (0, None, 0, 2 ** 63 - 1)


def _parts(seq_splits, threads: int):
    """(q_lo, q_hi, i_lo, i_hi) ranges that cover every (shard, row) of a call once: each shard's
    rows cut into about 4 * threads / W pieces, so that `threads` workers stay busy."""
    W = len(seq_splits)
    per = max(1, -(-4 * threads // W))
    out = []
    for q, s in enumerate(seq_splits):
        s = int(s)
        step = max(1, -(-s // per))
        for lo in range(0, s, step):
            out.append((q, q + 1, lo, min(s, lo + step)))
    return out


def _run_parts(call, seq_splits, threads: int):
    """call(q_lo, q_hi, i_lo, i_hi) -> status, over the whole call (threads <= 1) or its parts on
    a pool of host threads (the oracle's C functions run without the interpreter lock)."""
    if threads <= 1:
        q_lo, _, i_lo, i_hi = _WHOLE
        return [call(q_lo, len(seq_splits), i_lo, i_hi)]
    parts = _parts(seq_splits, threads)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        return list(pool.map(lambda pr: call(*pr), parts))


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a test's planted variant)."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = LIBRARY
            if _needs_build(lib_path, SOURCE):
                build(lib_path, SOURCE)
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        lib.orc_a2a_4d.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, _i64, ctypes.c_int, _p, _p]
        lib.orc_a2a_4d.restype = ctypes.c_int
        lib.orc_a2a_4d_source.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int,
                                           ctypes.c_int, _i64, ctypes.POINTER(ctypes.c_int), _pi64]
        lib.orc_a2a_4d_source.restype = ctypes.c_int
        fused_args = [ctypes.c_int, _i64, _pi64, _pi64, _i64, _p, _p, ctypes.c_double,
                      ctypes.c_double, _p]
        for name in ("orc_qk_fused_A", "orc_qk_fused_B"):
            getattr(lib, name).argtypes = fused_args
            getattr(lib, name).restype = ctypes.c_int
        lib.orc_qk_fused_A_part.argtypes = fused_args + _PART
        lib.orc_qk_fused_A_part.restype = ctypes.c_int
        lib.orc_qk_fused_row.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int, _i64,
                                         _i64, _i64, _p, _p, ctypes.c_double, ctypes.c_double, _p]
        lib.orc_qk_fused_row.restype = ctypes.c_int
        lib.orc_qkv_fused.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, _p, _p, _p,
                                      ctypes.c_double, ctypes.c_double, _p, _p, _p]
        lib.orc_qkv_fused.restype = ctypes.c_int
        lib.orc_qkv_fused_part.argtypes = lib.orc_qkv_fused.argtypes + _PART
        lib.orc_qkv_fused_part.restype = ctypes.c_int
        lib.orc_packed_fused.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, _i64, _p, _p, _p,
                                         ctypes.c_double, ctypes.c_double, _p, _p, _p]
        lib.orc_packed_fused.restype = ctypes.c_int
        lib.orc_packed_fused_bwd.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, _i64, _p, _p, _p, _p,
                                             ctypes.c_double, ctypes.c_double, _p, _p]
        lib.orc_packed_fused_bwd.restype = ctypes.c_int
        lib.orc_fused_row_bwd.argtypes = [_p, _p, _i64, _p, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, _p, _p]
        lib.orc_fused_row_bwd.restype = None
        lib.orc_qk_fused_bwd.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, _p, _p, _p,
                                         ctypes.c_double, ctypes.c_double, _p, _p]
        lib.orc_qk_fused_bwd.restype = ctypes.c_int
        lib.orc_qk_fused_bwd_part.argtypes = lib.orc_qk_fused_bwd.argtypes + _PART
        lib.orc_qk_fused_bwd_part.restype = ctypes.c_int
        lib.orc_rmsnorm.argtypes = [_p, _i64, _p, ctypes.c_double, _p]
        lib.orc_rmsnorm.restype = None
        lib.orc_rope.argtypes = [_p, _i64, ctypes.c_double, ctypes.c_double]
        lib.orc_rope.restype = None
        lib.orc_bf16_to_double_array.argtypes = [_p, _i64, _p]
        lib.orc_bf16_to_double_array.restype = None
        lib.orc_double_to_bf16_array.argtypes = [_p, _i64, _p]
        lib.orc_double_to_bf16_array.restype = None
        lib.orc_f16_to_double_array.argtypes = [_p, _i64, _p]
        lib.orc_f16_to_double_array.restype = None
        lib.orc_double_to_f16_array.argtypes = [_p, _i64, _p]
        lib.orc_double_to_f16_array.restype = None
        lib.orc_rope_half.argtypes = [_p, _i64, ctypes.c_double, ctypes.c_double]
        lib.orc_rope_half.restype = None
        lib.orc_fused_row_var.argtypes = [_p, _i64, ctypes.c_int, ctypes.c_int, _p, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_double, _p]
        lib.orc_fused_row_var.restype = None
        lib.orc_qk_fused_var.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int,
                                         ctypes.c_int, _p, _p, ctypes.c_double, ctypes.c_double, _p]
        lib.orc_qk_fused_var.restype = ctypes.c_int
        lib.orc_qk_fused_var_part.argtypes = lib.orc_qk_fused_var.argtypes + _PART
        lib.orc_qk_fused_var_part.restype = ctypes.c_int
        lib.orc_fused_row_bwd_var.argtypes = [_p, _p, _i64, ctypes.c_int, _p, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_double, _p, _p]
        lib.orc_fused_row_bwd_var.restype = None
        lib.orc_qk_fused_bwd_var.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, ctypes.c_int,
                                             ctypes.c_int, _p, _p, _p, ctypes.c_double,
                                             ctypes.c_double, _p, _p]
        lib.orc_qk_fused_bwd_var.restype = ctypes.c_int
        lib.orc_qk_fused_bwd_var_part.argtypes = lib.orc_qk_fused_bwd_var.argtypes + _PART
        lib.orc_qk_fused_bwd_var_part.restype = ctypes.c_int
        self.lib = lib

    # ---- relayout -------------------------------------------------------------------------
    @staticmethod
    def out_shapes(b, seq_splits, head_splits, d, mode):
        """Shapes the definition gives each rank's output (mode 0: (b, S, n_r, d))."""
        S, N = int(sum(seq_splits)), int(sum(head_splits))
        if mode == 0:
            return [(b, S, int(n), d) for n in head_splits]
        return [(b, int(s), N, d) for s in seq_splits]

    def a2a_4d(self, xs: Sequence[np.ndarray], seq_splits, head_splits, mode: int):
        """Relayout W host arrays (any dtype; moved as raw bytes). Returns W new arrays."""
        W = len(xs)
        b, d = xs[0].shape[0], xs[0].shape[3]
        e = xs[0].dtype.itemsize
        xs = [np.ascontiguousarray(x) for x in xs]
        outs = [np.empty(s, dtype=xs[0].dtype) for s in self.out_shapes(b, seq_splits, head_splits, d, mode)]
        rc = self.lib.orc_a2a_4d(W, b, _i64_array(seq_splits), _i64_array(head_splits), d, e, mode,
                                 ctypes.cast(_ptr_array(xs), _p), ctypes.cast(_ptr_array(outs), _p))
        if rc != 0:
            raise ValueError("oracle rejected the geometry")
        return outs

    def a2a_4d_raw(self, W, b, seq_splits, head_splits, d, e, mode, in_ptrs, out_ptrs):
        """Same as ``a2a_4d`` on raw host addresses (the caller sizes the buffers)."""
        rc = self.lib.orc_a2a_4d(W, b, _i64_array(seq_splits), _i64_array(head_splits), d, e, mode,
                                 ctypes.cast((ctypes.c_void_p * W)(*in_ptrs), _p),
                                 ctypes.cast((ctypes.c_void_p * W)(*out_ptrs), _p))
        if rc != 0:
            raise ValueError("oracle rejected the geometry")

    def a2a_4d_source(self, W, b, seq_splits, head_splits, d, mode, out_rank, out_elem):
        """(source rank, flat source element index) of one output element."""
        src_rank = ctypes.c_int(-1)
        src_elem = ctypes.c_int64(-1)
        rc = self.lib.orc_a2a_4d_source(W, b, _i64_array(seq_splits), _i64_array(head_splits), d,
                                        mode, out_rank, int(out_elem), ctypes.byref(src_rank),
                                        ctypes.byref(src_elem))
        if rc != 0:
            raise ValueError("oracle rejected the query")
        return src_rank.value, src_elem.value

    # ---- fused QK RMSNorm + RoPE ----------------------------------------------------------
    def _fused(self, fn, xs_bf16: Sequence[np.ndarray], seq_splits, head_splits, w, eps, theta,
               part_fn=None, threads=1):
        W = len(xs_bf16)
        b, d = xs_bf16[0].shape[0], xs_bf16[0].shape[3]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in xs_bf16]
        w64 = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        outs = [np.empty(s, dtype=np.float64) for s in self.out_shapes(b, seq_splits, head_splits, d, 0)]
        args = (W, b, _i64_array(seq_splits), _i64_array(head_splits), d,
                ctypes.cast(_ptr_array(xs), _p), w64.ctypes.data, float(eps), float(theta),
                ctypes.cast(_ptr_array(outs), _p))
        if part_fn is None:
            rcs = [fn(*args)]
        else:
            rcs = _run_parts(lambda *pr: part_fn(*args, *pr), seq_splits, threads)
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected the geometry")
        return outs

    def qk_fused_A(self, xs_bf16, seq_splits, head_splits, w, eps, theta, threads=1):
        """Transform at the source row, then place (unrounded double outputs). threads > 1 splits
        the call into parts (ranges of shards and rows) computed on that many host threads; the
        result is the same array."""
        return self._fused(self.lib.orc_qk_fused_A, xs_bf16, seq_splits, head_splits, w, eps, theta,
                           part_fn=self.lib.orc_qk_fused_A_part, threads=threads)

    def qk_fused_B(self, xs_bf16, seq_splits, head_splits, w, eps, theta):
        """Place the bf16 bytes, then transform at the destination row."""
        return self._fused(self.lib.orc_qk_fused_B, xs_bf16, seq_splits, head_splits, w, eps, theta)

    def qk_fused_row(self, xs_bf16, seq_splits, head_splits, w, eps, theta, r, bb, s, h):
        """One output row (rank r, batch bb, global position s, local head h) in double."""
        W = len(xs_bf16)
        b, d = xs_bf16[0].shape[0], xs_bf16[0].shape[3]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in xs_bf16]
        w64 = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        y = np.empty(d, dtype=np.float64)
        rc = self.lib.orc_qk_fused_row(W, b, _i64_array(seq_splits), _i64_array(head_splits), d, r,
                                       bb, s, h, ctypes.cast(_ptr_array(xs), _p), w64.ctypes.data,
                                       float(eps), float(theta), y.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected the query")
        return y

    def qkv_fused(self, qkv_bf16, seq_splits, head_splits, wq, wk, eps, theta, threads=1):
        """Interleaved (b, s_q, 3, N, d) inputs: q and k transformed and placed (double), v placed
        unchanged (uint16 bf16 bits). Returns (q_outs, k_outs, v_outs), each rank r (b, S, n_r, d).
        threads > 1: computed in parts on that many host threads (same result)."""
        W = len(qkv_bf16)
        b, d = qkv_bf16[0].shape[0], qkv_bf16[0].shape[4]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in qkv_bf16]
        wq64 = np.ascontiguousarray(np.asarray(wq, dtype=np.float64))
        wk64 = np.ascontiguousarray(np.asarray(wk, dtype=np.float64))
        shapes = self.out_shapes(b, seq_splits, head_splits, d, 0)
        qo = [np.empty(s, dtype=np.float64) for s in shapes]
        ko = [np.empty(s, dtype=np.float64) for s in shapes]
        vo = [np.empty(s, dtype=np.uint16) for s in shapes]
        args = (W, b, _i64_array(seq_splits), _i64_array(head_splits), d,
                ctypes.cast(_ptr_array(xs), _p), wq64.ctypes.data, wk64.ctypes.data, float(eps),
                float(theta), ctypes.cast(_ptr_array(qo), _p), ctypes.cast(_ptr_array(ko), _p),
                ctypes.cast(_ptr_array(vo), _p))
        if threads <= 1:
            rcs = [self.lib.orc_qkv_fused(*args)]
        else:
            rcs = _run_parts(lambda *pr: self.lib.orc_qkv_fused_part(*args, *pr), seq_splits, threads)
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected the geometry")
        return qo, ko, vo

    def packed_fused(self, packed, seq_splits, head_splits, d, planes, q_plane, k_plane, pitch,
                     wq, wk, eps, theta):
        """Packed inputs: rank q's array holds b * s_q tokens of `pitch` elements (uint16 bit
        patterns, any shape whose leading axes are (b, s_q)); plane c's head g of a token is at
        element c * N * d + g * d. Returns (q_outs, k_outs, plain_outs): the q and k planes
        transformed and placed (double), plain_outs[c] the other planes placed unchanged (uint16;
        None for the q and k planes); each rank r (b, S, n_r, d)."""
        W = len(packed)
        b = packed[0].shape[0]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in packed]
        wq64 = np.ascontiguousarray(np.asarray(wq, dtype=np.float64))
        wk64 = np.ascontiguousarray(np.asarray(wk, dtype=np.float64))
        shapes = self.out_shapes(b, seq_splits, head_splits, d, 0)
        qo = [np.empty(s, dtype=np.float64) for s in shapes]
        ko = [np.empty(s, dtype=np.float64) for s in shapes]
        plain = [None if c in (q_plane, k_plane) else [np.empty(s, dtype=np.uint16) for s in shapes]
                 for c in range(planes)]
        dummy = np.empty(1, dtype=np.uint16)
        flat = [plain[c][r] if plain[c] is not None else dummy for c in range(planes) for r in range(W)]
        rc = self.lib.orc_packed_fused(W, b, _i64_array(seq_splits), _i64_array(head_splits), d,
                                       planes, q_plane, k_plane, pitch,
                                       ctypes.cast(_ptr_array(xs), _p), wq64.ctypes.data,
                                       wk64.ctypes.data, float(eps), float(theta),
                                       ctypes.cast(_ptr_array(qo), _p),
                                       ctypes.cast(_ptr_array(ko), _p),
                                       ctypes.cast(_ptr_array(flat), _p))
        if rc != 0:
            raise ValueError("oracle rejected the geometry")
        return qo, ko, plain

    def packed_fused_bwd(self, packed, grads, seq_splits, head_splits, d, planes, q_plane, k_plane,
                         pitch, wq, wk, eps, theta):
        """Backward of packed_fused: packed (rank q's b * s_q tokens of `pitch` uint16 elements,
        leading axes (b, s_q)), grads[c][r] rank r's gradient of plane c's output (uint16 bf16 bit
        patterns, (b, S, n_r, d)). Returns (dpacked, dw): dpacked[q] a double array shaped like
        packed[q] (columns beyond the planes NaN: never written), dw (2, d)."""
        W = len(packed)
        b = packed[0].shape[0]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in packed]
        gs = [np.ascontiguousarray(grads[c][r]).view(np.uint16) for c in range(planes)
              for r in range(W)]
        wq64 = np.ascontiguousarray(np.asarray(wq, dtype=np.float64))
        wk64 = np.ascontiguousarray(np.asarray(wk, dtype=np.float64))
        dx = [np.full(x.shape, np.nan) for x in xs]
        dw = np.full(2 * d, np.nan)  # the oracle clears it
        rc = self.lib.orc_packed_fused_bwd(W, b, _i64_array(seq_splits), _i64_array(head_splits),
                                           d, planes, q_plane, k_plane, pitch,
                                           ctypes.cast(_ptr_array(xs), _p),
                                           ctypes.cast(_ptr_array(gs), _p), wq64.ctypes.data,
                                           wk64.ctypes.data, float(eps), float(theta),
                                           ctypes.cast(_ptr_array(dx), _p), dw.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected the geometry")
        return dx, dw.reshape(2, d)

    def fused_row_bwd(self, x, g, w, eps, p, theta):
        """(dL/dx, dL/dw) of one row y = R(p)(x * w / rms(x)) for dL/dy = g, in double."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = np.ascontiguousarray(g, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        dx = np.empty_like(x)
        dw = np.zeros_like(x)
        self.lib.orc_fused_row_bwd(x.ctypes.data, g.ctypes.data, x.size, w.ctypes.data,
                                   float(eps), float(p), float(theta), dx.ctypes.data, dw.ctypes.data)
        return dx, dw

    def qk_fused_bwd(self, x_bf16, g_bf16, seq_splits, head_splits, w, eps, theta, threads=1):
        """Backward of the fused mode-0 call for one tensor: forward inputs x (rank q's
        (b, s_q, N, d) bf16) and output gradients g (rank r's (b, S, n_r, d) bf16). Returns
        (dx per rank in double, (b, s_q, N, d); dw, d values). threads > 1: computed in parts on
        that many host threads; dx is the same array, dw the parts' sums added in part order."""
        W = len(x_bf16)
        b, d = x_bf16[0].shape[0], x_bf16[0].shape[3]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in x_bf16]
        gs = [np.ascontiguousarray(x).view(np.uint16) for x in g_bf16]
        w64 = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        dx = [np.empty(x.shape, dtype=np.float64) for x in xs]
        args = (W, b, _i64_array(seq_splits), _i64_array(head_splits), d,
                ctypes.cast(_ptr_array(xs), _p), ctypes.cast(_ptr_array(gs), _p), w64.ctypes.data,
                float(eps), float(theta), ctypes.cast(_ptr_array(dx), _p))
        return dx, self._bwd_parts(self.lib.orc_qk_fused_bwd, self.lib.orc_qk_fused_bwd_part,
                                   args, seq_splits, d, threads)

    @staticmethod
    def _bwd_parts(whole_fn, part_fn, args, seq_splits, d, threads):
        """dw of a backward call (its dx is written through args): the whole call, or one dw per
        part (each cleared by the oracle) added in part order."""
        if threads <= 1:
            dw = np.full(d, np.nan)  # the oracle clears it
            if whole_fn(*args, dw.ctypes.data) != 0:
                raise ValueError("oracle rejected the geometry")
            return dw
        parts = _parts(seq_splits, threads)
        dws = [np.full(d, np.nan) for _ in parts]

        def run(k):
            return part_fn(*args, dws[k].ctypes.data, *parts[k])

        with ThreadPoolExecutor(max_workers=threads) as pool:
            rcs = list(pool.map(run, range(len(parts))))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected the geometry")
        dw = np.zeros(d)
        for x in dws:
            dw += x
        return dw

    def rmsnorm(self, x, w, eps):
        x = np.ascontiguousarray(x, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.orc_rmsnorm(x.ctypes.data, x.size, w.ctypes.data, float(eps), y.ctypes.data)
        return y

    def rope(self, y, p, theta):
        y = np.array(y, dtype=np.float64, copy=True)
        self.lib.orc_rope(y.ctypes.data, y.size, float(p), float(theta))
        return y

    def bf16_to_double(self, h):
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.orc_bf16_to_double_array(h.ctypes.data, h.size, out.ctypes.data)
        return out

    def double_to_bf16(self, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.orc_double_to_bf16_array(x.ctypes.data, x.size, out.ctypes.data)
        return out


    # ---- variants of the fused call: fp16 elements, rotate-half pairs ----------------------
    def f16_to_double(self, h):
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.orc_f16_to_double_array(h.ctypes.data, h.size, out.ctypes.data)
        return out

    def double_to_f16(self, x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.orc_double_to_f16_array(x.ctypes.data, x.size, out.ctypes.data)
        return out

    def decode(self, h, f16):
        """Element bit patterns (uint16) -> double, bf16 or fp16."""
        return self.f16_to_double(h) if f16 else self.bf16_to_double(h)

    def rope_half(self, y, p, theta):
        y = np.array(y, dtype=np.float64, copy=True)
        self.lib.orc_rope_half(y.ctypes.data, y.size, float(p), float(theta))
        return y

    def fused_row_var(self, x_raw, f16, half_pairs, w, eps, p, theta):
        """One row of a variant: decode, RMSNorm, RoPE (adjacent or rotate-half pairs)."""
        x = np.ascontiguousarray(x_raw).view(np.uint16)
        w = np.ascontiguousarray(w, dtype=np.float64)
        y = np.empty(x.size, dtype=np.float64)
        self.lib.orc_fused_row_var(x.ctypes.data, x.size, int(f16), int(half_pairs), w.ctypes.data,
                                   float(eps), float(p), float(theta), y.ctypes.data)
        return y

    def qk_fused_var(self, xs, seq_splits, head_splits, w, eps, theta, f16, half_pairs, threads=1):
        """The fused call of a variant for one tensor (unrounded double outputs); threads > 1:
        computed in parts on that many host threads (same result)."""
        W = len(xs)
        b, d = xs[0].shape[0], xs[0].shape[3]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in xs]
        w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        outs = [np.empty(sh, dtype=np.float64)
                for sh in self.out_shapes(b, seq_splits, head_splits, d, 0)]
        args = (W, b, _i64_array(seq_splits), _i64_array(head_splits), d, int(f16),
                int(half_pairs), ctypes.cast(_ptr_array(xs), _p), w.ctypes.data, float(eps),
                float(theta), ctypes.cast(_ptr_array(outs), _p))
        if threads <= 1:
            rcs = [self.lib.orc_qk_fused_var(*args)]
        else:
            rcs = _run_parts(lambda *pr: self.lib.orc_qk_fused_var_part(*args, *pr), seq_splits,
                             threads)
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected the geometry")
        return outs

    def fused_row_bwd_var(self, x, g, half_pairs, w, eps, p, theta):
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = np.ascontiguousarray(g, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        dx = np.empty_like(x)
        dw = np.zeros_like(x)
        self.lib.orc_fused_row_bwd_var(x.ctypes.data, g.ctypes.data, x.size, int(half_pairs),
                                       w.ctypes.data, float(eps), float(p), float(theta),
                                       dx.ctypes.data, dw.ctypes.data)
        return dx, dw

    def qk_fused_bwd_var(self, xs, gs, seq_splits, head_splits, w, eps, theta, f16, half_pairs,
                         threads=1):
        """Backward of a variant's fused call for one tensor: (dx per rank in double, dw);
        threads > 1 as qk_fused_bwd."""
        W = len(xs)
        b, d = xs[0].shape[0], xs[0].shape[3]
        xs = [np.ascontiguousarray(x).view(np.uint16) for x in xs]
        gs = [np.ascontiguousarray(x).view(np.uint16) for x in gs]
        w64 = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        dx = [np.empty(x.shape, dtype=np.float64) for x in xs]
        args = (W, b, _i64_array(seq_splits), _i64_array(head_splits), d, int(f16), int(half_pairs),
                ctypes.cast(_ptr_array(xs), _p), ctypes.cast(_ptr_array(gs), _p), w64.ctypes.data,
                float(eps), float(theta), ctypes.cast(_ptr_array(dx), _p))
        return dx, self._bwd_parts(self.lib.orc_qk_fused_bwd_var, self.lib.orc_qk_fused_bwd_var_part,
                                   args, seq_splits, d, threads)


class SegmentMemcpy:
    """ctypes view of segment_memcpy.c: the relayout as one memcpy per (row, destination rank) run,
    rows shared among OpenMP threads. A timed CPU baseline, not the oracle; the tests check its
    bytes against the oracle's relayout."""

    def __init__(self):
        if _needs_build(SEGMENT_LIBRARY, SEGMENT_SOURCE):
            build_segment()
        lib = ctypes.CDLL(SEGMENT_LIBRARY)
        lib.seg_a2a_4d.argtypes = [ctypes.c_int, _i64, _pi64, _pi64, _i64, _i64, ctypes.c_int, _p,
                                   _p, ctypes.c_int]
        lib.seg_a2a_4d.restype = ctypes.c_int
        lib.seg_max_threads.argtypes = []
        lib.seg_max_threads.restype = ctypes.c_int
        self.lib = lib

    def max_threads(self) -> int:
        return int(self.lib.seg_max_threads())

    def a2a_4d(self, xs, seq_splits, head_splits, mode: int, threads: int = 0, outs=None):
        """Relayout W host arrays (raw bytes of any dtype) into `outs` (allocated when None)."""
        W = len(xs)
        b, d = xs[0].shape[0], xs[0].shape[3]
        e = xs[0].dtype.itemsize
        xs = [np.ascontiguousarray(x) for x in xs]
        if outs is None:
            outs = [np.empty(sh, dtype=xs[0].dtype)
                    for sh in Oracle.out_shapes(b, seq_splits, head_splits, d, mode)]
        rc = self.lib.seg_a2a_4d(W, b, _i64_array(seq_splits), _i64_array(head_splits), d, e, mode,
                                 ctypes.cast(_ptr_array(xs), _p), ctypes.cast(_ptr_array(outs), _p),
                                 int(threads))
        if rc != 0:
            raise ValueError("segment relayout rejected the geometry")
        return outs


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``ulysses_oracle.c`` (compiled on first use if needed)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
