"""Thin ctypes binding of libulysses.so: the C ABI of include/ulysses.h under the same names.

Only argument marshalling happens here (torch tensors -> device pointers, Python lists -> C
arrays, status codes -> exceptions); every step of the relayout runs in the library's kernels.
Loading fails loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.environ.get("ULYSSES_LIBRARY", os.path.join(PKG, "libulysses.so"))

ULY_OK, ULY_EINVAL, ULY_EALIGN, ULY_EOVERLAP, ULY_ECHUNK, ULY_ECUDA, ULY_ENOMEM, ULY_EDEVICE = (
    0, -1, -2, -3, -4, -5, -6, -7)
ULY_ESCRATCH = -8
ULYSSES_STATIC_SCRATCH_BYTES = 2 * 1024 * 1024
ULY_U8, ULY_F8E4M3, ULY_F8E5M2, ULY_I8, ULY_F16, ULY_BF16, ULY_F32 = 1, 2, 3, 4, 5, 6, 7
ULY_ENGINE_AUTO, ULY_ENGINE_TMA, ULY_ENGINE_VEC, ULY_ENGINE_CE, ULY_ENGINE_TENSOR = 0, 1, 2, 3, 4
ULY_ROPE_ADJACENT, ULY_ROPE_HALF = 0, 1

DTYPE_CODES = {"uint8": ULY_U8, "float8_e4m3fn": ULY_F8E4M3, "float8_e5m2": ULY_F8E5M2,
               "int8": ULY_I8, "float16": ULY_F16, "bfloat16": ULY_BF16, "float32": ULY_F32}

# Every symbol include/ulysses.h declares.
EXPORTS = ["ulysses_plan", "ulysses_plan_destroy", "ulysses_plan_set_chunk_bytes",
           "ulysses_plan_set_max_ctas", "ulysses_plan_set_rope_pairs",
           "ulysses_plan_bytes", "ulysses_plan_num_chunks", "ulysses_plan_chunk_rows",
           "ulysses_plan_auto_engine", "ulysses_plan_set_fused_engine", "ulysses_plan_fused_kernel",
           "ulysses_plan_fused_backward_kernel",
           "ulysses_plan_rank_segments",
           "ulysses_a2a_4d", "ulysses_a2a_4d_engine", "ulysses_a2a_4d_qk_fused",
           "ulysses_a2a_4d_qkv_fused", "ulysses_a2a_4d_packed_fused",
           "ulysses_a2a_4d_qk_fused_backward",
           "ulysses_qk_fused_backward_workspace", "ulysses_a2a_4d_qk_fused_backward_static",
           "ulysses_a2a_4d_qkv_fused_backward", "ulysses_a2a_4d_packed_fused_backward",
           "ulysses_a2a_4d_host", "ulysses_a2a_4d_qk_fused_host", "ulysses_device_status",
           "ulysses_selftest_wait_timeout", "ulysses_last_cuda_error", "ulysses_strerror",
           "ulysses_version"]


class UlyssesError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib().ulysses_strerror(status).decode()
        if status == ULY_ECUDA:
            msg += f" (cudaError {_lib().ulysses_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{status}]" if what else f"{msg} [{status}]")


_LIB = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_pp = ctypes.POINTER(ctypes.c_void_p)


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(f"libulysses.so is not built ({LIBRARY}); run "
                               "`python -m ulysses_sequence_all_gb300.build` first")
        lib = ctypes.CDLL(LIBRARY)
        lib.ulysses_plan.argtypes = [ctypes.c_int, _i64, ctypes.POINTER(_i64), ctypes.POINTER(_i64),
                                     _i64, ctypes.c_int, ctypes.POINTER(_p)]
        lib.ulysses_plan_destroy.argtypes = [_p]
        lib.ulysses_plan_set_chunk_bytes.argtypes = [_p, _i64]
        lib.ulysses_plan_set_max_ctas.argtypes = [_p, _i64]
        lib.ulysses_plan_set_rope_pairs.argtypes = [_p, ctypes.c_int]
        lib.ulysses_plan_bytes.argtypes = [_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_i64),
                                           ctypes.POINTER(_i64)]
        lib.ulysses_plan_num_chunks.argtypes = [_p, ctypes.c_int, ctypes.POINTER(_i64)]
        lib.ulysses_plan_auto_engine.argtypes = [_p, ctypes.POINTER(ctypes.c_int)]
        lib.ulysses_plan_set_fused_engine.argtypes = [_p, ctypes.c_int]
        lib.ulysses_plan_fused_kernel.argtypes = [_p, ctypes.POINTER(ctypes.c_int)]
        lib.ulysses_plan_fused_backward_kernel.argtypes = [_p, ctypes.POINTER(ctypes.c_int)]
        lib.ulysses_plan_chunk_rows.argtypes = [_p, ctypes.c_int, _i64, ctypes.POINTER(_i64),
                                                ctypes.POINTER(_i64)]
        lib.ulysses_plan_rank_segments.argtypes = [_p, ctypes.c_int, ctypes.c_int, _p]
        lib.ulysses_a2a_4d.argtypes = [_p, ctypes.c_int, _pp, _pp, _p]
        lib.ulysses_a2a_4d_engine.argtypes = [_p, ctypes.c_int, ctypes.c_int, _pp, _pp, _p]
        lib.ulysses_a2a_4d_qk_fused.argtypes = [_p, _pp, _pp, _pp, _pp, _p, ctypes.c_float,
                                                ctypes.c_float, _p]
        lib.ulysses_a2a_4d_qkv_fused.argtypes = [_p, _pp, _pp, _pp, _pp, _p, ctypes.c_float,
                                                 ctypes.c_float, _p]
        lib.ulysses_a2a_4d_packed_fused.argtypes = [_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    _i64, _pp, _pp, _p, ctypes.c_float,
                                                    ctypes.c_float, _p]
        lib.ulysses_a2a_4d_qk_fused_backward.argtypes = [_p, _pp, _pp, _pp, _pp, _pp, _pp, _p, _p,
                                                         ctypes.c_float, ctypes.c_float, _p,
                                                         ctypes.c_size_t, _p]
        lib.ulysses_qk_fused_backward_workspace.argtypes = [_p, ctypes.POINTER(ctypes.c_size_t)]
        lib.ulysses_a2a_4d_qkv_fused_backward.argtypes = [_p, _pp, _pp, _pp, _pp, _pp, _p, _p,
                                                          ctypes.c_float, ctypes.c_float, _p,
                                                          ctypes.c_size_t, _p]
        lib.ulysses_a2a_4d_packed_fused_backward.argtypes = [_p, ctypes.c_int, ctypes.c_int,
                                                             ctypes.c_int, _i64, _pp, _pp, _pp, _p,
                                                             _p, ctypes.c_float, ctypes.c_float,
                                                             _p, ctypes.c_size_t, _p]
        lib.ulysses_a2a_4d_qk_fused_backward_static.argtypes = [_p, _pp, _pp, _pp, _pp, _pp, _pp,
                                                                _p, _p, ctypes.c_float,
                                                                ctypes.c_float, _p]
        lib.ulysses_a2a_4d_host.argtypes = [_p, ctypes.c_int, _pp, _pp, _pp, _pp, _p]
        lib.ulysses_a2a_4d_qk_fused_host.argtypes = [_p, _pp, _pp, _pp, _pp, _pp, _pp, _pp, _pp, _p,
                                                     ctypes.c_float, ctypes.c_float, _p]
        lib.ulysses_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.ulysses_selftest_wait_timeout.argtypes = [ctypes.c_uint, _p]
        lib.ulysses_last_cuda_error.argtypes = []
        lib.ulysses_strerror.argtypes = [ctypes.c_int]
        lib.ulysses_strerror.restype = ctypes.c_char_p
        lib.ulysses_version.argtypes = []
        for name in EXPORTS:
            if name != "ulysses_strerror":
                getattr(lib, name).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    return _lib()


def _check(status: int, what: str):
    if status != ULY_OK:
        raise UlyssesError(status, what)


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()  # torch.Tensor


def _nbytes(x) -> int:
    """Size in bytes of a torch tensor (0 for None)."""
    if x is None:
        return 0
    return x.numel() * x.element_size()


def _ptrs(xs: Sequence) -> ctypes.Array:
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


class Plan:
    """Owns one ulysses_plan_t (host memory only)."""

    def __init__(self, handle: int, W: int, b: int, seq_splits, head_splits, d: int, dtype: str):
        self.handle = handle
        self.W, self.b, self.d, self.dtype = W, b, d, dtype
        self.seq_splits, self.head_splits = list(seq_splits), list(head_splits)

    def __del__(self):
        if getattr(self, "handle", None) and _LIB is not None:
            _LIB.ulysses_plan_destroy(self.handle)
            self.handle = None

    @property
    def _as_parameter_(self):
        return ctypes.c_void_p(self.handle)


def ulysses_plan(W: int, b: int, seq_splits, head_splits, d: int, dtype: str) -> Plan:
    out = ctypes.c_void_p()
    code = DTYPE_CODES.get(dtype, dtype if isinstance(dtype, int) else -1)
    _check(_lib().ulysses_plan(W, b, (_i64 * W)(*seq_splits), (_i64 * W)(*head_splits), d, code,
                               ctypes.byref(out)), "ulysses_plan")
    return Plan(out.value, W, b, seq_splits, head_splits, d, dtype)


def ulysses_plan_set_chunk_bytes(plan: Plan, max_chunk_bytes: int):
    _check(_lib().ulysses_plan_set_chunk_bytes(plan, max_chunk_bytes), "ulysses_plan_set_chunk_bytes")


def ulysses_plan_set_rope_pairs(plan: Plan, pairs: int):
    """RoPE pair layout of the fused calls with this plan: ULY_ROPE_ADJACENT or ULY_ROPE_HALF."""
    _check(_lib().ulysses_plan_set_rope_pairs(plan, pairs), "ulysses_plan_set_rope_pairs")


def ulysses_plan_set_max_ctas(plan: Plan, max_ctas: int):
    """Cap the CTAs of every launch with this plan (0: no cap)."""
    _check(_lib().ulysses_plan_set_max_ctas(plan, max_ctas), "ulysses_plan_set_max_ctas")


def ulysses_plan_set_fused_engine(plan: Plan, engine: int):
    """Kernel of the fused calls (forward, separate or packed, and their backward): ULY_ENGINE_AUTO,
    ULY_ENGINE_TMA (token units) or ULY_ENGINE_TENSOR (blocks of whole rows, grouped by head group
    through one tensor-map copy)."""
    _check(_lib().ulysses_plan_set_fused_engine(plan, engine), "ulysses_plan_set_fused_engine")


def ulysses_plan_fused_kernel(plan: Plan) -> int:
    """The kernel the fused forward with separate q and k takes for this plan: ULY_ENGINE_TENSOR
    (row blocks through tensor maps) or ULY_ENGINE_TMA (token units)."""
    e = ctypes.c_int()
    _check(_lib().ulysses_plan_fused_kernel(plan, ctypes.byref(e)), "ulysses_plan_fused_kernel")
    return e.value


def ulysses_plan_fused_backward_kernel(plan: Plan) -> int:
    """The kernel the fused call's backward takes for this plan: ULY_ENGINE_TENSOR (row blocks)
    or ULY_ENGINE_TMA (token units)."""
    e = ctypes.c_int()
    _check(_lib().ulysses_plan_fused_backward_kernel(plan, ctypes.byref(e)),
           "ulysses_plan_fused_backward_kernel")
    return e.value


def ulysses_plan_bytes(plan: Plan, mode: int, rank: int):
    i, o = _i64(), _i64()
    _check(_lib().ulysses_plan_bytes(plan, mode, rank, ctypes.byref(i), ctypes.byref(o)),
           "ulysses_plan_bytes")
    return i.value, o.value


def ulysses_plan_auto_engine(plan: Plan) -> int:
    """The engine ULY_ENGINE_AUTO takes for this plan on the current device (ULY_ENGINE_TENSOR or
    ULY_ENGINE_TMA)."""
    e = ctypes.c_int()
    _check(_lib().ulysses_plan_auto_engine(plan, ctypes.byref(e)), "ulysses_plan_auto_engine")
    return e.value


def ulysses_plan_num_chunks(plan: Plan, mode: int = 0) -> int:
    n = _i64()
    _check(_lib().ulysses_plan_num_chunks(plan, mode, ctypes.byref(n)), "ulysses_plan_num_chunks")
    return n.value


def ulysses_plan_chunk_rows(plan: Plan, mode: int, chunk: int):
    lo, cnt = (_i64 * plan.W)(), (_i64 * plan.W)()
    _check(_lib().ulysses_plan_chunk_rows(plan, mode, chunk, lo, cnt), "ulysses_plan_chunk_rows")
    return list(lo), list(cnt)


SEGMENT_FIELDS = ("peer", "rows", "row_bytes", "src_offset", "src_row_pitch", "src_batch_pitch",
                  "dst_offset", "dst_row_pitch", "dst_batch_pitch")


def ulysses_plan_rank_segments(plan: Plan, mode: int, rank: int) -> list:
    """The W segments rank `rank` sends in `mode`, as dicts of the ulysses_segment_t fields."""
    W = len(plan.seq_splits)
    buf = (ctypes.c_int64 * (W * len(SEGMENT_FIELDS)))()
    _check(_lib().ulysses_plan_rank_segments(plan, mode, rank, buf), "ulysses_plan_rank_segments")
    n = len(SEGMENT_FIELDS)
    return [dict(zip(SEGMENT_FIELDS, buf[k * n:(k + 1) * n])) for k in range(W)]


def ulysses_a2a_4d(plan: Plan, mode: int, ins: Sequence, outs: Sequence, stream=None):
    _check(_lib().ulysses_a2a_4d(plan, mode, _ptrs(ins), _ptrs(outs), _stream(stream)),
           "ulysses_a2a_4d")


def ulysses_a2a_4d_engine(plan: Plan, mode: int, engine: int, ins: Sequence, outs: Sequence,
                          stream=None):
    _check(_lib().ulysses_a2a_4d_engine(plan, mode, engine, _ptrs(ins), _ptrs(outs), _stream(stream)),
           "ulysses_a2a_4d_engine")


def ulysses_a2a_4d_qk_fused(plan: Plan, q_in, k_in, q_out, k_out, rms_w, eps: float,
                            rope_theta: float, stream=None):
    _check(_lib().ulysses_a2a_4d_qk_fused(plan, _ptrs(q_in), _ptrs(k_in), _ptrs(q_out), _ptrs(k_out),
                                          _addr(rms_w), eps, rope_theta, _stream(stream)),
           "ulysses_a2a_4d_qk_fused")


def ulysses_a2a_4d_qkv_fused(plan: Plan, qkv_in, q_out, k_out, v_out, rms_w, eps: float,
                             rope_theta: float, stream=None):
    _check(_lib().ulysses_a2a_4d_qkv_fused(plan, _ptrs(qkv_in), _ptrs(q_out), _ptrs(k_out),
                                           _ptrs(v_out), _addr(rms_w), eps, rope_theta,
                                           _stream(stream)), "ulysses_a2a_4d_qkv_fused")


def ulysses_a2a_4d_packed_fused(plan: Plan, planes: int, q_plane: int, k_plane: int,
                                token_pitch: int, packed_in, outs, rms_w, eps: float,
                                rope_theta: float, stream=None):
    """outs: one sequence of W output tensors per plane (planes lists), flattened plane-major."""
    flat = [t for plane in outs for t in plane]
    _check(_lib().ulysses_a2a_4d_packed_fused(plan, planes, q_plane, k_plane, token_pitch,
                                              _ptrs(packed_in), _ptrs(flat), _addr(rms_w), eps,
                                              rope_theta, _stream(stream)),
           "ulysses_a2a_4d_packed_fused")


def ulysses_qk_fused_backward_workspace(plan: Plan) -> int:
    """Workspace bytes ulysses_a2a_4d_qk_fused_backward needs for `plan` on the current device."""
    n = ctypes.c_size_t()
    _check(_lib().ulysses_qk_fused_backward_workspace(plan, ctypes.byref(n)),
           "ulysses_qk_fused_backward_workspace")
    return n.value


def ulysses_a2a_4d_qk_fused_backward(plan: Plan, dq_out, dk_out, q_in, k_in, dq_in, dk_in, rms_w,
                                     dw, eps: float, rope_theta: float, workspace, stream=None):
    """Backward of the fused call. `workspace` is a device tensor of at least
    ulysses_qk_fused_backward_workspace(plan) bytes."""
    _check(_lib().ulysses_a2a_4d_qk_fused_backward(
        plan, _ptrs(dq_out), _ptrs(dk_out), _ptrs(q_in), _ptrs(k_in), _ptrs(dq_in), _ptrs(dk_in),
        _addr(rms_w), _addr(dw), eps, rope_theta, _addr(workspace), _nbytes(workspace),
        _stream(stream)), "ulysses_a2a_4d_qk_fused_backward")


def ulysses_a2a_4d_qkv_fused_backward(plan: Plan, dqkv_out, qkv_in, dq_in, dk_in, dv_in, rms_w,
                                      dw, eps: float, rope_theta: float, workspace, stream=None):
    """Backward of the interleaved QKV call into packed (b, s_q, 3, N, d) gradients."""
    _check(_lib().ulysses_a2a_4d_qkv_fused_backward(
        plan, _ptrs(dqkv_out), _ptrs(qkv_in), _ptrs(dq_in), _ptrs(dk_in), _ptrs(dv_in),
        _addr(rms_w), _addr(dw), eps, rope_theta, _addr(workspace), _nbytes(workspace),
        _stream(stream)), "ulysses_a2a_4d_qkv_fused_backward")


def ulysses_a2a_4d_packed_fused_backward(plan: Plan, planes: int, q_plane: int, k_plane: int,
                                         token_pitch: int, dpacked_out, packed_in, grads, rms_w,
                                         dw, eps: float, rope_theta: float, workspace,
                                         stream=None):
    """grads: one sequence of W gradient tensors per plane, flattened plane-major."""
    flat = [t for plane in grads for t in plane]
    _check(_lib().ulysses_a2a_4d_packed_fused_backward(
        plan, planes, q_plane, k_plane, token_pitch, _ptrs(dpacked_out), _ptrs(packed_in),
        _ptrs(flat), _addr(rms_w), _addr(dw), eps, rope_theta, _addr(workspace),
        _nbytes(workspace), _stream(stream)), "ulysses_a2a_4d_packed_fused_backward")


def ulysses_a2a_4d_qk_fused_backward_static(plan: Plan, dq_out, dk_out, q_in, k_in, dq_in, dk_in,
                                            rms_w, dw, eps: float, rope_theta: float, stream=None):
    """Backward of the fused call with the dw partial sums in the library's static scratch array
    (no workspace argument; the call allocates nothing). Calls that may run at the same time on
    one device race on that array."""
    _check(_lib().ulysses_a2a_4d_qk_fused_backward_static(
        plan, _ptrs(dq_out), _ptrs(dk_out), _ptrs(q_in), _ptrs(k_in), _ptrs(dq_in), _ptrs(dk_in),
        _addr(rms_w), _addr(dw), eps, rope_theta, _stream(stream)),
        "ulysses_a2a_4d_qk_fused_backward_static")


def ulysses_a2a_4d_host(plan: Plan, mode: int, host_in, host_out, dev_in, dev_out, stream=None):
    _check(_lib().ulysses_a2a_4d_host(plan, mode, _ptrs(host_in), _ptrs(host_out), _ptrs(dev_in),
                                      _ptrs(dev_out), _stream(stream)), "ulysses_a2a_4d_host")


def ulysses_a2a_4d_qk_fused_host(plan: Plan, q_host_in, k_host_in, q_host_out, k_host_out, q_in,
                                 k_in, q_out, k_out, rms_w, eps: float, rope_theta: float,
                                 stream=None):
    _check(_lib().ulysses_a2a_4d_qk_fused_host(
        plan, _ptrs(q_host_in), _ptrs(k_host_in), _ptrs(q_host_out), _ptrs(k_host_out), _ptrs(q_in),
        _ptrs(k_in), _ptrs(q_out), _ptrs(k_out), _addr(rms_w), eps, rope_theta, _stream(stream)),
        "ulysses_a2a_4d_qk_fused_host")


def ulysses_device_status() -> int:
    """Synchronise; return and clear the kernels' device status word (0 = no wait timed out)."""
    st = ctypes.c_uint()
    rc = _lib().ulysses_device_status(ctypes.byref(st))
    if rc not in (ULY_OK, ULY_EDEVICE):
        _check(rc, "ulysses_device_status")
    return st.value


def ulysses_selftest_wait_timeout(limit_us: int, stream=None):
    """Queue the failure-path self-test kernel (a wait that must time out after limit_us)."""
    _check(_lib().ulysses_selftest_wait_timeout(limit_us, _stream(stream)),
           "ulysses_selftest_wait_timeout")


def ulysses_strerror(status: int) -> str:
    return _lib().ulysses_strerror(status).decode()


def ulysses_version() -> int:
    return _lib().ulysses_version()
