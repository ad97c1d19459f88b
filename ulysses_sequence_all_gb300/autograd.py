"""Differentiable forms of the library calls for PyTorch callers.

The pages' collective is differentiable and its backward uses the plan saved by its forward
(fast-ulysses 0.2.1, README, "Quick start" and "Limits"; FastVideo, "Ulysses performance on
GB200"). Here each call is a ``torch.autograd.Function`` over the C entry points, keeping the
plan for the backward:

* ``a2a_4d(plan, xs, mode)``: the relayout; its backward is the relayout in the other mode on
  the same plan (the relayout is a permutation, so its adjoint is its inverse).
* ``qk_fused(plan, q, k, rms_w, eps, rope_theta)``: the fused mode-0 call; its backward is
  ``ulysses_a2a_4d_qk_fused_backward`` (dq, dk and the gradient of ``rms_w``), with a workspace
  allocated by torch.
* ``qkv_fused(plan, qkv, rms_w, eps, rope_theta)``: the interleaved packed-QKV call; its backward
  is ``ulysses_a2a_4d_qkv_fused_backward`` (packed dqkv and the gradient of ``rms_w``).
* ``packed_fused(plan, packed, planes, q_plane, k_plane, rms_w, eps, rope_theta)``: the call on
  any packing of C planes per token (QKVG, ...); its backward is
  ``ulysses_a2a_4d_packed_fused_backward``; a token's columns beyond its planes get zero gradient.

Inputs and outputs are lists of W tensors (one per virtual rank) on the current CUDA device;
the outputs are new tensors the caller owns. Nothing here computes: every step runs in the
library's kernels, on the current stream.
"""
from __future__ import annotations

import torch

from . import binding as B


def _shapes(plan: B.Plan, mode: int):
    """Output shapes of a call in `mode`: rank r's (b, S, n_r, d) for mode 0, rank q's
    (b, s_q, N, d) for mode 1."""
    S, N = sum(plan.seq_splits), sum(plan.head_splits)
    if mode == 0:
        return [(plan.b, S, n, plan.d) for n in plan.head_splits]
    return [(plan.b, s, N, plan.d) for s in plan.seq_splits]


def _empty(plan: B.Plan, mode: int, like: torch.Tensor):
    return [torch.empty(sh, dtype=like.dtype, device=like.device) for sh in _shapes(plan, mode)]


def _grads(grads, plan: B.Plan, mode: int, like: torch.Tensor):
    """Contiguous gradients of a call's outputs (mode: the call's), zeros where autograd passes
    None; `like` gives dtype and device."""
    out = []
    for g, sh in zip(grads, _shapes(plan, mode)):
        if g is None:
            g = torch.zeros(sh, dtype=like.dtype, device=like.device)
        out.append(g.contiguous())
    return out


class _A2A4D(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, mode, *xs):
        xs = [x.contiguous() for x in xs]
        outs = _empty(plan, mode, xs[0])
        B.ulysses_a2a_4d(plan, mode, xs, outs)
        ctx.plan, ctx.mode = plan, mode
        ctx.like = torch.empty(0, dtype=xs[0].dtype, device=xs[0].device)
        return tuple(outs)

    @staticmethod
    def backward(ctx, *grads):
        plan, mode = ctx.plan, ctx.mode
        gs = _grads(grads, plan, mode, ctx.like)
        back = _empty(plan, 1 - mode, gs[0])
        B.ulysses_a2a_4d(plan, 1 - mode, gs, back)
        return (None, None, *back)


def a2a_4d(plan: B.Plan, xs, mode: int = 0):
    """The relayout of W tensors, differentiable (backward: the other mode, same plan)."""
    if mode not in (0, 1):
        raise ValueError("mode must be 0 or 1")
    return list(_A2A4D.apply(plan, mode, *xs))


class _QKFused(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, eps, rope_theta, rms_w, *qk):
        W = len(qk) // 2
        q = [x.contiguous() for x in qk[:W]]
        k = [x.contiguous() for x in qk[W:]]
        rms_w = rms_w.contiguous()
        qo, ko = _empty(plan, 0, q[0]), _empty(plan, 0, q[0])
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, rms_w, eps, rope_theta)
        ctx.plan, ctx.eps, ctx.theta, ctx.W = plan, eps, rope_theta, W
        ctx.save_for_backward(rms_w, *q, *k)
        return tuple(qo + ko)

    @staticmethod
    def backward(ctx, *grads):
        plan, W = ctx.plan, ctx.W
        rms_w, *qk = ctx.saved_tensors
        q, k = qk[:W], qk[W:]
        like = q[0]
        gq = _grads(grads[:W], plan, 0, like)
        gk = _grads(grads[W:], plan, 0, like)
        dq, dk = _empty(plan, 1, like), _empty(plan, 1, like)
        dw = torch.empty_like(rms_w, dtype=torch.float32)
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device=like.device)
        B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, rms_w, dw, ctx.eps,
                                           ctx.theta, ws)
        return (None, None, None, dw, *dq, *dk)


class _QKVFused(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, eps, rope_theta, rms_w, *qkv):
        qkv = [x.contiguous() for x in qkv]
        rms_w = rms_w.contiguous()
        like = qkv[0]
        qo, ko, vo = _empty(plan, 0, like), _empty(plan, 0, like), _empty(plan, 0, like)
        B.ulysses_a2a_4d_qkv_fused(plan, qkv, qo, ko, vo, rms_w, eps, rope_theta)
        ctx.plan, ctx.eps, ctx.theta, ctx.W = plan, eps, rope_theta, len(qkv)
        ctx.save_for_backward(rms_w, *qkv)
        return tuple(qo + ko + vo)

    @staticmethod
    def backward(ctx, *grads):
        plan, W = ctx.plan, ctx.W
        rms_w, *qkv = ctx.saved_tensors
        like = qkv[0]
        gq = _grads(grads[:W], plan, 0, like)
        gk = _grads(grads[W:2 * W], plan, 0, like)
        gv = _grads(grads[2 * W:], plan, 0, like)
        dqkv = [torch.empty_like(x) for x in qkv]
        dw = torch.empty_like(rms_w, dtype=torch.float32)
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device=like.device)
        B.ulysses_a2a_4d_qkv_fused_backward(plan, dqkv, qkv, gq, gk, gv, rms_w, dw, ctx.eps,
                                            ctx.theta, ws)
        return (None, None, None, dw, *dqkv)


def qkv_fused(plan: B.Plan, qkv, rms_w: torch.Tensor, eps: float, rope_theta: float):
    """The interleaved call on packed (b, s_q, 3, N, d) inputs, differentiable in qkv and rms_w.
    Returns (q_out, k_out, v_out), lists of W tensors."""
    out = _QKVFused.apply(plan, eps, rope_theta, rms_w, *qkv)
    W = len(qkv)
    return list(out[:W]), list(out[W:2 * W]), list(out[2 * W:])


def qk_fused(plan: B.Plan, q, k, rms_w: torch.Tensor, eps: float, rope_theta: float):
    """The fused mode-0 call (QK RMSNorm + RoPE in the scatter), differentiable in q, k and
    rms_w ((2, d) fp32). Returns (q_out, k_out), lists of W tensors."""
    out = _QKFused.apply(plan, eps, rope_theta, rms_w, *q, *k)
    W = len(q)
    return list(out[:W]), list(out[W:])


class _PackedFused(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, planes, q_plane, k_plane, eps, rope_theta, rms_w, *packed):
        packed = [x.contiguous() for x in packed]
        rms_w = rms_w.contiguous()
        like = packed[0]
        pitch = like[0, 0].numel() * like.element_size() if like.dim() > 2 else like.element_size()
        outs = [_empty(plan, 0, like) for _ in range(planes)]
        B.ulysses_a2a_4d_packed_fused(plan, planes, q_plane, k_plane, pitch, packed, outs, rms_w,
                                      eps, rope_theta)
        ctx.plan, ctx.eps, ctx.theta, ctx.W = plan, eps, rope_theta, len(packed)
        ctx.planes, ctx.q_plane, ctx.k_plane, ctx.pitch = planes, q_plane, k_plane, pitch
        ctx.save_for_backward(rms_w, *packed)
        return tuple(t for plane in outs for t in plane)

    @staticmethod
    def backward(ctx, *grads):
        plan, W = ctx.plan, ctx.W
        rms_w, *packed = ctx.saved_tensors
        like = packed[0]
        gs = [_grads(grads[c * W:(c + 1) * W], plan, 0, like) for c in range(ctx.planes)]
        dpacked = [torch.zeros_like(x) for x in packed]  # columns beyond the planes: zero
        dw = torch.empty_like(rms_w, dtype=torch.float32)
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device=like.device)
        B.ulysses_a2a_4d_packed_fused_backward(plan, ctx.planes, ctx.q_plane, ctx.k_plane,
                                               ctx.pitch, dpacked, packed, gs, rms_w, dw, ctx.eps,
                                               ctx.theta, ws)
        return (None, None, None, None, None, None, dw, *dpacked)


def packed_fused(plan: B.Plan, packed, planes: int, q_plane: int, k_plane: int,
                 rms_w: torch.Tensor, eps: float, rope_theta: float):
    """The fused call on packed inputs (rank q's tensor: (b, s_q, ...) with `planes` planes of
    N * d elements at the start of each token, the token pitch being the product of the trailing
    dimensions), differentiable in packed and rms_w. Returns one list of W tensors per plane."""
    out = _PackedFused.apply(plan, planes, q_plane, k_plane, eps, rope_theta, rms_w, *packed)
    W = len(packed)
    return [list(out[c * W:(c + 1) * W]) for c in range(planes)]
