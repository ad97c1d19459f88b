"""The differentiable forms (ulysses_sequence_all_gb300.autograd): gradients through the relayout
are the other mode on the same plan, bit for bit, and through the fused call they are the
library's fused backward (dq, dk, dw), checked against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import host_raw
from test_gpu_fused import EPS, THETA, make_inputs
from test_gpu_fused_bwd import check_dw, check_dx, make_grads
from ulysses_sequence_all_gb300 import autograd as A
from ulysses_sequence_all_gb300 import binding as B

pytestmark = pytest.mark.gpu

G = (5, 2, [30, 31, 0, 30, 29], [9, 8, 8, 8, 7], 128)


@pytest.mark.parametrize("mode", [0, 1])
def test_relayout_gradient_is_the_other_mode(oracle, mode):
    W, b, seq, heads, d = G
    plan = B.ulysses_plan(*G, "bfloat16")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(3 + mode)
    S, N = sum(seq), sum(heads)
    in_shapes = [(b, s, N, d) for s in seq] if mode == 0 else [(b, S, n, d) for n in heads]
    out_shapes = [(b, S, n, d) for n in heads] if mode == 0 else [(b, s, N, d) for s in seq]
    xs = [torch.randn(sh, generator=gen).to(torch.bfloat16).cuda().requires_grad_() for sh in in_shapes]
    gs = [torch.randn(sh, generator=gen).to(torch.bfloat16).cuda() for sh in out_shapes]
    outs = A.a2a_4d(plan, xs, mode)
    torch.autograd.backward(outs, gs)
    want = oracle.a2a_4d([host_raw(g) for g in gs], seq, heads, 1 - mode)
    for x, w in zip(xs, want):
        assert np.array_equal(host_raw(x.grad), w)
    fwd = oracle.a2a_4d([host_raw(x.detach()) for x in xs], seq, heads, mode)
    for o, w in zip(outs, fwd):
        assert np.array_equal(host_raw(o.detach()), w)


def test_round_trip_gradient_is_identity():
    W, b, seq, heads, d = G
    plan = B.ulysses_plan(*G, "bfloat16")
    q, _, _ = make_inputs(G, seed=8)
    xs = [x.clone().requires_grad_() for x in q]
    back = A.a2a_4d(plan, A.a2a_4d(plan, xs, 0), 1)
    gs = [torch.randn_like(x) for x in back]
    torch.autograd.backward(back, gs)
    for x, g, y in zip(xs, gs, back):
        assert torch.equal(y.detach().view(torch.int16), x.detach().view(torch.int16))
        assert torch.equal(x.grad.view(torch.int16), g.view(torch.int16))


def test_fused_gradients_match_the_backward_call(oracle):
    W, b, seq, heads, d = G
    plan = B.ulysses_plan(*G, "bfloat16")
    q, k, w = make_inputs(G, seed=9)
    gq, gk = make_grads(G, seed=10)
    qr = [x.clone().requires_grad_() for x in q]
    kr = [x.clone().requires_grad_() for x in k]
    wr = w.clone().requires_grad_()
    qo, ko = A.qk_fused(plan, qr, kr, wr, EPS, THETA)
    torch.autograd.backward(qo + ko, gq + gk)
    # the direct calls on the same inputs
    ref_qo = [torch.empty_like(x) for x in gq]
    ref_ko = [torch.empty_like(x) for x in gk]
    B.ulysses_a2a_4d_qk_fused(plan, q, k, ref_qo, ref_ko, w, EPS, THETA)
    dq = [torch.empty_like(x) for x in q]
    dk = [torch.empty_like(x) for x in k]
    dw = torch.empty_like(w)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qk_fused_backward(plan, dq, dk, q, k, gq, gk, w, dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    for a, c in zip(qo + ko + [x.grad for x in qr + kr], ref_qo + ref_ko + dq + dk):
        assert torch.equal(a.detach().view(torch.int16), c.view(torch.int16))
    assert torch.equal(wr.grad.view(torch.int32), dw.view(torch.int32))
    # and against the oracle
    wn = w.cpu().numpy().astype(np.float64)
    n_rows = b * sum(seq) * sum(heads)
    for t, (x, g, got) in enumerate(((q, gq, qr), (k, gk, kr))):
        ref_dx, ref_dw = oracle.qk_fused_bwd([host_raw(v) for v in x], [host_raw(v) for v in g],
                                             seq, heads, wn[t], EPS, THETA)
        for r in range(W):
            check_dx(oracle, host_raw(got[r].grad), ref_dx[r], f"autograd t{t} r{r}")
        check_dw(wr.grad[t].cpu().numpy(), ref_dw, n_rows, f"autograd dw {t}")
    assert B.ulysses_device_status() == 0


def test_qkv_gradients_match_the_backward_call():
    W, b, seq, heads, d = G
    plan = B.ulysses_plan(*G, "bfloat16")
    q, k, w = make_inputs(G, seed=19)
    v, _, _ = make_inputs(G, seed=20)
    qkv = [torch.stack([a, c, e], dim=2) for a, c, e in zip(q, k, v)]
    gq, gk = make_grads(G, seed=21)
    gv, _ = make_grads(G, seed=22)
    xr = [x.clone().requires_grad_() for x in qkv]
    wr = w.clone().requires_grad_()
    qo, ko, vo = A.qkv_fused(plan, xr, wr, EPS, THETA)
    torch.autograd.backward(qo + ko + vo, gq + gk + gv)
    dqkv = [torch.empty_like(x) for x in qkv]
    dw = torch.empty_like(w)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_qkv_fused_backward(plan, dqkv, qkv, gq, gk, gv, w, dw, EPS, THETA, ws)
    torch.cuda.synchronize()
    for x, ref in zip(xr, dqkv):
        assert torch.equal(x.grad.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(wr.grad.view(torch.int32), dw.view(torch.int32))



def test_packed_gradients_match_the_backward_call():
    """QKVG packed with extra columns per token (q plane 2, k plane 0): autograd's gradients equal
    the direct backward call's bytes, and the extra columns get exactly zero gradient."""
    W, b, seq, heads, d = G
    N, S = sum(heads), sum(seq)
    planes, extra = 4, 16
    pitch = planes * N * d + extra
    gen = torch.Generator(device="cpu")
    gen.manual_seed(23)
    packed = [torch.randn((b, s, pitch), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    grads = [[torch.randn((b, S, n, d), generator=gen).to(torch.bfloat16).cuda() for n in heads]
             for _ in range(planes)]
    w = make_inputs(G, seed=24)[2]
    plan = B.ulysses_plan(*G, "bfloat16")
    xr = [x.clone().requires_grad_() for x in packed]
    wr = w.clone().requires_grad_()
    outs = A.packed_fused(plan, xr, planes, 2, 0, wr, EPS, THETA)
    torch.autograd.backward([t for plane in outs for t in plane],
                            [t for plane in grads for t in plane])
    dpk = [torch.zeros_like(x) for x in packed]
    dw = torch.empty_like(w)
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    B.ulysses_a2a_4d_packed_fused_backward(plan, planes, 2, 0, pitch * 2, dpk, packed, grads, w, dw,
                                           EPS, THETA, ws)
    torch.cuda.synchronize()
    for x, ref in zip(xr, dpk):
        assert torch.equal(x.grad.view(torch.int16), ref.view(torch.int16))
        assert int(torch.count_nonzero(x.grad[:, :, planes * N * d:].float())) == 0
    assert torch.equal(wr.grad.view(torch.int32), dw.view(torch.int32))
