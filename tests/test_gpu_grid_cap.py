"""A cap on the CTAs of each launch (ulysses_plan_set_max_ctas) changes no result: the relayout
and the fused forward give the same bytes, the backward the same dq and dk bytes and dw within
the summation bound (its partial sums are grouped by CTA)."""
import numpy as np
import pytest
import torch

from test_gpu_fused import EPS, THETA, make_inputs
from test_gpu_fused_bwd import check_dw, make_grads
from ulysses_sequence_all_gb300 import binding as B

pytestmark = pytest.mark.gpu

G = (5, 2, [100, 110, 90, 105, 95], [9, 8, 8, 8, 7], 128)
G_EQUAL = (5, 2, [100, 110, 90, 105, 95], [8] * 5, 128)  # row-block fused kernel, tensor relayout


def _plan(cap, g=G):
    plan = B.ulysses_plan(*g, "bfloat16")
    B.ulysses_plan_set_max_ctas(plan, cap)
    return plan


@pytest.mark.parametrize("engine", [B.ULY_ENGINE_TMA, B.ULY_ENGINE_VEC, B.ULY_ENGINE_TENSOR])
@pytest.mark.parametrize("cap", [1, 7, 152])
def test_relayout_capped_equals_uncapped(engine, cap):
    W, b, seq, heads, d = G
    q, _, _ = make_inputs(G, seed=3)
    outs = []
    for c in (0, cap):
        head = [torch.empty((b, sum(seq), n, d), dtype=torch.bfloat16, device="cuda") for n in heads]
        back = [torch.empty_like(x) for x in q]
        plan = _plan(c)
        B.ulysses_a2a_4d_engine(plan, 0, engine, q, head)
        B.ulysses_a2a_4d_engine(plan, 1, engine, head, back)
        torch.cuda.synchronize()
        outs.append(head + back)
    for x, y in zip(*outs):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert B.ulysses_device_status() == 0


@pytest.mark.parametrize("g", [G, G_EQUAL], ids=["uneven_heads", "equal_heads"])
@pytest.mark.parametrize("cap", [1, 9, 300])
def test_fused_and_backward_capped(cap, g):
    W, b, seq, heads, d = g
    q, k, w = make_inputs(g, seed=4)
    dq, dk = make_grads(g, seed=5)
    res = []
    for c in (0, cap):
        plan = _plan(c, g)
        qo = [torch.empty((b, sum(seq), n, d), dtype=torch.bfloat16, device="cuda") for n in heads]
        ko = [torch.empty_like(x) for x in qo]
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA)
        dqo = [torch.empty_like(x) for x in q]
        dko = [torch.empty_like(x) for x in k]
        dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8,
                         device="cuda")
        B.ulysses_a2a_4d_qk_fused_backward(plan, dqo, dko, q, k, dq, dk, w, dw, EPS, THETA, ws)
        torch.cuda.synchronize()
        res.append((qo + ko + dqo + dko, dw))
    for x, y in zip(res[0][0], res[1][0]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    check_dw(res[1][1].cpu().numpy(), res[0][1].cpu().numpy().astype(np.float64),
             b * sum(seq) * sum(heads), f"dw under cap {cap}")
    assert B.ulysses_device_status() == 0
