"""The backward of the fused call with the library's static scratch array
(ulysses_a2a_4d_qk_fused_backward_static) against the workspace form
(ulysses_a2a_4d_qk_fused_backward): two calls in a row give the same bytes as the workspace
form, dw included, and device memory in use does not change across them. Named to run after the
other GPU test modules; it passes alone and after them."""
import numpy as np
import pytest
import torch

from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4

GEOMS = [
    (8, 1, [300] * 8, [5] * 8, 128),
    (5, 2, [100, 110, 90, 105, 95], [9, 8, 8, 8, 7], 128),
    (3, 2, [5, 0, 7], [3, 2, 1], 64),
    (1, 1, [4], [100], 256),
]


def _inputs(g, seed):
    W, b, seq, heads, d = g
    N, S = sum(heads), sum(seq)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    bf = lambda shape: torch.randn(shape, generator=gen).to(torch.bfloat16).cuda()  # noqa: E731
    q = [bf((b, s, N, d)) for s in seq]
    k = [bf((b, s, N, d)) for s in seq]
    dq = [bf((b, S, n, d)) for n in heads]
    dk = [bf((b, S, n, d)) for n in heads]
    return q, k, dq, dk, wl.rms_weights(d, seed=seed + 1).cuda()


@pytest.mark.parametrize("g", GEOMS, ids=[f"static{i}" for i in range(len(GEOMS))])
def test_static_scratch_matches_workspace_form(g):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    W, b, seq, heads, d = g
    q, k, dq, dk, w = _inputs(g, seed=sum(seq) + d)
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    need = B.ulysses_qk_fused_backward_workspace(plan)
    assert need <= B.ULYSSES_STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = ([torch.empty_like(x) for x in q], [torch.empty_like(x) for x in k],
           torch.empty((2, d), dtype=torch.float32, device="cuda"))
    B.ulysses_a2a_4d_qk_fused_backward(plan, ref[0], ref[1], q, k, dq, dk, w, ref[2], EPS, THETA, ws)
    torch.cuda.synchronize()

    # set-up: the first call on a device looks up the array (and the runtime may load the
    # library's device code holding it); the calls measured below come after it
    B.ulysses_a2a_4d_qk_fused_backward_static(plan, [torch.empty_like(x) for x in q],
                                              [torch.empty_like(x) for x in k],
                                              q, k, dq, dk, w, torch.empty_like(ref[2]), EPS, THETA)
    torch.cuda.synchronize()
    outs = []
    for call in range(2):  # two calls in a row, the second reusing the scratch the first left
        o = ([torch.full_like(x, float("nan")) for x in q], [torch.full_like(x, float("nan")) for x in k],
             torch.full((2, d), float("nan"), dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        B.ulysses_a2a_4d_qk_fused_backward_static(plan, o[0], o[1], q, k, dq, dk, w, o[2], EPS, THETA)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, f"call {call}: device memory changed"
        outs.append(o)
    for o in outs:
        for x, y in zip(o[0] + o[1], ref[0] + ref[1]):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        assert torch.equal(o[2].view(torch.int32), ref[2].view(torch.int32))
        assert np.isfinite(o[2].cpu().numpy()).all()
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def test_static_scratch_checks_arguments_like_the_workspace_form():
    g = (2, 1, [16, 16], [4, 4], 128)
    W, b, seq, heads, d = g
    q, k, dq, dk, w = _inputs(g, seed=5)
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    dqo = [torch.empty_like(x) for x in q]
    dko = [torch.empty_like(x) for x in k]
    dw = torch.empty((2, d), dtype=torch.float32, device="cuda")
    with pytest.raises(B.UlyssesError):  # dq output on top of the forward input
        B.ulysses_a2a_4d_qk_fused_backward_static(plan, q, dko, q, k, dq, dk, w, dw, EPS, THETA)
    with pytest.raises(B.UlyssesError):  # the fused path needs bf16 or fp16
        B.ulysses_a2a_4d_qk_fused_backward_static(B.ulysses_plan(*g, "float32"), dqo, dko, q, k,
                                                  dq, dk, w, dw, EPS, THETA)
    B.ulysses_a2a_4d_qk_fused_backward_static(plan, dqo, dko, q, k, dq, dk, w, dw, EPS, THETA)
    assert B.ulysses_device_status() == 0
