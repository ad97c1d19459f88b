"""The library's calls inside a CUDA graph: after one ordinary call (the first-call set-up: device
attributes, kernel attributes), the exchange step (fused q,k mode 0, v mode 0, attention output
mode 1) and the fused backward are captured on a side stream and replayed; each replay, with new
contents in the same input buffers, gives the bytes the direct calls give."""
import pytest
import torch

from test_gpu_fused import EPS, THETA
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

G = (8, 1, [300] * 8, [5] * 8, 128)


def _buffers(g):
    W, b, seq, heads, d = g
    S, N = sum(seq), sum(heads)
    seq_side = lambda: [torch.empty((b, s, N, d), dtype=torch.bfloat16, device="cuda") for s in seq]  # noqa: E731
    head_side = lambda: [torch.empty((b, S, n, d), dtype=torch.bfloat16, device="cuda") for n in heads]  # noqa: E731
    return {"q": seq_side(), "k": seq_side(), "v": seq_side(), "o": head_side(),
            "qo": head_side(), "ko": head_side(), "vo": head_side(), "oo": seq_side(),
            "dq": seq_side(), "dk": seq_side()}


def _fill(bufs, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    for name in ("q", "k", "v", "o"):
        for t in bufs[name]:
            t.copy_(torch.randn(t.shape, generator=gen, device="cuda").to(torch.bfloat16))


def _calls(plan, bufs, w, dw, ws, stream):
    B.ulysses_a2a_4d_qk_fused(plan, bufs["q"], bufs["k"], bufs["qo"], bufs["ko"], w, EPS, THETA, stream)
    B.ulysses_a2a_4d(plan, 0, bufs["v"], bufs["vo"], stream)
    B.ulysses_a2a_4d(plan, 1, bufs["o"], bufs["oo"], stream)
    B.ulysses_a2a_4d_qk_fused_backward(plan, bufs["dq"], bufs["dk"], bufs["q"], bufs["k"],
                                       bufs["qo"], bufs["ko"], w, dw, EPS, THETA, ws, stream)


def test_step_and_backward_replay_in_a_graph():
    assert torch.cuda.is_available()
    plan = B.ulysses_plan(*G, "bfloat16")
    w = wl.rms_weights(G[4], seed=3).cuda()
    ws = torch.empty(B.ulysses_qk_fused_backward_workspace(plan), dtype=torch.uint8, device="cuda")
    graph_bufs, direct_bufs = _buffers(G), _buffers(G)
    dw_graph = torch.empty((2, G[4]), dtype=torch.float32, device="cuda")
    dw_direct = torch.empty_like(dw_graph)
    side = torch.cuda.Stream()
    _fill(graph_bufs, 0)
    _calls(plan, graph_bufs, w, dw_graph, ws, side)  # first-call set-up outside the capture
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        _calls(plan, graph_bufs, w, dw_graph, ws, torch.cuda.current_stream())
    ws_direct = torch.empty_like(ws)
    for seed in (11, 12):
        _fill(graph_bufs, seed)
        _fill(direct_bufs, seed)
        graph.replay()
        _calls(plan, direct_bufs, w, dw_direct, ws_direct, torch.cuda.current_stream())
        torch.cuda.synchronize()
        for name in ("qo", "ko", "vo", "oo", "dq", "dk"):
            for a, c in zip(graph_bufs[name], direct_bufs[name]):
                assert torch.equal(a.view(torch.int16), c.view(torch.int16)), name
        assert torch.equal(dw_graph.view(torch.int32), dw_direct.view(torch.int32))
    assert B.ulysses_device_status() == 0
