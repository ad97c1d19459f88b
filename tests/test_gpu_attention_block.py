"""A sequence-parallel self-attention block on W virtual ranks, forward and backward, against
the same block computed without sequence parallelism (the check the fast-ulysses 0.2.1 README
describes for its DiT attention example, "Quick start": sequence-parallel forward and backward
compared with the plain block).

Each rank holds a sequence shard of the input x (b, s_q, H). The block: the QKV projection of
the shard, packed (b, s_q, 3, N, d) as a fused projection writes it; q and k RMSNorm + RoPE
fused into the mode-0 relayout (the library's fused call, or its interleaved QKV form), v by
the plain mode-0 relayout; attention of rank r's n_r heads over the whole sequence; the mode-1
relayout back to sequence shards; the output projection. The reference computes the same block
on the unsharded input with every head, its norm and rotation written in plain PyTorch. Every
library call runs through the differentiable forms, so the gradients of x, of both projections
and of the two norm weights come back through the library's backward kernels.

The two computations differ only in rounding (bf16 at the library's inputs and outputs, the
order of the attention and projection sums), so they agree to about 1e-2 of the largest value;
a wrong head, position or rank mapping anywhere gives errors of order 1."""
import pytest
import torch
import torch.nn.functional as F

from ulysses_sequence_all_gb300 import autograd as A
from ulysses_sequence_all_gb300 import binding as B

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4
W, b, d = 4, 2, 64
SEQ = [70, 60, 0, 126]       # uneven sequence shards, one rank without tokens
HEADS = [3, 2, 2, 1]         # uneven head shares
N, S = sum(HEADS), sum(SEQ)
H = N * d
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def params(seed):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    x = torch.randn((b, S, H), generator=gen)
    wqkv = torch.randn((H, 3 * H), generator=gen) / H ** 0.5
    wo = torch.randn((H, H), generator=gen) / H ** 0.5
    rms_w = 1.0 + 0.1 * torch.randn((2, d), generator=gen)
    gy = torch.randn((b, S, H), generator=gen)
    return [t.cuda() for t in (x, wqkv, wo, rms_w, gy)]


def attention(q, k, v):
    """(b, S, n, d) bf16 each -> (b, S, n, d) bf16; softmax attention over the whole sequence."""
    o = F.scaled_dot_product_attention(q.float().transpose(1, 2), k.float().transpose(1, 2),
                                       v.float().transpose(1, 2))
    return o.transpose(1, 2).to(torch.bfloat16)


def norm_rope(x, w, pos):
    """RMSNorm over d, then adjacent-pair RoPE at positions `pos`, fp32, one rounding to bf16."""
    xf = x.float()
    y = xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + EPS) * w
    j = torch.arange(d // 2, dtype=torch.float64, device=x.device)
    ang = pos.double()[:, None] * THETA ** (-2.0 * j / d)
    c, s = torch.cos(ang).float()[None, :, None, :], torch.sin(ang).float()[None, :, None, :]
    e, o = y[..., 0::2], y[..., 1::2]
    return torch.stack((e * c - o * s, e * s + o * c), dim=-1).flatten(-2).to(torch.bfloat16)


def reference_block(x, wqkv, wo, rms_w):
    qkv = (x @ wqkv).to(torch.bfloat16).view(b, S, 3, N, d)
    pos = torch.arange(S, device=x.device)
    q = norm_rope(qkv[:, :, 0], rms_w[0], pos)
    k = norm_rope(qkv[:, :, 1], rms_w[1], pos)
    o = attention(q, k, qkv[:, :, 2])
    return o.reshape(b, S, H).float() @ wo


def parallel_block(x, wqkv, wo, rms_w, packed):
    plan = B.ulysses_plan(W, b, SEQ, HEADS, d, "bfloat16")
    offs = [sum(SEQ[:q]) for q in range(W)]
    # per rank: the projection of its sequence shard, packed (b, s_q, 3, N, d)
    qkv = [(x[:, o:o + s] @ wqkv).to(torch.bfloat16).view(b, s, 3, N, d).contiguous()
           for o, s in zip(offs, SEQ)]
    if packed:
        qh, kh, vh = A.qkv_fused(plan, qkv, rms_w, EPS, THETA)
    else:
        q = [t[:, :, 0].contiguous() for t in qkv]
        k = [t[:, :, 1].contiguous() for t in qkv]
        v = [t[:, :, 2].contiguous() for t in qkv]
        qh, kh = A.qk_fused(plan, q, k, rms_w, EPS, THETA)
        vh = A.a2a_4d(plan, v, 0)
    # rank r: its n_r heads over the whole sequence
    oh = [attention(qr, kr, vr) for qr, kr, vr in zip(qh, kh, vh)]
    os_ = A.a2a_4d(plan, oh, 1)  # back to sequence shards (b, s_q, N, d)
    y = [t.reshape(b, s, H).float() @ wo for t, s in zip(os_, SEQ)]
    return torch.cat(y, dim=1)


def rel_err(a, b_):
    return float((a - b_).abs().max() / b_.abs().max())


@pytest.mark.parametrize("packed", [False, True], ids=["qk_fused+v", "qkv_fused"])
def test_parallel_block_matches_plain_block(packed):
    x0, wqkv0, wo0, w0, gy = params(seed=41)
    leaves = {}
    outs = {}
    for name in ("ref", "sp"):
        x, wqkv, wo, rms_w = (t.clone().requires_grad_() for t in (x0, wqkv0, wo0, w0))
        y = (reference_block(x, wqkv, wo, rms_w) if name == "ref"
             else parallel_block(x, wqkv, wo, rms_w, packed))
        (y * gy).sum().backward()
        outs[name] = y.detach()
        leaves[name] = {"x": x.grad, "wqkv": wqkv.grad, "wo": wo.grad, "rms_w": rms_w.grad}
    assert rel_err(outs["sp"], outs["ref"]) < TOL
    for key in ("x", "wqkv", "wo", "rms_w"):
        err = rel_err(leaves["sp"][key], leaves["ref"][key])
        assert err < TOL, (key, err)
