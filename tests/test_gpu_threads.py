"""Several host threads calling the library at once, each on its own CUDA stream with its own plan
and buffers: the device relayout, the fused call and the host-buffer call. ctypes releases the
GIL during the foreign calls, so the calls (first-use set-up included) really overlap on the host.
Every thread's results must equal those of the same calls made one after another."""
import threading

import pytest
import torch

from gpu_util import random_bytes_tensor
from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS, THETA = 1e-6, 1e4
THREADS = 4


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.library()
    yield
    assert B.ulysses_device_status() == 0, "a kernel recorded a wait timeout"


def make_case(i):
    """Thread i's geometry and inputs (different splits per thread)."""
    W, b, d = 3, 1, 128
    seq = [200 + 17 * i, 150, 311 - 9 * i]
    # odd threads: equal head groups (the tensor-map relayout and the row-block fused kernel)
    heads = [2, 2, 2] if i % 2 else [2 + (i % 4 == 2), 3, 1]
    N, S = sum(heads), sum(seq)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(500 + i)
    q = [torch.randn((b, s, N, d), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    k = [torch.randn((b, s, N, d), generator=gen).to(torch.bfloat16).cuda() for s in seq]
    raw = [random_bytes_tensor((b, s, N, d), torch.bfloat16, gen, "cpu") for s in seq]
    w = wl.rms_weights(d, seed=7 + i).cuda()
    return (W, b, seq, heads, d), q, k, raw, w


def run_case(case, stream):
    """The three calls on `stream`; returns every output as CPU tensors."""
    (W, b, seq, heads, d), q, k, raw, w = case
    N, S = sum(heads), sum(seq)
    plan = B.ulysses_plan(W, b, seq, heads, d, "bfloat16")
    head = [(b, S, n, d) for n in heads]
    with torch.cuda.stream(stream):
        rel = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in head]
        qo = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in head]
        ko = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in head]
        dev_in = [torch.empty(x.shape, dtype=torch.bfloat16, device="cuda") for x in raw]
        dev_out = [torch.empty(sh, dtype=torch.bfloat16, device="cuda") for sh in head]
    host_in = [x.pin_memory() for x in raw]
    host_out = [torch.zeros(sh, dtype=torch.bfloat16).pin_memory() for sh in head]
    outs = []
    for _ in range(3):
        B.ulysses_a2a_4d(plan, 0, q, rel, stream)
        B.ulysses_a2a_4d_qk_fused(plan, q, k, qo, ko, w, EPS, THETA, stream)
        B.ulysses_a2a_4d_host(plan, 0, host_in, host_out, dev_in, dev_out, stream)
        stream.synchronize()
        outs.append([t.cpu() for t in rel + qo + ko] + [t.clone() for t in host_out])
    return outs


def test_concurrent_host_threads_match_serial_calls():
    cases = [make_case(i) for i in range(THREADS)]
    torch.cuda.synchronize()
    serial = [run_case(c, torch.cuda.Stream()) for c in cases]
    results, errors = [None] * THREADS, []

    def worker(i):
        try:
            results[i] = run_case(cases[i], torch.cuda.Stream())
        except Exception as exc:  # reported below, with the thread's index
            errors.append((i, repr(exc)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    for i in range(THREADS):
        for rep in range(3):
            for got, want in zip(results[i][rep], serial[i][0]):
                assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (i, rep)
