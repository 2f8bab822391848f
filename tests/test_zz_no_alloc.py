"""The allocation-free forward (h3attn_forward_noalloc).

It is for callers that may not allocate device memory -- code running inside
a host framework that owns all device memory in its own pool, or a loop where
a cudaMalloc would stall the device -- and so cannot create a plan.  It runs
the same kernel as h3attn_forward with its work list and error word in a
static device array shared by all calls.

The first test calls it twice in a row through the C ABI (a larger layout,
then a smaller one, so stale contents of the shared array would show) and
compares each output with the fp64 oracle and with the plan-based
h3attn_forward on the same inputs, within the parity tolerance of the other
tests.  The two CUDA paths are not byte-identical: a plan splits the last
round of work units along the keys and merges the pieces (that needs the
plan's partial buffers), while the allocation-free path always runs whole
units, so the two sum the same terms in a different order.

The second test has two host threads share one stream, each calling the
entry point several times with its own layout; every output must be
byte-identical to a single-threaded call on the same layout, and guard rows
around each output must stay untouched (a kernel that read the other
thread's work list would write the wrong rows).

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import threading

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch, torch_bf16_to_f64
from tests.gpu_cases import check_attention, docs_1d, random_tensors

SCALE = 1.0 / np.sqrt(128.0)


def _inputs(lengths, num_heads, seed):
    S = sum(lengths)
    W = num_heads * 128
    t = random_tensors(S, num_heads, seed)
    q = bf16_to_torch(t.q).view(S, W)
    k = bf16_to_torch(t.k).view(S, W)
    v = bf16_to_torch(t.v).view(S, W)
    return S, W, q, k, v


def _plan_forward(lengths, num_heads, q, k, v):
    S, W = q.shape
    o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((num_heads, S), float("nan"), dtype=torch.float32, device="cuda")
    with H.Plan(docs_1d(lengths), num_heads) as p:
        H.h3attn_forward(p.handle, q, k, v, o, SCALE, lse)
        H.h3attn_get_device_error(p.handle)
    return o, lse


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


@pytest.mark.gpu
def test_noalloc_forward_matches_oracle_and_plan_forward_on_two_calls(lib):
    cases = [([700, 1, 129, 2048, 300], 5, 31),   # first call: more work units
             ([257, 64, 1000], 3, 32)]             # second call: fewer, different layout
    for lengths, num_heads, seed in cases:
        S, W, q, k, v = _inputs(lengths, num_heads, seed)
        o_ref, lse_ref = _plan_forward(lengths, num_heads, q, k, v)
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((num_heads, S), float("nan"), dtype=torch.float32, device="cuda")
        H.h3attn_forward_noalloc(_cu(lengths), num_heads, q, k, v, o, SCALE, lse)
        torch.cuda.synchronize()
        o_got = torch_bf16_to_f64(o).reshape(S, num_heads, 128)
        # against the fp64 oracle on the same bf16 q, k, v
        f64 = lambda x: torch_bf16_to_f64(x).reshape(S, num_heads, 128)
        o_or, lse_or = oatt.attention_rows(f64(q), f64(k), f64(v), _cu(lengths), SCALE, range(num_heads),
                                           np.arange(S))
        check_attention(o_got, o_or, lse.cpu().numpy(), lse_or, f"noalloc vs oracle, layout {lengths}")
        # against the plan-based forward (same kernel, different key order in the split last wave)
        check_attention(o_got, torch_bf16_to_f64(o_ref).reshape(S, num_heads, 128), lse.cpu().numpy(),
                        lse_ref.cpu().numpy(), f"noalloc vs plan forward, layout {lengths}")


@pytest.mark.gpu
def test_noalloc_two_host_threads_on_one_stream(lib):
    layouts = [([700, 129, 2048], 3, 41), ([257, 64, 1000, 5], 2, 42)]
    guard = 64
    stream = torch.cuda.Stream()
    jobs = []
    for lengths, num_heads, seed in layouts:
        S, W, q, k, v = _inputs(lengths, num_heads, seed)
        expect = torch.empty(S, W, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()  # inputs were made on the default stream
        H.h3attn_forward_noalloc(_cu(lengths), num_heads, q, k, v, expect, SCALE, stream=stream)
        stream.synchronize()
        # several outputs per thread, each inside guard rows of a known bit pattern
        outs = []
        for _ in range(4):
            buf = torch.full((S + 2 * guard, W), 0, dtype=torch.int16, device="cuda")
            buf.fill_(0x7FC1)  # a NaN pattern the kernel never writes
            outs.append(buf)
        jobs.append(dict(lengths=lengths, heads=num_heads, q=q, k=k, v=v, S=S, expect=expect, outs=outs))
    torch.cuda.synchronize()

    errors = []

    def worker(job):
        try:
            for rep in range(3):
                for buf in job["outs"]:
                    o = buf.view(torch.bfloat16)[guard:guard + job["S"]]
                    H.h3attn_forward_noalloc(_cu(job["lengths"]), job["heads"], job["q"], job["k"], job["v"],
                                             o, SCALE, stream=stream)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    stream.synchronize()
    assert not errors, errors
    for job in jobs:
        want = job["expect"].view(torch.int16).cpu().numpy()
        for buf in job["outs"]:
            got = buf.cpu().numpy()
            assert np.all(got[:guard] == 0x7FC1) and np.all(got[guard + job["S"]:] == 0x7FC1), \
                f"guard rows written, layout {job['lengths']}"
            assert np.array_equal(got[guard:guard + job["S"]], want), \
                f"output differs from a single-threaded call, layout {job['lengths']}"


@pytest.mark.gpu
def test_noalloc_rejects_layouts_beyond_its_limit(lib):
    # 32768 work units at most: 129 documents of 256 rows x 255 heads needs 32895
    S, W = 8, 255 * 128
    x = torch.zeros(S, W, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(x)
    cu = np.arange(0, 129 * 256 + 1, 256, dtype=np.int32)
    with pytest.raises(H.H3AttnError) as e:
        H.h3attn_forward_noalloc(cu, 255, x, x, x, o, 0.1)
    assert e.value.status == H.H3ATTN_EINVAL
    assert "at most 32768" in str(e.value)
