"""The allocation-free forward (h3attn_forward_noalloc).

It is for callers that may not allocate device memory -- code running inside
a host framework that owns all device memory in its own pool, or a loop where
a cudaMalloc would stall the device -- and so cannot create a plan.  It runs
the same kernel as h3attn_forward with its work list and error word in a
static device array shared by all calls.  The test calls it twice in a row
through the C ABI (a larger layout, then a smaller one, so stale contents of
the shared array would show) and compares each output with the plan-based
h3attn_forward on the same inputs, within the parity tolerance of the other
tests.  This file sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch, torch_bf16_to_f64
from tests.gpu_cases import check_attention, docs_1d, random_tensors


def _inputs(lengths, num_heads, seed):
    S = sum(lengths)
    W = num_heads * 128
    t = random_tensors(S, num_heads, seed)
    q = bf16_to_torch(t.q).view(S, W)
    k = bf16_to_torch(t.k).view(S, W)
    v = bf16_to_torch(t.v).view(S, W)
    return S, W, q, k, v


def _plan_forward(lengths, num_heads, q, k, v, scale):
    S, W = q.shape
    o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((num_heads, S), float("nan"), dtype=torch.float32, device="cuda")
    with H.Plan(docs_1d(lengths), num_heads) as p:
        H.h3attn_forward(p.handle, q, k, v, o, scale, lse)
        H.h3attn_get_device_error(p.handle)
    return o, lse


@pytest.mark.gpu
def test_noalloc_forward_matches_plan_forward_on_two_calls(lib):
    scale = 1.0 / np.sqrt(128.0)
    cases = [([700, 1, 129, 2048, 300], 5, 31),   # first call: more work units
             ([257, 64, 1000], 3, 32)]             # second call: fewer, different layout
    for lengths, num_heads, seed in cases:
        S, W, q, k, v = _inputs(lengths, num_heads, seed)
        o_ref, lse_ref = _plan_forward(lengths, num_heads, q, k, v, scale)
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((num_heads, S), float("nan"), dtype=torch.float32, device="cuda")
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        H.h3attn_forward_noalloc(cu, num_heads, q, k, v, o, scale, lse)
        torch.cuda.synchronize()
        check_attention(torch_bf16_to_f64(o), torch_bf16_to_f64(o_ref), lse.cpu().numpy(),
                        lse_ref.cpu().numpy(), f"noalloc vs plan forward, layout {lengths}")


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
