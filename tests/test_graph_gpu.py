"""One plan serving every attention block of a denoising step, captured once
as a CUDA graph and replayed: the per-request loop of the DiT (the plan is
built once per request; each of the 50 blocks runs prologue + forward on its
own q/k/v).  The graph replay must give byte-identical outputs to eager
calls, and the plan's work list and tables must survive the replays."""
import numpy as np
import pytest
import torch

from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch
from tests.gpu_cases import docs_1d, random_tensors

pytestmark = pytest.mark.gpu

N_BLOCKS = 50


def _block_inputs(S, Hh, n_blocks):
    dev = torch.device("cuda")
    blocks = []
    for b in range(n_blocks):
        t = random_tensors(S, Hh, seed=500 + b)
        W = Hh * 128
        blocks.append(dict(
            q=bf16_to_torch(t.q).view(S, W), k=bf16_to_torch(t.k).view(S, W),
            v=bf16_to_torch(t.v).view(S, W),
            gq=torch.from_numpy(t.gain_q).to(dev), gk=torch.from_numpy(t.gain_k).to(dev),
            qh=torch.empty(S, W, dtype=torch.bfloat16, device=dev),
            kh=torch.empty(S, W, dtype=torch.bfloat16, device=dev),
            o=torch.zeros(S, W, dtype=torch.bfloat16, device=dev),
            lse=torch.zeros(Hh, S, dtype=torch.float32, device=dev)))
    return blocks


def _run_blocks(plan, blocks, stream):
    scale = 1.0 / np.sqrt(128.0)
    for b in blocks:
        H.h3attn_qk_prologue(plan.handle, b["q"], b["k"], b["qh"], b["kh"], b["gq"], b["gk"], 1e-6,
                             stream=stream)
        H.h3attn_forward(plan.handle, b["qh"], b["kh"], b["v"], b["o"], scale, b["lse"], stream=stream)


def test_fifty_blocks_one_plan_cuda_graph(lib):
    lens = [700, 131, 1200]  # a split last wave is not needed here; ragged tails are
    Hh = 3
    S = sum(lens)
    blocks = _block_inputs(S, Hh, N_BLOCKS)
    side = torch.cuda.Stream()
    with H.Plan(docs_1d(lens), Hh, stream=side) as plan:
        with torch.cuda.stream(side):
            _run_blocks(plan, blocks, side)
        side.synchronize()
        H.h3attn_get_device_error(plan.handle, stream=side)
        eager = [(b["o"].view(torch.int16).cpu().numpy().copy(), b["lse"].cpu().numpy().copy()) for b in blocks]
        for b in blocks:
            b["o"].zero_()
            b["lse"].zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            _run_blocks(plan, blocks, side)
        for rep in range(2):
            graph.replay()
            torch.cuda.synchronize()
            H.h3attn_get_device_error(plan.handle)
            for b, (o_e, lse_e) in zip(blocks, eager):
                assert np.array_equal(b["o"].view(torch.int16).cpu().numpy(), o_e), f"replay {rep}: o differs"
                assert np.array_equal(b["lse"].cpu().numpy(), lse_e), f"replay {rep}: lse differs"
