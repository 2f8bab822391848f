"""The FP8 (e4m3) variant: quantisation bit-exact against the oracle's fp32
quantisers (codes and scales), and -- once the FP8 forward exists -- its
output against exact attention on the dequantised values within the bound of
its P rounding."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as ofp8
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch
from tests.gpu_cases import docs_1d, random_tensors

pytestmark = pytest.mark.gpu


def fp8_buffers(S, Hh):
    dev = torch.device("cuda")
    s_pad = (S + 15) // 16 * 16
    return dict(q8=torch.empty(S, Hh * 128, dtype=torch.uint8, device=dev),
                k8=torch.empty(S, Hh * 128, dtype=torch.uint8, device=dev),
                v8t=torch.empty(Hh, 128, s_pad, dtype=torch.uint8, device=dev),
                sq=torch.empty(Hh, S, dtype=torch.float32, device=dev),
                sk=torch.empty(Hh, S, dtype=torch.float32, device=dev),
                sv=torch.empty(Hh, 128, dtype=torch.float32, device=dev))


def run_quantize(plan, S, Hh, q_bits, k_bits, v_bits):
    W = Hh * 128
    q = bf16_to_torch(q_bits).view(S, W)
    k = bf16_to_torch(k_bits).view(S, W)
    v = bf16_to_torch(v_bits).view(S, W)
    b = fp8_buffers(S, Hh)
    H.h3attn_fp8_quantize(plan.handle, q, k, v, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"])
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in b.items()}


def check_quantize(lens, Hh, t, what):
    S = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    with H.Plan(docs_1d(lens), Hh) as plan:
        g = run_quantize(plan, S, Hh, t.q, t.k, t.v)
    q8, sq, k8, sk, v8, sv = ofp8.quantize(synth.bf16_bits_to_f64(t.q), synth.bf16_bits_to_f64(t.k),
                                          synth.bf16_bits_to_f64(t.v), cu)
    assert np.array_equal(g["sq"], sq), f"{what}: q scales"
    assert np.array_equal(g["q8"].reshape(S, Hh, 128), q8), f"{what}: q codes"
    assert np.array_equal(g["sk"], sk), f"{what}: k scales"
    assert np.array_equal(g["k8"].reshape(S, Hh, 128), k8), f"{what}: k codes"
    assert np.array_equal(g["sv"], sv), f"{what}: v scales"
    assert np.array_equal(g["v8t"][:, :, :S], v8.transpose(1, 2, 0)), f"{what}: v codes (transposed)"


@pytest.mark.parametrize("lens,Hh", [([1000, 3, 513, 129, 1], 3), ([255, 256, 257], 2), ([4096], 4)])
def test_quantize_bit_exact(lib, lens, Hh):
    t = random_tensors(sum(lens), Hh, seed=sum(lens) + Hh)
    check_quantize(lens, Hh, t, f"{lens}")


def test_quantize_zero_rows_tiles_channels(lib):
    lens = [300, 200]
    Hh = 2
    t = random_tensors(sum(lens), Hh, seed=31)
    q, k, v = t.q.copy(), t.k.copy(), t.v.copy()
    q[7, 1] = 0                      # an all-zero q row
    k[300:428, 0] = 0                # an all-zero key tile (doc 2's first tile, head 0)
    v[:, 1, 5] = 0                   # an all-zero v channel
    v[:, 0, 9] = 0x8000              # negative zeros
    check_quantize(lens, Hh, synth.Tensors(q, k, v, t.gain_q, t.gain_k), "zeros")


def test_quantize_workload_grid(lib):
    w = synth.config(2)
    t = synth.make_tensors(w)
    check_quantize(list(w.doc_lengths), w.num_heads, t, "config 2")
