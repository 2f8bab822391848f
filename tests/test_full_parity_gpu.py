"""Full-output parity on the three large workloads: every row and every head
of the CUDA path's output against the fp64 oracle (max abs <= 2e-2, mean abs
<= 2e-3 over all S x H x 128 elements, lse within 1e-2), and the FP8 variant
on the Ref2VA-shaped workload within the bound of its P rounding at every
element.

Pages: vllm.cpp PR #26 "feat(minimax-h3)", PR description (per-document
bidirectional attention, the cu_seqlens varlen contract with causal=false).

The oracle's rows are independent, so the comparison runs on a spawn process
pool over (head, block of query rows) tasks (tests/oracle_pool.py); each
workload takes on the order of a minute of host time.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as ofp8
from oracle import plan as oplan
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch
from tests import oracle_pool
from tests.gpu_cases import ATTN_MAX_ABS, ATTN_MEAN_ABS, LSE_MAX_ABS, run_product

pytestmark = pytest.mark.gpu


def _bits(a, S, Hh):
    return np.asarray(a).view(np.uint16).reshape(S, Hh, 128)


def _check(stats, what, report):
    report(f"{what}: max abs {stats['max']:.3e}, mean abs {stats['mean']:.3e}, lse max {stats['lse_max']:.3e} "
           f"over {stats['n']} elements")
    assert stats["finite"], f"{what}: non-finite output"
    assert stats["max"] <= ATTN_MAX_ABS, f"{what}: max abs err {stats['max']:.3e} > {ATTN_MAX_ABS}"
    assert stats["mean"] <= ATTN_MEAN_ABS, f"{what}: mean abs err {stats['mean']:.3e} > {ATTN_MEAN_ABS}"
    assert stats["lse_max"] <= LSE_MAX_ABS, f"{what}: lse max abs err {stats['lse_max']:.3e}"


@pytest.mark.parametrize("n", [3, 4, 5])
def test_workload_full_output_every_row(lib, n, parity_report):
    w = synth.config(n)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    S, Hh = w.S, w.num_heads
    r = run_product(docs, Hh, t)
    cu = oplan.cu_seqlens(docs)
    pos = oplan.positions(docs)
    o_bits = _bits(r.o_bits, S, Hh)
    # end to end: the oracle's own prologue on the raw inputs, then attention
    e2e = oracle_pool.run(oracle_pool.exact_tasks("e2e", cu, pos, t.q, t.k, t.v, o_bits, r.lse, t.gain_q,
                                                  t.gain_k, w.eps, w.softmax_scale))
    _check(e2e, f"{w.name} end to end", parity_report)
    # the attention step alone, on the CUDA prologue's own bf16 outputs
    attn = oracle_pool.run(oracle_pool.exact_tasks("attn", cu, pos, _bits(r.q_bits, S, Hh), _bits(r.k_bits, S, Hh),
                                                   t.v, o_bits, r.lse, t.gain_q, t.gain_k, w.eps, w.softmax_scale))
    _check(attn, f"{w.name} attention only", parity_report)


def test_fp8_forward_ref2va_every_row(lib, parity_report):
    w = synth.config(3)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    S, Hh, W = w.S, w.num_heads, w.num_heads * 128
    dev = torch.device("cuda")
    cu = oplan.cu_seqlens(docs)
    with H.Plan(docs, Hh) as plan:
        q, k, v = (bf16_to_torch(x).view(S, W) for x in (t.q, t.k, t.v))
        gq, gk = torch.from_numpy(t.gain_q).to(dev), torch.from_numpy(t.gain_k).to(dev)
        qh, kh = torch.empty_like(q), torch.empty_like(k)
        H.h3attn_qk_prologue(plan.handle, q, k, qh, kh, gq, gk, w.eps)
        vk = H.h3attn_plan_fp8_v_keys(plan.handle)
        b = dict(q8=torch.empty(S, W, dtype=torch.uint8, device=dev), k8=torch.empty(S, W, dtype=torch.uint8, device=dev),
                 v8t=torch.zeros(Hh, 128, vk, dtype=torch.uint8, device=dev),
                 sq=torch.empty(Hh, S, dtype=torch.float32, device=dev), sk=torch.empty(Hh, S, dtype=torch.float32, device=dev),
                 sv=torch.empty(Hh, 128, dtype=torch.float32, device=dev))
        H.h3attn_fp8_quantize(plan.handle, qh, kh, v, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"])
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((Hh, S), float("nan"), dtype=torch.float32, device=dev)
        H.h3attn_forward_fp8(plan.handle, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"], o, w.softmax_scale, lse)
        H.h3attn_get_device_error(plan.handle)
        o_bits = _bits(o.view(torch.int16).cpu().numpy(), S, Hh)
        lse = lse.cpu().numpy()
        qh64 = qh.double().cpu().numpy().reshape(S, Hh, 128)
        kh64 = kh.double().cpu().numpy().reshape(S, Hh, 128)
        g = {n: x.cpu().numpy() for n, x in b.items()}
    # the oracle's quantisation of the CUDA prologue's outputs; the codes are
    # the kernel's own (bit-exact), so its dequantised values serve
    q8, sq, k8, sk, v8, sv = ofp8.quantize(qh64, kh64, synth.bf16_bits_to_f64(t.v), cu)
    assert np.array_equal(g["q8"].reshape(S, Hh, 128), q8) and np.array_equal(g["sq"], sq)
    assert np.array_equal(g["k8"].reshape(S, Hh, 128), k8) and np.array_equal(g["sk"], sk)
    assert np.array_equal(g["sv"], sv)
    st = oracle_pool.run(oracle_pool.fp8_tasks(cu, q8, sq, k8, sk, v8, sv, o_bits, lse, w.softmax_scale))
    parity_report(f"{w.name} FP8: max abs {st['max']:.3e}, mean abs {st['mean']:.3e} against exact attention "
                  f"on the dequantised inputs; largest error / bound {st['ratio_max']:.3f}; lse max {st['lse_max']:.3e} "
                  f"over {st['n']} elements")
    assert st["finite"], "FP8 Ref2VA: non-finite output"
    assert st["ratio_max"] <= 1.0, f"FP8 Ref2VA: error exceeds the P-rounding bound (ratio {st['ratio_max']:.3f})"
    assert st["lse_max"] <= 1e-3, f"FP8 Ref2VA: lse max abs err {st['lse_max']:.3e}"
