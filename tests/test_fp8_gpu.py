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


def v_offsets(lens):
    """first key of every document in the transposed V (16-key aligned starts)"""
    pads = [(L + 15) // 16 * 16 for L in lens]
    return np.concatenate([[0], np.cumsum(pads)])


def fp8_buffers(S, Hh, v_keys):
    dev = torch.device("cuda")
    return dict(q8=torch.empty(S, Hh * 128, dtype=torch.uint8, device=dev),
                k8=torch.empty(S, Hh * 128, dtype=torch.uint8, device=dev),
                v8t=torch.full((Hh, 128, v_keys), 0x7F, dtype=torch.uint8, device=dev),  # NaN codes: gaps must be written
                sq=torch.empty(Hh, S, dtype=torch.float32, device=dev),
                sk=torch.empty(Hh, S, dtype=torch.float32, device=dev),
                sv=torch.empty(Hh, 128, dtype=torch.float32, device=dev))


def run_quantize(plan, S, Hh, q_bits, k_bits, v_bits):
    W = Hh * 128
    q = bf16_to_torch(q_bits).view(S, W)
    k = bf16_to_torch(k_bits).view(S, W)
    v = bf16_to_torch(v_bits).view(S, W)
    b = fp8_buffers(S, Hh, H.h3attn_plan_fp8_v_keys(plan.handle))
    H.h3attn_fp8_quantize(plan.handle, q, k, v, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"])
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in b.items()}, b


def check_quantize(lens, Hh, t, what):
    S = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    with H.Plan(docs_1d(lens), Hh) as plan:
        assert H.h3attn_plan_fp8_v_keys(plan.handle) == v_offsets(lens)[-1]
        g, _ = run_quantize(plan, S, Hh, t.q, t.k, t.v)
    q8, sq, k8, sk, v8, sv = ofp8.quantize(synth.bf16_bits_to_f64(t.q), synth.bf16_bits_to_f64(t.k),
                                          synth.bf16_bits_to_f64(t.v), cu)
    assert np.array_equal(g["sq"], sq), f"{what}: q scales"
    assert np.array_equal(g["q8"].reshape(S, Hh, 128), q8), f"{what}: q codes"
    assert np.array_equal(g["sk"], sk), f"{what}: k scales"
    assert np.array_equal(g["k8"].reshape(S, Hh, 128), k8), f"{what}: k codes"
    assert np.array_equal(g["sv"], sv), f"{what}: v scales"
    vo = v_offsets(lens)
    for d, L in enumerate(lens):
        a = int(cu[d])
        seg = g["v8t"][:, :, vo[d]:vo[d + 1]]
        assert np.array_equal(seg[:, :, :L], v8[a:a + L].transpose(1, 2, 0)), f"{what}: v codes, doc {d}"
        assert not seg[:, :, L:].any(), f"{what}: v gap after doc {d} not zero"


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


def run_fp8(lens, Hh, t, scale=None):
    """prologue (bf16) -> FP8 quantisation -> FP8 forward; returns the GPU
    output, its lse, and the quantised inputs (host)"""
    S = sum(lens)
    W = Hh * 128
    scale = 1.0 / np.sqrt(128.0) if scale is None else scale
    dev = torch.device("cuda")
    with H.Plan(docs_1d(lens), Hh) as plan:
        q = bf16_to_torch(t.q).view(S, W)
        k = bf16_to_torch(t.k).view(S, W)
        v = bf16_to_torch(t.v).view(S, W)
        qh, kh = torch.empty_like(q), torch.empty_like(k)
        H.h3attn_qk_prologue(plan.handle, q, k, qh, kh, torch.from_numpy(t.gain_q).to(dev),
                             torch.from_numpy(t.gain_k).to(dev), 1e-6)
        b = fp8_buffers(S, Hh, H.h3attn_plan_fp8_v_keys(plan.handle))
        H.h3attn_fp8_quantize(plan.handle, qh, kh, v, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"])
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((Hh, S), float("nan"), dtype=torch.float32, device=dev)
        H.h3attn_forward_fp8(plan.handle, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"], o, scale, lse)
        H.h3attn_get_device_error(plan.handle)
        host = {n: x.cpu().numpy() for n, x in b.items()}
        return (o.double().cpu().numpy().reshape(S, Hh, 128), lse.cpu().numpy(),
                qh.double().cpu().numpy().reshape(S, Hh, 128), kh.double().cpu().numpy().reshape(S, Hh, 128), host)


def check_fp8_forward(lens, Hh, t, rows=None, what=""):
    from oracle import attention as oatt
    S = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    scale = 1.0 / np.sqrt(128.0)
    o, lse, qh, kh, g = run_fp8(lens, Hh, t, scale)
    # the quantised inputs are the oracle's (bit-exact), so the oracle's dequantised values serve
    q8, sq, k8, sk, v8, sv = ofp8.quantize(qh, kh, synth.bf16_bits_to_f64(t.v), cu)
    assert np.array_equal(g["q8"].reshape(S, Hh, 128), q8) and np.array_equal(g["sk"], sk)
    qd, kd, vd = ofp8.dequantize(q8, sq, k8, sk, v8, sv)
    rows = np.arange(S) if rows is None else rows
    o_ref, lse_ref = oatt.attention_rows(qd[rows], kd, vd, cu, scale, range(Hh), rows)
    bound = ofp8.error_bound(qd, kd, vd, cu, scale, range(Hh), rows)
    tol = bound + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    err = np.abs(o[rows] - o_ref)
    assert np.all(np.isfinite(o[rows])), f"{what}: non-finite output"
    worst = float((err / tol).max())
    assert worst <= 1.0, f"{what}: error {err.max():.3e} exceeds the P-rounding bound (ratio {worst:.2f})"
    assert float(np.abs(lse[:, rows] - lse_ref).max()) <= 1e-3, f"{what}: lse"
    return float(err.max()), float(err.mean())


@pytest.mark.parametrize("lens,Hh", [([1000, 3, 513, 129, 1], 3), ([255, 256, 257, 700], 2)])
def test_fp8_forward_within_bound(lib, lens, Hh):
    t = random_tensors(sum(lens), Hh, seed=17 + len(lens))
    check_fp8_forward(lens, Hh, t, what=str(lens))


def test_fp8_rejects_bad_arguments(lib):
    lens, Hh = [300, 40], 2
    S = sum(lens)
    dev = torch.device("cuda")
    with H.Plan(docs_1d(lens), Hh) as plan:
        vk = H.h3attn_plan_fp8_v_keys(plan.handle)
        assert vk == 304 + 48
        x = torch.zeros(S, Hh * 128, dtype=torch.bfloat16, device=dev)
        b = fp8_buffers(S, Hh, vk)
        args = [b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"]]
        # an output overlapping an input, two overlapping outputs, a misaligned scale pointer
        for bad in ([x.view(torch.uint8)[:, :Hh * 128]] + args[1:], [args[0], args[0]] + args[2:],
                    args[:3] + [b["sq"].view(-1)[1:]] + args[4:]):
            with pytest.raises(H.H3AttnError) as e:
                H.h3attn_fp8_quantize(plan.handle, x, x, x, *bad)
            assert e.value.status == H.H3ATTN_EINVAL
        o = torch.zeros(S, Hh * 128, dtype=torch.bfloat16, device=dev)
        with pytest.raises(H.H3AttnError):
            H.h3attn_forward_fp8(plan.handle, *args, o, float("nan"))
        with pytest.raises(H.H3AttnError):  # o overlapping q8
            H.h3attn_forward_fp8(plan.handle, *args, b["q8"].view(torch.bfloat16), 0.1)
        H.h3attn_fp8_quantize(plan.handle, x, x, x, *args)  # valid calls still work
        H.h3attn_forward_fp8(plan.handle, *args, o, 0.1)
        H.h3attn_get_device_error(plan.handle)
        assert H.h3attn_plan_forward_kernels(plan.handle) in (1, 2)


def fused_vs_two_calls(docs, Hh, t, fused_qkv=False, per_head_gains=False):
    """h3attn_qk_prologue_fp8 against h3attn_qk_prologue + h3attn_fp8_quantize:
    every code and scale bit-identical (and the transposed V's gaps zero)."""
    dev = torch.device("cuda")
    S = int(t.q.shape[0])
    W = Hh * 128
    if fused_qkv:  # q, k, v as views of one [S, 3 W] buffer
        buf = torch.empty(S, 3 * W, dtype=torch.bfloat16, device=dev)
        q, k, v = buf[:, :W], buf[:, W:2 * W], buf[:, 2 * W:]
        for dst, bits in ((q, t.q), (k, t.k), (v, t.v)):
            dst.copy_(bf16_to_torch(bits).view(S, W))
    else:
        q, k, v = (bf16_to_torch(x).view(S, W) for x in (t.q, t.k, t.v))
    if per_head_gains:
        rng = np.random.default_rng(5)
        gq = torch.from_numpy((1 + 0.1 * rng.standard_normal((Hh, 128))).astype(np.float32)).to(dev)
        gk = torch.from_numpy((1 + 0.1 * rng.standard_normal((Hh, 128))).astype(np.float32)).to(dev)
        ghs = 128
    else:
        gq, gk, ghs = torch.from_numpy(t.gain_q).to(dev), torch.from_numpy(t.gain_k).to(dev), 0
    with H.Plan(docs, Hh) as plan:
        vk = H.h3attn_plan_fp8_v_keys(plan.handle)
        qh = torch.empty(S, W, dtype=torch.bfloat16, device=dev)
        kh = torch.empty_like(qh)
        H.h3attn_qk_prologue(plan.handle, q, k, qh, kh, gq, gk, 1e-6, gain_head_stride=ghs)
        a = fp8_buffers(S, Hh, vk)
        H.h3attn_fp8_quantize(plan.handle, qh, kh, v.contiguous(), a["q8"], a["k8"], a["v8t"], a["sq"], a["sk"],
                              a["sv"])
        b = fp8_buffers(S, Hh, vk)
        H.h3attn_qk_prologue_fp8(plan.handle, q, k, v, gq, gk, 1e-6, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"],
                                 b["sv"], gain_head_stride=ghs)
        H.h3attn_get_device_error(plan.handle)
        for n in a:
            assert torch.equal(a[n], b[n]), f"{n} differs between the fused and the two-call paths"


@pytest.mark.parametrize("case", ["ragged", "grid_video", "ref2va", "fused_qkv_per_head_gains"])
def test_prologue_fp8_matches_prologue_then_quantize(lib, case):
    if case == "ragged":
        lens, Hh = [1000, 3, 513, 129, 1], 3
        fused_vs_two_calls(docs_1d(lens), Hh, random_tensors(sum(lens), Hh, seed=41))
    elif case in ("grid_video", "ref2va"):
        w = synth.config(2 if case == "grid_video" else 3)
        fused_vs_two_calls(synth.spans_to_tuples(w.docs), w.num_heads, synth.make_tensors(w))
    else:
        lens, Hh = [777, 300, 64], 7
        fused_vs_two_calls(docs_1d(lens), Hh, random_tensors(sum(lens), Hh, seed=43), fused_qkv=True,
                           per_head_gains=True)


def test_prologue_fp8_forward_within_bound(lib):
    # the FP8 step through the fused call, against exact attention on the
    # dequantised values of the oracle's own quantisation of the bf16 prologue
    from oracle import attention as oatt
    lens, Hh = [700, 129, 1, 300], 2
    S = sum(lens)
    W = Hh * 128
    cu = np.concatenate([[0], np.cumsum(lens)])
    scale = 1.0 / np.sqrt(128.0)
    t = random_tensors(S, Hh, seed=47)
    dev = torch.device("cuda")
    q, k, v = (bf16_to_torch(x).view(S, W) for x in (t.q, t.k, t.v))
    gq, gk = torch.from_numpy(t.gain_q).to(dev), torch.from_numpy(t.gain_k).to(dev)
    with H.Plan(docs_1d(lens), Hh) as plan:
        qh, kh = torch.empty_like(q), torch.empty_like(k)
        H.h3attn_qk_prologue(plan.handle, q, k, qh, kh, gq, gk, 1e-6)
        b = fp8_buffers(S, Hh, H.h3attn_plan_fp8_v_keys(plan.handle))
        H.h3attn_qk_prologue_fp8(plan.handle, q, k, v, gq, gk, 1e-6, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"],
                                 b["sv"])
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device=dev)
        H.h3attn_forward_fp8(plan.handle, b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"], o, scale)
        H.h3attn_get_device_error(plan.handle)
        o = o.double().cpu().numpy().reshape(S, Hh, 128)
        qh = qh.double().cpu().numpy().reshape(S, Hh, 128)
        kh = kh.double().cpu().numpy().reshape(S, Hh, 128)
    q8, sq, k8, sk, v8, sv = ofp8.quantize(qh, kh, synth.bf16_bits_to_f64(t.v), cu)
    assert np.array_equal(b["q8"].cpu().numpy().reshape(S, Hh, 128), q8)
    assert np.array_equal(b["k8"].cpu().numpy().reshape(S, Hh, 128), k8)
    assert np.array_equal(b["sk"].cpu().numpy(), sk) and np.array_equal(b["sv"].cpu().numpy(), sv)
    qd, kd, vd = ofp8.dequantize(q8, sq, k8, sk, v8, sv)
    rows = np.arange(S)
    o_ref, _ = oatt.attention_rows(qd, kd, vd, cu, scale, range(Hh), rows)
    tol = ofp8.error_bound(qd, kd, vd, cu, scale, range(Hh), rows) + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    assert np.all(np.abs(o - o_ref) <= tol)


def test_prologue_fp8_rejects_bad_arguments(lib):
    lens, Hh = [300, 40], 2
    S = sum(lens)
    dev = torch.device("cuda")
    x = torch.zeros(S, Hh * 128, dtype=torch.bfloat16, device=dev)
    g = torch.ones(128, dtype=torch.float32, device=dev)
    with H.Plan(docs_1d(lens), Hh) as plan:
        b = fp8_buffers(S, Hh, H.h3attn_plan_fp8_v_keys(plan.handle))
        outs = [b["q8"], b["k8"], b["v8t"], b["sq"], b["sk"], b["sv"]]
        for call in (lambda: H.h3attn_qk_prologue_fp8(plan.handle, x, x, x, None, g, 1e-6, *outs),
                     lambda: H.h3attn_qk_prologue_fp8(plan.handle, x, x, x, g, g, -1.0, *outs),
                     lambda: H.h3attn_qk_prologue_fp8(plan.handle, x, x, x, g, g, 1e-6, *outs, gain_head_stride=64),
                     lambda: H.h3attn_qk_prologue_fp8(plan.handle, x, x, x, g, g, 1e-6,
                                                      x.view(torch.uint8)[:, :Hh * 128], *outs[1:])):
            with pytest.raises(H.H3AttnError) as e:
                call()
            assert e.value.status == H.H3ATTN_EINVAL
        H.h3attn_qk_prologue_fp8(plan.handle, x, x, x, g, g, 1e-6, *outs)  # a valid call still works
        H.h3attn_get_device_error(plan.handle)
