"""Prologue parity: the CUDA RMSNorm + rot96 kernel against the fp64 oracle,
element by element, plus layout and stream invariance (byte-identical)."""
import numpy as np
import pytest
import torch

import synth
from oracle import plan as oplan
from oracle import prologue as opro
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch, torch_bf16_to_f64
from tests.gpu_cases import check_prologue, random_tensors

pytestmark = pytest.mark.gpu


def _oracle(docs, x_bits, gain, eps=1e-6):
    pos = oplan.positions(docs)
    return opro.qk_prologue(synth.bf16_bits_to_f64(x_bits), gain.astype(np.float64), pos, eps)


def _run(plan, q_in, k_in, q_out, k_out, gq, gk, eps=1e-6, ghs=0, stream=None):
    H.h3attn_qk_prologue(plan.handle, q_in, k_in, q_out, k_out, gq, gk, eps,
                         gain_head_stride=ghs, stream=stream)
    torch.cuda.synchronize()


@pytest.mark.parametrize("n", [1, 2, 3])
def test_prologue_matches_oracle(lib, n):
    w = synth.config(n)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    S, W = w.S, w.num_heads * 128
    with H.Plan(docs, w.num_heads) as p:
        q = bf16_to_torch(t.q).view(S, W)
        k = bf16_to_torch(t.k).view(S, W)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        _run(p, q, k, qo, ko, torch.from_numpy(t.gain_q).cuda(), torch.from_numpy(t.gain_k).cuda())
        yq = torch_bf16_to_f64(qo).reshape(S, w.num_heads, 128)
        yk = torch_bf16_to_f64(ko).reshape(S, w.num_heads, 128)
    check_prologue(yq, _oracle(docs, t.q, t.gain_q), "q")
    check_prologue(yk, _oracle(docs, t.k, t.gain_k), "k")


def test_prologue_layouts_and_streams_are_byte_identical(lib):
    docs = [[(3, 5, 7, (-2.0, 0.0, 0.0), (1.0, 1.0, 1.0))], [(77, 1, 1, (0.0, 0.0, 0.0), (1.0, 0.0, 0.0))]]
    Hh = 5
    S, W = 105 + 77, 5 * 128
    t = random_tensors(S, Hh, 77)
    gq, gk = torch.from_numpy(t.gain_q).cuda(), torch.from_numpy(t.gain_k).cuda()
    with H.Plan(docs, Hh) as p:
        q = bf16_to_torch(t.q).view(S, W)
        k = bf16_to_torch(t.k).view(S, W)
        q0, k0 = torch.empty_like(q), torch.empty_like(k)
        _run(p, q, k, q0, k0, gq, gk)
        ref = (q0.clone(), k0.clone())
        # non-default stream
        s = torch.cuda.Stream()
        q1, k1 = torch.empty_like(q), torch.empty_like(k)
        with torch.cuda.stream(s):
            _run(p, q, k, q1, k1, gq, gk, stream=s)
        assert torch.equal(q1.view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(k1.view(torch.int16), ref[1].view(torch.int16))
        # fused qkv input, strided output, in place
        buf = torch.zeros(S, 3 * W, dtype=torch.bfloat16, device="cuda")
        buf[:, :W].copy_(q)
        buf[:, W:2 * W].copy_(k)
        _run(p, buf[:, :W], buf[:, W:2 * W], buf[:, :W], buf[:, W:2 * W], gq, gk)
        assert torch.equal(buf[:, :W].view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(buf[:, W:2 * W].view(torch.int16), ref[1].view(torch.int16))
        # padded output rows
        out = torch.zeros(S, W + 64, dtype=torch.bfloat16, device="cuda")
        out2 = torch.zeros(S, W + 64, dtype=torch.bfloat16, device="cuda")
        H.h3attn_qk_prologue(p.handle, q, k, out, out2, gq, gk, 1e-6, in_row_stride=W,
                             out_row_stride=W + 64)
        torch.cuda.synchronize()
        assert torch.equal(out[:, :W].view(torch.int16), ref[0].view(torch.int16))
        assert torch.all(out[:, W:] == 0)


def test_prologue_per_head_gains(lib):
    docs = [[(2, 6, 6, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    Hh, S = 4, 72
    t = random_tensors(S, Hh, 91)
    rng = np.random.default_rng(1)
    gq = (1 + 0.3 * rng.standard_normal((Hh, 132))).astype(np.float32)  # padded head stride
    gk = (1 + 0.3 * rng.standard_normal((Hh, 132))).astype(np.float32)
    with H.Plan(docs, Hh) as p:
        q = bf16_to_torch(t.q).view(S, Hh * 128)
        k = bf16_to_torch(t.k).view(S, Hh * 128)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        _run(p, q, k, qo, ko, torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda(), ghs=132)
        yq = torch_bf16_to_f64(qo).reshape(S, Hh, 128)
    check_prologue(yq, _oracle(docs, t.q, gq[:, :128]), "per-head gain")


def test_prologue_extreme_scales(lib):
    # tiny and large inputs: the norm removes the scale; eps = 0 and a large eps
    docs = [[(1, 4, 4, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    Hh, S = 2, 16
    rng = np.random.default_rng(2)
    for scale, eps in ((1e-3, 1e-6), (300.0, 1e-6), (1.0, 0.0), (1.0, 10.0)):
        x = (rng.standard_normal((S, Hh, 128)) * scale).astype(np.float32)
        bits = synth.f32_to_bf16_bits(x)
        g = np.ones(128, dtype=np.float32)
        with H.Plan(docs, Hh) as p:
            q = bf16_to_torch(bits).view(S, Hh * 128)
            qo, ko = torch.empty_like(q), torch.empty_like(q)
            gg = torch.from_numpy(g).cuda()
            _run(p, q, q.clone(), qo, ko, gg, gg, eps=eps)
            y = torch_bf16_to_f64(qo).reshape(S, Hh, 128)
        check_prologue(y, _oracle(docs, bits, g, eps), f"scale {scale} eps {eps}")


def test_prologue_rejects_bad_arguments(lib):
    docs = [[(1, 4, 4, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    with H.Plan(docs, 2) as p:
        q = torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros_like(q)
        o1, o2 = torch.zeros_like(q), torch.zeros_like(q)
        g = torch.ones(128, device="cuda")
        bad = [
            dict(q_out=q.view(-1)[8:], k_out=o2, in_row_stride=256, out_row_stride=256),  # misaligned/partial overlap
            dict(q_out=o1, k_out=o1),                                                   # outputs overlap
            dict(q_out=k, k_out=o2),                                                    # q_out aliases k_in
        ]
        for kw in bad:
            with pytest.raises(H.H3AttnError) as e:
                H.h3attn_qk_prologue(p.handle, q, k, kw["q_out"], kw["k_out"], g, g, 1e-6,
                                     in_row_stride=kw.get("in_row_stride"),
                                     out_row_stride=kw.get("out_row_stride"))
            assert e.value.status == H.H3ATTN_EINVAL
        with pytest.raises(H.H3AttnError):
            H.h3attn_qk_prologue(p.handle, q, k, o1, o2, g, g, -1.0)
        with pytest.raises(H.H3AttnError):
            H.h3attn_qk_prologue(p.handle, q, k, o1, o2, g, g, 1e-6, in_row_stride=200, out_row_stride=256)


@pytest.mark.parametrize("Hh,k_only", [(200, False), (21, True), (3, True)])
def test_prologue_kernel_paths(lib, Hh, k_only):
    # 200 heads (a wide token row); k only: the mode used with the fused-Q
    # forward.  Both against the oracle, and k only byte-identical to the q+k
    # call's k.
    lens = [37, 130] if Hh == 200 else [700, 93, 1]
    docs = [[(L, 1, 1, (0.0, 0.0, 0.0), (1.0, 0.0, 0.0))] for L in lens]
    S, W = sum(lens), Hh * 128
    t = random_tensors(S, Hh, seed=Hh + (7 if k_only else 0))
    gq, gk = torch.from_numpy(t.gain_q).cuda(), torch.from_numpy(t.gain_k).cuda()
    with H.Plan(docs, Hh) as p:
        q = bf16_to_torch(t.q).view(S, W)
        k = bf16_to_torch(t.k).view(S, W)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        _run(p, q, k, qo, ko, gq, gk)
        yk = torch_bf16_to_f64(ko).reshape(S, Hh, 128)
        check_prologue(yk, _oracle(docs, t.k, t.gain_k), f"k, {Hh} heads")
        yq = torch_bf16_to_f64(qo).reshape(S, Hh, 128)
        check_prologue(yq, _oracle(docs, t.q, t.gain_q), f"q, {Hh} heads")
        if k_only:
            ko2 = torch.empty_like(k)
            _run(p, None, k, None, ko2, None, gk)
            assert torch.equal(ko2.view(torch.int16), ko.view(torch.int16))


@pytest.mark.parametrize("Hh,S", [(21, 4096), (56, 1024), (16, 4096)])
def test_prologue_per_head_gains_full_grid(lib, Hh, S):
    # More rows than one pass of the grid (8 blocks of 16 rows per SM), so every
    # 16-lane group runs several rows: the grid-stride step must keep each
    # group on one head, whose gains it loads once (21, 56 and 16 heads give
    # grid units of 21, 7 and 1 blocks).
    docs = [[(S // 64, 8, 8, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    t = random_tensors(S, Hh, 97 + Hh)
    rng = np.random.default_rng(Hh)
    gq = (1 + 0.3 * rng.standard_normal((Hh, 128))).astype(np.float32)
    gk = (1 + 0.3 * rng.standard_normal((Hh, 128))).astype(np.float32)
    with H.Plan(docs, Hh) as p:
        q = bf16_to_torch(t.q).view(S, Hh * 128)
        k = bf16_to_torch(t.k).view(S, Hh * 128)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        _run(p, q, k, qo, ko, torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda(), ghs=128)
        yq = torch_bf16_to_f64(qo).reshape(S, Hh, 128)
        yk = torch_bf16_to_f64(ko).reshape(S, Hh, 128)
    check_prologue(yq, _oracle(docs, t.q, gq), f"per-head q gains, {Hh} heads")
    check_prologue(yk, _oracle(docs, t.k, gk), f"per-head k gains, {Hh} heads")
