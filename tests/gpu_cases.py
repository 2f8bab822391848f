"""Running the library and the oracle on the same seeded inputs (test helper).

``run_product`` drives the CUDA path through the C ABI (plan, prologue,
forward); ``oracle_reference`` computes the same quantities with the fp64
oracle, optionally on a sample of query rows.  The two share nothing but the
seeded bf16 inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import attention as oatt
from oracle import plan as oplan
from oracle import prologue as opro
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch, torch_bf16_to_f64

# Tolerances of the CUDA path against the fp64 oracle (bf16 I/O, fp32 accumulation).
ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-2
# prologue: one bf16 rounding of an fp32 result (half an ulp = 2^-8 relative)
# plus fp32 arithmetic on O(1) operands
PRO_REL = 2.0 ** -8
PRO_ABS = 2e-5


def random_tensors(S, H_, seed, gain_scale=0.1):
    """Seeded N(0,1) bf16 tensors for ad-hoc document layouts."""
    n = S * H_ * 128
    q = synth.normal_bf16_bits(seed, synth.STREAM_Q, n).reshape(S, H_, 128)
    k = synth.normal_bf16_bits(seed, synth.STREAM_K, n).reshape(S, H_, 128)
    v = synth.normal_bf16_bits(seed, synth.STREAM_V, n).reshape(S, H_, 128)
    gq = (1.0 + gain_scale * synth.normal(seed, synth.STREAM_GAIN_Q, 128)).astype(np.float32)
    gk = (1.0 + gain_scale * synth.normal(seed, synth.STREAM_GAIN_K, 128)).astype(np.float32)
    return synth.Tensors(q, k, v, gq, gk)


def docs_1d(lengths):
    """Documents that are plain 1D runs of the given lengths."""
    return [[(L, 1, 1, (0.0, 0.0, 0.0), (1.0, 0.0, 0.0))] for L in lengths]


class ProductResult:
    pass


def run_product(docs, num_heads, t: synth.Tensors, eps=1e-6, scale=None, stream=None,
                fused=False, want_lse=True, keep_device=False, fused_q=False):
    """Plan + prologue + forward through the C ABI; returns host copies.
    fused=True reads q/k/v from one fused-qkv buffer (prologue in place);
    fused_q=True runs the k-only prologue and the forward with the Q prologue
    fused in (q_hat is then not materialised: r.q_hat is None)."""
    scale = (1.0 / np.sqrt(128.0)) if scale is None else scale
    dev = torch.device("cuda")
    with H.Plan(docs, num_heads, stream=stream) as plan:
        S = plan.info["S"]
        W = num_heads * 128
        if fused:
            buf = torch.zeros(S, 3 * W, dtype=torch.bfloat16, device=dev)
            q_in, k_in, v = buf[:, :W], buf[:, W:2 * W], buf[:, 2 * W:]
            q_in.copy_(bf16_to_torch(t.q).view(S, W))
            k_in.copy_(bf16_to_torch(t.k).view(S, W))
            v.copy_(bf16_to_torch(t.v).view(S, W))
        else:
            q_in = bf16_to_torch(t.q).view(S, W)
            k_in = bf16_to_torch(t.k).view(S, W)
            v = bf16_to_torch(t.v).view(S, W)
        gq = torch.from_numpy(t.gain_q).to(dev)
        gk = torch.from_numpy(t.gain_k).to(dev)
        if fused:
            # prologue in place inside the fused buffer, so q, k and v share one row stride
            q_hat, k_hat = q_in, k_in
        else:
            q_hat = torch.empty(S, W, dtype=torch.bfloat16, device=dev)
            k_hat = torch.empty_like(q_hat)
        o = torch.full((S, W), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((num_heads, S), float("nan"), dtype=torch.float32, device=dev) if want_lse else None
        if fused_q:
            H.h3attn_qk_prologue(plan.handle, None, k_in, None, k_hat, None, gk, eps, stream=stream)
            H.h3attn_forward_fused_q(plan.handle, q_in, k_hat, v, o, gq, scale, eps, lse, stream=stream)
        else:
            H.h3attn_qk_prologue(plan.handle, q_in, k_in, q_hat, k_hat, gq, gk, eps, stream=stream)
            H.h3attn_forward(plan.handle, q_hat, k_hat, v, o, scale, lse, stream=stream)
        H.h3attn_get_device_error(plan.handle, stream=stream)
        r = ProductResult()
        r.S = S
        r.q_hat = None if fused_q else torch_bf16_to_f64(q_hat).reshape(S, num_heads, 128)
        r.k_hat = torch_bf16_to_f64(k_hat).reshape(S, num_heads, 128)
        r.o = torch_bf16_to_f64(o).reshape(S, num_heads, 128)
        r.o_bits = o.view(torch.int16).cpu().numpy()
        r.k_bits = k_hat.view(torch.int16).cpu().numpy()
        r.q_bits = None if fused_q else q_hat.view(torch.int16).cpu().numpy()
        r.lse = lse.cpu().numpy() if want_lse else None
        if keep_device:
            r.dev = dict(q_hat=q_hat, k_hat=k_hat, v=v, o=o)
        return r


def sample_rows(cu, per_edge=40, interior=48, seed=0):
    """First and last rows of every document plus random interior rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for d in range(len(cu) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        rows.extend(range(a, min(b, a + per_edge)))
        rows.extend(range(max(a, b - per_edge), b))
        if b - a > 2 * per_edge:
            rows.extend(rng.integers(a + per_edge, b - per_edge, interior).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))


def oracle_reference(docs, t: synth.Tensors, eps=1e-6, scale=None, rows=None, q_hat=None,
                     k_hat=None):
    """fp64 oracle.  Without q_hat/k_hat it runs the oracle prologue on the
    bf16 inputs; with them (fp64 arrays of the GPU prologue's bf16 outputs)
    it checks the attention step alone."""
    scale = (1.0 / np.sqrt(128.0)) if scale is None else scale
    pos = oplan.positions(docs)
    cu = oplan.cu_seqlens(docs)
    S = int(cu[-1])
    rows = np.arange(S) if rows is None else np.asarray(rows)
    if q_hat is None:
        xq = synth.bf16_bits_to_f64(t.q[rows])
        q_sel = opro.qk_prologue(xq, t.gain_q.astype(np.float64), pos[rows], eps)
        xk = synth.bf16_bits_to_f64(t.k)
        k_full = opro.qk_prologue(xk, t.gain_k.astype(np.float64), pos, eps)
    else:
        q_sel, k_full = q_hat[rows], k_hat
    v = synth.bf16_bits_to_f64(t.v)
    H_ = t.q.shape[1]
    o, lse = oatt.attention_rows(q_sel, k_full, v, cu, scale, range(H_), rows)
    return rows, o, lse, cu


def check_attention(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what=""):
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= ATTN_MAX_ABS, f"{what}: max abs err {mx:.3e} > {ATTN_MAX_ABS}"
    assert mean <= ATTN_MEAN_ABS, f"{what}: mean abs err {mean:.3e} > {ATTN_MEAN_ABS}"
    if lse_gpu is not None:
        le = float(np.abs(lse_gpu - lse_ref).max())
        assert le <= LSE_MAX_ABS, f"{what}: lse max abs err {le:.3e}"
    return mx, mean


def check_prologue(y_gpu, y_ref, what=""):
    bad = np.abs(y_gpu - y_ref) > PRO_REL * np.abs(y_ref) + PRO_ABS
    n = int(bad.sum())
    assert n == 0, (f"{what}: {n} prologue elements out of tolerance; worst "
                    f"{np.abs(y_gpu - y_ref).max():.3e}")
