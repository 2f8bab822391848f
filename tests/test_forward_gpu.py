"""Attention parity: the CUDA path (prologue + forward, through the C ABI)
against the fp64 oracle on the two smaller workloads and on edge cases (the
three large workloads are compared on every row in test_full_parity_gpu.py);
segment isolation must hold bit for bit."""
import numpy as np
import pytest
import torch

import synth
from packed_varlen_non_gb300 import h3attn as H
from synth.device import bf16_to_torch
from tests.gpu_cases import (check_attention, docs_1d, oracle_reference, random_tensors,
                             run_product, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 2])
def test_workload_full_output(lib, n):
    w = synth.config(n)
    t = synth.make_tensors(w)
    docs = synth.spans_to_tuples(w.docs)
    r = run_product(docs, w.num_heads, t)
    rows, o, lse, _ = oracle_reference(docs, t)
    check_attention(r.o, o, r.lse, lse, f"config {n} end to end")
    # the attention step alone, on the GPU prologue's own bf16 outputs
    rows, o2, lse2, _ = oracle_reference(docs, t, q_hat=r.q_hat, k_hat=r.k_hat)
    check_attention(r.o, o2, r.lse, lse2, f"config {n} attention only")


EDGE_LAYOUTS = {
    "one_token": [1],
    "single_tiles": [1, 7, 127, 128, 129],
    "tile_boundaries": [255, 256, 257, 383, 384, 385],
    "long_ragged": [1000, 3, 513],
    "many_tiny": [int(x) for x in np.random.default_rng(11).integers(1, 40, 60)],
    # about six units per CTA pair, consecutive units switching between one
    # and two active query tiles and between one and several key tiles
    "mixed_query_tiles": [700, 600, 200, 300, 100, 128, 257, 1, 513] * 12,
}


@pytest.mark.parametrize("name", sorted(EDGE_LAYOUTS))
def test_edge_layouts(lib, name):
    lens = EDGE_LAYOUTS[name]
    docs = docs_1d(lens)
    Hh = 3
    t = random_tensors(sum(lens), Hh, seed=len(lens) * 7 + 1)
    r = run_product(docs, Hh, t)
    _, o, lse, _ = oracle_reference(docs, t, q_hat=r.q_hat, k_hat=r.k_hat)
    check_attention(r.o, o, r.lse, lse, name)


def test_one_token_documents_return_v(lib):
    docs = docs_1d([1, 1, 1, 5, 1])
    t = random_tensors(9, 2, seed=3)
    r = run_product(docs, 2, t)
    v = synth.bf16_bits_to_f64(t.v)
    for i in (0, 1, 2, 8):
        np.testing.assert_array_equal(r.o[i], v[i])


def test_zero_gain_gives_document_mean(lib):
    lens = [130, 77, 300]
    docs = docs_1d(lens)
    t = random_tensors(sum(lens), 2, seed=4)
    t.gain_q[:] = 0.0
    r = run_product(docs, 2, t)
    v = synth.bf16_bits_to_f64(t.v)
    a = 0
    for L in lens:
        mean = v[a:a + L].mean(axis=0)
        check_attention(r.o[a:a + L], np.broadcast_to(mean, (L, 2, 128)), what=f"mean of doc len {L}")
        a += L


def test_segment_isolation_bit_exact(lib):
    lens = [300, 517, 129]
    docs = docs_1d(lens)
    Hh = 3
    t = random_tensors(sum(lens), Hh, seed=21)
    r0 = run_product(docs, Hh, t)
    t2 = synth.Tensors(t.q.copy(), t.k.copy(), t.v.copy(), t.gain_q, t.gain_k)
    rng = np.random.default_rng(0)
    for arr in (t2.q, t2.k, t2.v):
        idx = 300 + rng.integers(0, 517, 20)
        arr[idx] ^= np.uint16(0x0040)  # flip a mantissa bit of a few doc-2 tokens
    r1 = run_product(docs, Hh, t2)
    assert np.array_equal(r1.o_bits[:300], r0.o_bits[:300])
    assert np.array_equal(r1.o_bits[817:], r0.o_bits[817:])
    assert not np.array_equal(r1.o_bits[300:817], r0.o_bits[300:817])


def test_streams_and_fused_layout_are_byte_identical(lib):
    lens = [400, 250]
    docs = docs_1d(lens)
    t = random_tensors(650, 4, seed=8)
    r0 = run_product(docs, 4, t)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r1 = run_product(docs, 4, t, stream=s)
    r2 = run_product(docs, 4, t, fused=True)
    assert np.array_equal(r0.o_bits, r1.o_bits)
    assert np.array_equal(r0.o_bits, r2.o_bits)
    r3 = run_product(docs, 4, t, want_lse=False)
    assert np.array_equal(r0.o_bits, r3.o_bits)


def test_forward_rejects_bad_arguments(lib):
    docs = docs_1d([64])
    with H.Plan(docs, 2) as p:
        q = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda")
        k, v, o = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
        for args in ((q, k, v, q), (q, k, v, v)):  # o aliases an input
            with pytest.raises(H.H3AttnError) as e:
                H.h3attn_forward(p.handle, *args, 0.1)
            assert e.value.status == H.H3ATTN_EINVAL
        with pytest.raises(H.H3AttnError):
            H.h3attn_forward(p.handle, q, k, v, o, float("nan"))
        with pytest.raises(H.H3AttnError):
            H.h3attn_forward(p.handle, q.view(-1)[4:], k, v, o, 0.1, qkv_row_stride=256, o_row_stride=256)
        with pytest.raises(H.H3AttnError):
            H.h3attn_forward(p.handle, q, k, v, o, 0.1, qkv_row_stride=100, o_row_stride=256)
        H.h3attn_forward(p.handle, q, k, v, o, 0.1)  # valid call still works
        H.h3attn_get_device_error(p.handle)


def test_shipped_dit_geometry_fused_qkv(lib):
    # the shipped DiT block: 56 heads x 128 (hidden 7168), q/k/v read straight
    # out of a fused-qkv buffer [S, 3*H*128] through the row stride, prologue in place
    lens = [1000, 777]
    docs = docs_1d(lens)
    Hh = 56
    t = random_tensors(sum(lens), Hh, seed=56)
    r = run_product(docs, Hh, t, fused=True)
    cu = np.concatenate([[0], np.cumsum(lens)])
    rows = sample_rows(cu, per_edge=24, interior=24, seed=56)
    _, o, lse, _ = oracle_reference(docs, t, rows=rows)
    check_attention(r.o[rows], o, r.lse[:, rows], lse, "56 heads, fused qkv, end to end")


def _bf16_round(x):
    """fp64 -> nearest-even bf16 values (as fp64), for crafted inputs."""
    return synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


@pytest.mark.parametrize("col", [20, 100])
def test_running_max_jump_rescales_o(lib, col):
    # Every query carries the same direction u; keys are small noise except one
    # key per head in key tile 3 whose score is ~9.5 log2-units above the rest,
    # so the running max grows by more than 2^8 in the middle of a unit (in the
    # first or second half of the tile's columns) and O and l must be rescaled.
    # About as much weight sits before the jump as after it.
    L, Hh = 700, 2
    rng = np.random.default_rng(col)
    u = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    q = _bf16_round(u[None, None, :] + 0.2 * rng.standard_normal((L, Hh, 128)))
    k = _bf16_round(0.05 * rng.standard_normal((L, Hh, 128)))
    jump = 3 * 128 + col
    k[jump, 0] = _bf16_round(0.58 * u)
    k[jump, 1] = _bf16_round(0.58 * u)
    v = _bf16_round(rng.standard_normal((L, Hh, 128)))
    scale = 1.0 / np.sqrt(128.0)
    dev = torch.device("cuda")
    to_dev = lambda x: torch.from_numpy(x.reshape(L, Hh * 128)).to(dev).to(torch.bfloat16)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full((L, Hh * 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((Hh, L), float("nan"), dtype=torch.float32, device=dev)
    with H.Plan(docs_1d([L]), Hh) as plan:
        H.h3attn_forward(plan.handle, qd, kd, vd, o, scale, lse)
        H.h3attn_get_device_error(plan.handle)
    o_gpu = o.double().cpu().numpy().reshape(L, Hh, 128)
    from oracle import attention as oatt
    o_ref, lse_ref = oatt.attention_rows(q, k, v, np.array([0, L]), scale, range(Hh), np.arange(L))
    # the inputs do what the test needs: the jump clears 2^8 for every row, and
    # the weight is split between the keys before it and the jump key
    s2 = np.einsum("ihd,jhd->hij", q, k) * scale / np.log(2.0)
    others = np.delete(s2, jump, axis=2)
    assert (s2[:, :, jump] - others.max(axis=2)).min() > 8.5
    w = np.exp2(s2 - s2.max(axis=2, keepdims=True))
    share = w[:, :, jump] / w.sum(axis=2)
    assert 0.2 < share.min() and share.max() < 0.8
    check_attention(o_gpu, o_ref, lse.cpu().numpy(), lse_ref, f"running max jump at column {col}")


@pytest.mark.parametrize("offset,pad", [(8, 0), (0, 8), (8, 8)])
def test_output_alignments_are_byte_identical(lib, offset, pad):
    # o starting 16 bytes past a 32-byte boundary and/or a row stride that is a
    # multiple of 8 but not of 16 elements: the same bytes from the epilogue's
    # TMA tile stores (warps whose rows all lie in their document) and from its
    # direct stores (warps at a document end), which take 16-byte stores
    # instead of 32-byte ones here.  Ragged documents and a split last wave
    # (units that write partial results) included.
    lens = [1000, 3, 513, 129, 1]
    Hh = 3
    S, W = sum(lens), Hh * 128
    t = random_tensors(S, Hh, seed=61)
    r0 = run_product(docs_1d(lens), Hh, t)
    dev = torch.device("cuda")
    with H.Plan(docs_1d(lens), Hh) as p:
        q, k, v = (bf16_to_torch(x).view(S, W) for x in (t.q, t.k, t.v))
        gq, gk = torch.from_numpy(t.gain_q).to(dev), torch.from_numpy(t.gain_k).to(dev)
        qh, kh = torch.empty_like(q), torch.empty_like(k)
        H.h3attn_qk_prologue(p.handle, q, k, qh, kh, gq, gk, 1e-6)
        stride = W + pad
        base = torch.zeros(S * stride + offset + 16, dtype=torch.bfloat16, device=dev)
        assert base.data_ptr() % 32 == 0
        o = base[offset:offset + S * stride].view(S, stride)[:, :W]
        H.h3attn_forward(p.handle, qh, kh, v, o, 1.0 / np.sqrt(128.0), None, o_row_stride=stride)
        H.h3attn_get_device_error(p.handle)
        got = o.contiguous().view(torch.int16).cpu().numpy().reshape(S, Hh, 128)
    assert np.array_equal(got, np.asarray(r0.o_bits).reshape(S, Hh, 128))
