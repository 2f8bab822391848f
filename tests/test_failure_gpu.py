"""Failure detection without a GPU fault: a bounded device wait runs out,
the kernel records the timeout and returns, the host reads ETIMEOUT, and the
context stays usable."""
import numpy as np
import pytest

from packed_varlen_non_gb300 import h3attn as H
from tests.gpu_cases import check_attention, docs_1d, oracle_reference, random_tensors, run_product

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(lib):
    st = H.h3attn_selftest_bounded_wait(2_000_000)  # 2 ms
    assert st == H.H3ATTN_ETIMEOUT, H.h3attn_last_error()
    # the GPU keeps working after the timeout
    docs = docs_1d([200])
    t = random_tensors(200, 2, seed=5)
    r = run_product(docs, 2, t)
    _, o, lse, _ = oracle_reference(docs, t, q_hat=r.q_hat, k_hat=r.k_hat)
    check_attention(r.o, o, r.lse, lse, "after timeout")
