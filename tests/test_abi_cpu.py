"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from packed_varlen_non_gb300 import h3attn as H

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "h3attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("h3attn_plan_create", "h3attn_qk_prologue", "h3attn_forward",
                     "h3attn_plan_destroy", "h3attn_get_device_error", "h3attn_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.library_path())
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(H, n), n


def _status(fn):
    with pytest.raises(H.H3AttnError) as e:
        fn()
    return e.value.status


GOOD_DOCS = [[(2, 4, 8, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]


def test_plan_create_rejects_bad_arguments_on_the_host(lib):
    assert _status(lambda: H.h3attn_plan_create([], 2, stream=False)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_plan_create(GOOD_DOCS, 0, stream=False)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_plan_create(GOOD_DOCS, 2, head_dim=64, stream=False)) == H.H3ATTN_EUNSUPPORTED
    assert _status(lambda: H.h3attn_plan_create(GOOD_DOCS, 2, rope_dims=64, stream=False)) == H.H3ATTN_EUNSUPPORTED
    assert _status(lambda: H.h3attn_plan_create(GOOD_DOCS, 2, rope_base=1.0, stream=False)) == H.H3ATTN_EINVAL
    empty_span = [[(0, 4, 8, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    assert _status(lambda: H.h3attn_plan_create(empty_span, 2, stream=False)) == H.H3ATTN_EINVAL
    no_spans = [GOOD_DOCS[0], []]
    assert _status(lambda: H.h3attn_plan_create(no_spans, 2, stream=False)) == H.H3ATTN_EINVAL
    nan_step = [[(2, 1, 1, (0.0, 0.0, 0.0), (float("nan"), 0.0, 0.0))]]
    assert _status(lambda: H.h3attn_plan_create(nan_step, 2, stream=False)) == H.H3ATTN_EINVAL
    huge = [[(1 << 20, 1 << 11, 1, (0.0, 0.0, 0.0), (1.0, 1.0, 1.0))]]
    assert _status(lambda: H.h3attn_plan_create(huge, 2, stream=False)) == H.H3ATTN_EINVAL
    assert "span" in H.h3attn_last_error() or "S" in H.h3attn_last_error() or H.h3attn_last_error()


def test_compute_calls_reject_a_null_plan(lib):
    assert _status(lambda: H.h3attn_forward(None, 16, 16, 16, 16, 0.1, qkv_row_stride=128,
                                            o_row_stride=128, stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_qk_prologue(None, 16, 16, 16, 16, 16, 16, 1e-6,
                                                in_row_stride=128, out_row_stride=128,
                                                stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_get_device_error(None, stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_plan_info(None)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_forward_fused_q(None, 16, 16, 16, 16, 16, 0.1, qkv_row_stride=128,
                                                    o_row_stride=128, stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_fp8_quantize(None, 16, 16, 16, 16, 16, 16, 16, 16, 16, qkv_row_stride=128,
                                                 stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_qk_prologue_fp8(None, 16, 16, 16, 16, 16, 1e-6, 16, 16, 16, 16, 16, 16,
                                                    qkv_row_stride=128, stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_forward_fp8(None, 16, 16, 16, 16, 16, 16, 16, 0.1, o_row_stride=128,
                                                stream=0)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_plan_fp8_v_keys(None)) == H.H3ATTN_EINVAL
    assert _status(lambda: H.h3attn_plan_forward_kernels(None)) == H.H3ATTN_EINVAL
    H.h3attn_plan_destroy(None)  # accepted and ignored


def test_selftest_rejects_out_of_range_limits(lib):
    assert H.h3attn_selftest_bounded_wait(10, stream=0) == H.H3ATTN_EINVAL
    assert H.h3attn_selftest_bounded_wait(10 ** 11, stream=0) == H.H3ATTN_EINVAL


def test_product_path_has_no_oracle_import():
    pkg = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "packed_varlen_non_gb300")
    for dirpath, _dirs, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
