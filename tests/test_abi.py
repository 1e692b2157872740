"""The C-ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
none of these calls reaches the device)."""
import ctypes
import glob
import os
import re

import pytest

from chunked_prefill_paged_cpa_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(cpa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return ops.load(build_if_missing=True)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("cpa_kv_append", "cpa_attention_forward", "cpa_workspace_bytes",
                     "cpa_status_string", "cpa_read_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _desc(**kw):
    d = ops.CpaDesc(32, 8, 128, 16, 1000, 64, ops.CPA_BF16, 10, None, 0)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert ops.cpa_status_string(code).startswith("CPA_")
    assert "unknown" in ops.cpa_status_string(7)


def test_workspace_bytes_host_arithmetic(lib):
    d = _desc()
    n1 = ops.cpa_workspace_bytes(d, 1)
    n256 = ops.cpa_workspace_bytes(d, 256)
    assert n1 >= 256 and n256 > n1 and n256 % 256 == 0
    assert ops.cpa_workspace_bytes(_desc(head_dim=96), 4) == 0
    assert ops.cpa_workspace_bytes(_desc(num_q_heads=30), 4) == 0


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, ops.CPA_ERR_UNSUPPORTED),
    ("page_size", 32, ops.CPA_ERR_UNSUPPORTED),
    ("num_q_heads", 12, ops.CPA_ERR_ARG),       # not a multiple of 8 kv heads
    ("num_q_heads", 8 * 16, ops.CPA_ERR_UNSUPPORTED),  # group of 16
    ("dtype", 5, ops.CPA_ERR_UNSUPPORTED),
    ("num_pages", 0, ops.CPA_ERR_ARG),
])
def test_bad_descriptor_rejected_before_launch(lib, field, value, code):
    d = _desc(**{field: value})
    P = ctypes.c_void_p(256)
    assert ops.cpa_kv_append(P, P, P, P, P, d, None) == code
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 2, 0.1, P, None, d) == code
    assert ops.cpa_append_attention_forward(P, P, P, P, P, P, P, P, P, 2, 0.1, P, None, d) == code


def test_fused_append_call_validates_both_halves(lib):
    d = _desc()
    P = ctypes.c_void_p(4096)
    fa = ops.cpa_append_attention_forward
    # the append's arguments
    assert fa(P, None, P, P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, P, None, P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, P, P, None, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, ctypes.c_void_p(4100), P, P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, P, P, ctypes.c_void_p(4100), P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    # the attention's arguments
    assert fa(P, P, P, P, P, P, None, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, P, P, P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_WORKSPACE
    d.workspace, d.workspace_bytes = 4096, 1 << 30
    assert fa(P, P, P, P, P, P, P, P, P, 2, -1.0, P, None, d) == ops.CPA_ERR_ARG
    assert fa(P, P, P, P, P, P, P, P, P, 11, 0.1, P, None, d) == ops.CPA_ERR_ARG
    # empty step
    assert fa(P, P, P, P, P, P, P, P, P, 0, 0.1, P, None, _desc(num_tokens=0)) == ops.CPA_OK


def test_null_and_misaligned_pointers_rejected(lib):
    d = _desc()
    P = ctypes.c_void_p(4096)
    assert ops.cpa_kv_append(None, P, P, P, P, d, None) == ops.CPA_ERR_ARG
    assert ops.cpa_kv_append(ctypes.c_void_p(4100), P, P, P, P, d, None) == ops.CPA_ERR_ARG
    assert ops.cpa_attention_forward(P, P, P, None, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_ARG
    # missing workspace
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_WORKSPACE
    # too small workspace
    d.workspace, d.workspace_bytes = 4096, 512
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 2, 0.1, P, None, d) == ops.CPA_ERR_WORKSPACE
    # bad scale and more sequences than tokens
    d.workspace_bytes = 1 << 30
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 2, -1.0, P, None, d) == ops.CPA_ERR_ARG
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 11, 0.1, P, None, d) == ops.CPA_ERR_ARG


def test_empty_step_is_a_no_op(lib):
    d = _desc(num_tokens=0)
    P = ctypes.c_void_p(4096)
    assert ops.cpa_kv_append(P, P, P, P, P, d, None) == ops.CPA_OK
    assert ops.cpa_attention_forward(P, P, P, P, P, P, 0, 0.1, P, None, d) == ops.CPA_OK


def test_noalloc_scratch_size_is_exported(lib):
    """The binding reads the no-alloc scratch size from the library; it must
    be the header's value."""
    text = open(os.path.join(ROOT, "include", "cpa.h")).read()
    m = re.search(r"#define CPA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m, "CPA_NOALLOC_SCRATCH_BYTES not found in cpa.h"
    assert ops.cpa_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_noalloc_rejects_bad_arguments_before_touching_the_device(lib):
    P = ctypes.c_void_p(4096)
    d = _desc()
    f = ops.cpa_attention_forward_noalloc
    assert f(P, P, P, P, P, P, -1, 0.1, P, None, d) == ops.CPA_ERR_ARG
    assert f(P, P, P, P, P, P, 2, 0.1, P, None, _desc(head_dim=96)) == ops.CPA_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, 2, 0.1, P, None, _desc(max_pages_per_seq=0)) == ops.CPA_ERR_ARG
    # far beyond the built-in scratch
    assert f(P, P, P, P, P, P, 4096, 0.1, P, None,
             _desc(num_tokens=4096, max_pages_per_seq=4096)) == ops.CPA_ERR_WORKSPACE
    assert load_status_null(lib) == ops.CPA_ERR_ARG


def load_status_null(lib):
    return lib.cpa_noalloc_read_device_status(None, None)


def test_cache_dtype_descriptions(lib):
    # binary16 activations take the same shapes as bf16
    assert ops.cpa_workspace_bytes(_desc(dtype=ops.CPA_F16), 8) == \
        ops.cpa_workspace_bytes(_desc(), 8)
    # an E4M3 cache: 16-bit activations only, positive finite scales
    e = dict(kv_dtype=ops.CPA_KV_E4M3, k_scale=0.5, v_scale=2.0)
    assert ops.cpa_workspace_bytes(_desc(**e, dtype=ops.CPA_F32), 8) == 0
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert ops.cpa_workspace_bytes(_desc(**dict(e, k_scale=ks, v_scale=vs)), 8) == 0
    assert ops.cpa_workspace_bytes(_desc(kv_dtype=5), 8) == 0
    # bf16 queries read by binary16 MMAs: room for their binary16 copy
    T, Hq, D = 10, 32, 128
    n_bf16 = ops.cpa_workspace_bytes(_desc(**e), 8)
    n_f16 = ops.cpa_workspace_bytes(_desc(**e, dtype=ops.CPA_F16), 8)
    assert n_f16 == ops.cpa_workspace_bytes(_desc(), 8)
    assert n_bf16 == n_f16 + -(-2 * T * Hq * D // 256) * 256


def test_e4m3_append_rejects_bad_scales_before_launch(lib):
    d = _desc(kv_dtype=ops.CPA_KV_E4M3, k_scale=-1.0, v_scale=1.0)
    buf = ctypes.c_void_p(0x1000)
    assert ops.cpa_kv_append(buf, buf, ctypes.c_void_p(0x2000), buf, buf, d, None) == ops.CPA_ERR_ARG
