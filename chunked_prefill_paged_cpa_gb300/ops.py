"""Thin Python binding of libcpa (include/cpa.h): argument marshalling only.

The ``cpa_*`` functions mirror the C entry points one to one and return the
C status code.  ``kv_append`` / ``attention_forward`` are conveniences that
build the descriptor from torch tensors, call the C entry point on torch's
current stream and raise on a non-zero status.  Every step of the computation
runs in the library's CUDA kernels; there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

CPA_OK, CPA_ERR_ARG, CPA_ERR_UNSUPPORTED, CPA_ERR_WORKSPACE, CPA_ERR_CUDA, CPA_ERR_DEVICE = (
    0, -1, -2, -3, -4, -5)
CPA_F32, CPA_BF16, CPA_F16 = 0, 1, 2
CPA_KV_SAME, CPA_KV_E4M3 = 0, 1

_lock = threading.Lock()
_lib = None


class CpaDesc(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("max_pages_per_seq", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("num_tokens", ctypes.c_int64),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


class CpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {cpa_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libcpa.so.  Raises if it is not built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"libcpa.so not built ({path}); run __graft_entry__.build() or "
                    "python -m chunked_prefill_paged_cpa_gb300.build")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I32, F, Z = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        D = ctypes.POINTER(CpaDesc)
        lib.cpa_status_string.argtypes = [ctypes.c_int]
        lib.cpa_status_string.restype = ctypes.c_char_p
        lib.cpa_workspace_bytes.argtypes = [D, I32]
        lib.cpa_workspace_bytes.restype = Z
        lib.cpa_kv_append.argtypes = [P, P, P, P, P, D, P]
        lib.cpa_kv_append.restype = ctypes.c_int
        lib.cpa_attention_forward.argtypes = [P, P, P, P, P, P, I32, F, P, P, D]
        lib.cpa_attention_forward.restype = ctypes.c_int
        lib.cpa_append_attention_forward.argtypes = [P, P, P, P, P, P, P, P, P, I32, F, P, P, D]
        lib.cpa_append_attention_forward.restype = ctypes.c_int
        lib.cpa_attention_forward_noalloc.argtypes = [P, P, P, P, P, P, I32, F, P, P, D]
        lib.cpa_attention_forward_noalloc.restype = ctypes.c_int
        lib.cpa_read_device_status.argtypes = [D, P, ctypes.POINTER(I32)]
        lib.cpa_read_device_status.restype = ctypes.c_int
        lib.cpa_noalloc_scratch_bytes.argtypes = []
        lib.cpa_noalloc_scratch_bytes.restype = Z
        lib.cpa_noalloc_read_device_status.argtypes = [P, ctypes.POINTER(I32)]
        lib.cpa_noalloc_read_device_status.restype = ctypes.c_int
        _lib = lib
        return lib


# ---- one-to-one mirrors of the C ABI -------------------------------------

def cpa_status_string(status: int) -> str:
    return load().cpa_status_string(int(status)).decode()


def cpa_workspace_bytes(desc: CpaDesc, num_seqs: int) -> int:
    return int(load().cpa_workspace_bytes(ctypes.byref(desc), int(num_seqs)))


def cpa_kv_append(k, v, slot_mapping, k_cache, v_cache, desc: CpaDesc, stream) -> int:
    return int(load().cpa_kv_append(k, v, slot_mapping, k_cache, v_cache,
                                    ctypes.byref(desc), stream))


def cpa_attention_forward(q, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                          num_seqs, scale, out, stream, desc: CpaDesc) -> int:
    return int(load().cpa_attention_forward(q, k_cache, v_cache, block_table,
                                            query_start_loc, seq_lens, int(num_seqs),
                                            float(scale), out, stream, ctypes.byref(desc)))


def cpa_append_attention_forward(q, k, v, slot_mapping, k_cache, v_cache, block_table,
                                 query_start_loc, seq_lens, num_seqs, scale, out, stream,
                                 desc: CpaDesc) -> int:
    return int(load().cpa_append_attention_forward(q, k, v, slot_mapping, k_cache, v_cache,
                                                   block_table, query_start_loc, seq_lens,
                                                   int(num_seqs), float(scale), out, stream,
                                                   ctypes.byref(desc)))


def cpa_attention_forward_noalloc(q, k_cache, v_cache, block_table, query_start_loc,
                                  seq_lens, num_seqs, scale, out, stream,
                                  desc: CpaDesc) -> int:
    """Mirror of the C entry point for callers that cannot allocate device
    memory: the scratch is a fixed array inside the library and
    desc.workspace is ignored."""
    return int(load().cpa_attention_forward_noalloc(q, k_cache, v_cache, block_table,
                                                    query_start_loc, seq_lens, int(num_seqs),
                                                    float(scale), out, stream,
                                                    ctypes.byref(desc)))


def cpa_noalloc_scratch_bytes() -> int:
    """Size of the no-alloc entry point's built-in scratch array, as the
    library was compiled."""
    return int(load().cpa_noalloc_scratch_bytes())


def cpa_noalloc_read_device_status(stream) -> int:
    """Read and clear the status word of the no-alloc scratch array (waits
    for ``stream``); CPA_OK or CPA_ERR_DEVICE."""
    st = ctypes.c_int32(0)
    rc = load().cpa_noalloc_read_device_status(stream, ctypes.byref(st))
    if rc != CPA_OK:
        raise CpaError(rc, "cpa_noalloc_read_device_status")
    return int(st.value)


def cpa_read_device_status(desc: CpaDesc, stream) -> int:
    st = ctypes.c_int32(0)
    rc = load().cpa_read_device_status(ctypes.byref(desc), stream, ctypes.byref(st))
    if rc != CPA_OK:
        raise CpaError(rc, "cpa_read_device_status")
    return int(st.value)


# ---- torch conveniences ---------------------------------------------------

def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return CPA_BF16
    if dtype == torch.float32:
        return CPA_F32
    if dtype == torch.float16:
        return CPA_F16
    raise TypeError(f"unsupported dtype {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_desc(k_cache: torch.Tensor, num_q_heads: int, num_tokens: int,
              max_pages_per_seq: int, workspace: torch.Tensor | None = None,
              act_dtype: torch.dtype | None = None, k_scale: float = 1.0,
              v_scale: float = 1.0) -> CpaDesc:
    """Descriptor for a cache tensor: a uint8 cache holds E4M3 codes (its
    activations then have ``act_dtype``, bf16 by default, and the codes the
    per-tensor scales); any other cache holds the activation dtype."""
    num_pages, Hkv, page, D = k_cache.shape
    e4m3 = k_cache.dtype == torch.uint8
    dt = (act_dtype or torch.bfloat16) if e4m3 else k_cache.dtype
    return CpaDesc(int(num_q_heads), int(Hkv), int(D), int(page), int(num_pages),
                   int(max_pages_per_seq), _dtype_code(dt), int(num_tokens),
                   None if workspace is None else workspace.data_ptr(),
                   0 if workspace is None else workspace.numel() * workspace.element_size(),
                   CPA_KV_E4M3 if e4m3 else CPA_KV_SAME,
                   float(k_scale) if e4m3 else 0.0, float(v_scale) if e4m3 else 0.0)


def workspace_for(k_cache: torch.Tensor, num_q_heads: int, max_pages_per_seq: int,
                  num_seqs: int, num_tokens: int,
                  act_dtype: torch.dtype | None = None) -> torch.Tensor:
    """A zero-filled device workspace sized by cpa_workspace_bytes for steps of
    at most ``num_seqs`` sequences and ``num_tokens`` packed tokens on the
    current device (``act_dtype``: the queries' dtype for a uint8 E4M3 cache)."""
    desc = make_desc(k_cache, num_q_heads, num_tokens, max_pages_per_seq, act_dtype=act_dtype)
    n = cpa_workspace_bytes(desc, num_seqs)
    if n == 0:
        raise CpaError(CPA_ERR_ARG, "cpa_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=k_cache.device)


def kv_append(k, v, slot_mapping, k_cache, v_cache, workspace=None, stream=None,
              k_scale=1.0, v_scale=1.0) -> None:
    desc = make_desc(k_cache, 1, k.shape[0], 1, workspace, k.dtype, k_scale, v_scale)
    desc.num_q_heads = desc.num_kv_heads
    rc = cpa_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                       desc, _stream(stream))
    if rc != CPA_OK:
        raise CpaError(rc, "cpa_kv_append")


def attention_forward(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
                      workspace, out=None, stream=None, k_scale=1.0, v_scale=1.0) -> torch.Tensor:
    if out is None:
        out = torch.empty_like(q)
    desc = make_desc(k_cache, q.shape[1], q.shape[0], block_table.shape[1], workspace,
                     q.dtype, k_scale, v_scale)
    rc = cpa_attention_forward(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                               _ptr(query_start_loc), _ptr(seq_lens), seq_lens.shape[0],
                               scale, _ptr(out), _stream(stream), desc)
    if rc != CPA_OK:
        raise CpaError(rc, "cpa_attention_forward")
    return out


def append_attention_forward(q, k, v, slot_mapping, k_cache, v_cache, block_table,
                             query_start_loc, seq_lens, scale, workspace, out=None,
                             stream=None, k_scale=1.0, v_scale=1.0) -> torch.Tensor:
    """kv_append followed by attention_forward, as one C-ABI call (the append
    fused into the attention kernels where they take the shape)."""
    if out is None:
        out = torch.empty_like(q)
    desc = make_desc(k_cache, q.shape[1], q.shape[0], block_table.shape[1], workspace,
                     q.dtype, k_scale, v_scale)
    rc = cpa_append_attention_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                      _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                      _ptr(query_start_loc), _ptr(seq_lens), seq_lens.shape[0],
                                      scale, _ptr(out), _stream(stream), desc)
    if rc != CPA_OK:
        raise CpaError(rc, "cpa_append_attention_forward")
    return out


def device_status(k_cache, num_q_heads, max_pages_per_seq, workspace, stream=None) -> int:
    desc = make_desc(k_cache, num_q_heads, 0, max_pages_per_seq, workspace)
    return cpa_read_device_status(desc, _stream(stream))
