"""fp64 CPU oracle for one chunked-prefill attention step over a paged KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library and never loads it.

Two independent oracles live here:

* ``attention`` / ``probs`` / ``kv_append`` / ``slot_mapping`` -- plain C in
  double precision (``cpa_oracle.c``), reading K/V through the block table
  exactly as the paged cache stores them.  Compiled with gcc on first use.
  Caches may also hold OCP FP8 E4M3 codes (``torch.uint8`` tensors) with a
  per-tensor scale; ``e4m3_encode`` / ``e4m3_decode`` / ``kv_append_e4m3``
  are that format's quantiser, its values and the append that quantises.
* ``dense.attention_dense`` -- a brute-force numpy/scipy version that never
  touches pages: it materialises each sequence's full [q_len, ctx] visibility
  mask and runs a dense softmax.  It is the second opinion used to pin the
  first on small inputs.

Parity status: pinned (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcpa_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F16, E4M3 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain C, no vector intrinsics)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_variant(src_text: str, out_path: str) -> ctypes.CDLL:
    """Compile an edited copy of the oracle source (used by the mutation tests,
    which plant a mistake in a copy and check that the pins catch it)."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    c_path, "-o", out_path, "-lm"], check=True)
    return _declare(ctypes.CDLL(out_path))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_attention.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, D, P,
                                     I64, P, I]
    lib.oracle_attention.restype = I
    F = ctypes.c_float
    lib.oracle_attention_kv.argtypes = [P, I, P, P, I, D, D, P, I, P, P, I, I, I, I, I, D,
                                        P, I64, P, I]
    lib.oracle_attention_kv.restype = I
    lib.oracle_e4m3_encode.argtypes = [P, I, I64, F, P]
    lib.oracle_e4m3_encode.restype = None
    lib.oracle_e4m3_decode.argtypes = [P, I64, P]
    lib.oracle_e4m3_decode.restype = None
    lib.oracle_f16_decode.argtypes = [P, I64, P]
    lib.oracle_f16_decode.restype = None
    lib.oracle_kv_append_e4m3.argtypes = [P, P, I, P, I64, I, I, I, F, F, P, P]
    lib.oracle_kv_append_e4m3.restype = None
    lib.oracle_probs.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, D, I64, I,
                                 P, P]
    lib.oracle_probs.restype = I64
    lib.oracle_kv_append.argtypes = [P, P, P, I64, I, I, I, I, P, P]
    lib.oracle_kv_append.restype = None
    lib.oracle_slot_mapping.argtypes = [P, I, P, P, I, I, P]
    lib.oracle_slot_mapping.restype = I
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.uint8:
        return E4M3  # a cache of OCP FP8 E4M3 codes
    raise TypeError(f"oracle supports fp32, bf16, fp16 and E4M3-code storage, got {t.dtype}")


def _cpu(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu").contiguous()


def attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
              rows=None, nthreads=None, impl=None, k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """fp64 attention output [len(rows), Hq, D] for the packed tokens ``rows``
    (all tokens when None).  Tensors may live on any device; they are read on
    the host.  ``q`` is [T, Hq, D]; caches are [num_pages, Hkv, page, D] and
    hold K / k_scale and V / v_scale (uint8 caches: E4M3 codes)."""
    L = impl or lib()
    q, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_table).to(torch.int32)
    qsl = _cpu(query_start_loc).to(torch.int32)
    sl = _cpu(seq_lens).to(torch.int32)
    T, Hq, D = q.shape
    _, Hkv, page, _ = kc.shape
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), Hq, D), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    if kc.dtype == q.dtype and k_scale == 1.0 and v_scale == 1.0:
        rc = L.oracle_attention(q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                _dtype_code(q), bt.data_ptr(), bt.shape[1],
                                qsl.data_ptr(), sl.data_ptr(), sl.shape[0], Hq, Hkv, D,
                                page, float(scale), rows.ctypes.data, len(rows),
                                out.ctypes.data, int(nthreads))
    else:
        assert vc.dtype == kc.dtype
        rc = L.oracle_attention_kv(q.data_ptr(), _dtype_code(q), kc.data_ptr(),
                                   vc.data_ptr(), _dtype_code(kc), float(k_scale),
                                   float(v_scale), bt.data_ptr(), bt.shape[1],
                                   qsl.data_ptr(), sl.data_ptr(), sl.shape[0], Hq, Hkv, D,
                                   page, float(scale), rows.ctypes.data, len(rows),
                                   out.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return out


def probs(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
          token: int, head: int, impl=None):
    """Softmax weights (over visible keys) and output of one (token, head)."""
    L = impl or lib()
    q, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_table).to(torch.int32)
    qsl = _cpu(query_start_loc).to(torch.int32)
    sl = _cpu(seq_lens).to(torch.int32)
    T, Hq, D = q.shape
    _, Hkv, page, _ = kc.shape
    p = np.zeros(int(sl.max()) + 1, dtype=np.float64)
    o = np.zeros(D, dtype=np.float64)
    n = L.oracle_probs(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), _dtype_code(q),
                       bt.data_ptr(), bt.shape[1], qsl.data_ptr(), sl.data_ptr(),
                       sl.shape[0], Hq, Hkv, D, page, float(scale), int(token),
                       int(head), p.ctypes.data, o.ctypes.data)
    if n < 0:
        raise ValueError(f"oracle_probs failed with status {n}")
    return p[:n], o


def kv_append(k_cache: torch.Tensor, v_cache: torch.Tensor, k: torch.Tensor,
              v: torch.Tensor, slot_mapping: torch.Tensor, impl=None) -> None:
    """In-place host scatter of new K/V rows into host caches (memcpy)."""
    L = impl or lib()
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous()
    assert v_cache.device.type == "cpu" and v_cache.is_contiguous()
    k, v = _cpu(k), _cpu(v)
    sm = _cpu(slot_mapping).to(torch.int64)
    T, Hkv, D = k.shape
    page = k_cache.shape[2]
    L.oracle_kv_append(k.data_ptr(), v.data_ptr(), sm.data_ptr(), T, Hkv, D, page,
                       k.element_size(), k_cache.data_ptr(), v_cache.data_ptr())


def slot_mapping(block_table, query_start_loc, seq_lens, page_size: int,
                 impl=None) -> torch.Tensor:
    """The oracle's own cache slot for every new token of the step."""
    L = impl or lib()
    bt = _cpu(block_table).to(torch.int32)
    qsl = _cpu(query_start_loc).to(torch.int32)
    sl = _cpu(seq_lens).to(torch.int32)
    out = torch.full((int(qsl[-1]),), -1, dtype=torch.int64)
    rc = L.oracle_slot_mapping(bt.data_ptr(), bt.shape[1], qsl.data_ptr(),
                               sl.data_ptr(), sl.shape[0], page_size, out.data_ptr())
    if rc != 0:
        raise ValueError("malformed metadata")
    return out


def e4m3_encode(x: torch.Tensor, scale: float = 1.0, impl=None) -> torch.Tensor:
    """OCP FP8 E4M3 codes (uint8, same shape) of x / scale, the quotient taken
    in binary32; round to nearest even, saturating at +-448."""
    L = impl or lib()
    x = _cpu(x)
    out = torch.empty(x.shape, dtype=torch.uint8)
    L.oracle_e4m3_encode(x.data_ptr(), _dtype_code(x), x.numel(), float(scale), out.data_ptr())
    return out


def e4m3_decode(codes: torch.Tensor, impl=None) -> np.ndarray:
    """Values (float64) of E4M3 codes."""
    L = impl or lib()
    c = _cpu(codes).to(torch.uint8)
    out = np.zeros(tuple(c.shape), dtype=np.float64)
    L.oracle_e4m3_decode(c.data_ptr(), c.numel(), out.ctypes.data)
    return out


def f16_decode(bits: torch.Tensor, impl=None) -> np.ndarray:
    """Values (float64) of IEEE binary16 bit patterns (int16/uint16 storage)."""
    L = impl or lib()
    b = _cpu(bits).view(torch.int16)
    out = np.zeros(tuple(b.shape), dtype=np.float64)
    L.oracle_f16_decode(b.data_ptr(), b.numel(), out.ctypes.data)
    return out


def kv_append_e4m3(k_cache: torch.Tensor, v_cache: torch.Tensor, k: torch.Tensor,
                   v: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                   v_scale: float, impl=None) -> None:
    """In-place host append into uint8 E4M3 caches: the codes of k / k_scale
    and v / v_scale at each token's slot."""
    L = impl or lib()
    assert k_cache.dtype == torch.uint8 and v_cache.dtype == torch.uint8
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous() and v_cache.is_contiguous()
    k, v = _cpu(k), _cpu(v)
    sm = _cpu(slot_mapping).to(torch.int64)
    T, Hkv, D = k.shape
    page = k_cache.shape[2]
    L.oracle_kv_append_e4m3(k.data_ptr(), v.data_ptr(), _dtype_code(k), sm.data_ptr(), T, Hkv,
                            D, page, float(k_scale), float(v_scale), k_cache.data_ptr(),
                            v_cache.data_ptr())
