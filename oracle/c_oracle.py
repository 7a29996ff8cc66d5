"""ctypes front end for the plain-C fp64 oracle (TEST INFRASTRUCTURE ONLY).

``build()`` compiles ``pagedkv_oracle.c`` with gcc into ``oracle/_build``; the
functions below pass numpy buffers straight to it.  The C file is an
independent restatement of the definitions ``np_oracle`` follows; the tests
cross-check the two and pin both against closed forms and library routines.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpagedkv_oracle.so")
_DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
_FMT_CODE = {"fp8_e4m3": 3, "int8": 4}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (plain -O2, no fast-math) if it is missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, L, I, D = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double
            lib.oracle_decode_elem.argtypes = [P, ctypes.c_size_t, I]
            lib.oracle_decode_elem.restype = D
            lib.oracle_append.argtypes = [P, P, L, L, L, L, I, P, P, P, L]
            lib.oracle_append.restype = L
            lib.oracle_copy_blocks.argtypes = [P, P, L, L, L, L, I, P, L]
            lib.oracle_copy_blocks.restype = L
            lib.oracle_decode.argtypes = [P, P, P, I, L, L, L, L, P, L, P, L, L,
                                          D, P, I]
            lib.oracle_decode.restype = L
            F = ctypes.c_float
            lib.oracle_e4m3_decode.argtypes = [I]
            lib.oracle_e4m3_decode.restype = D
            lib.oracle_e4m3_encode.argtypes = [F]
            lib.oracle_e4m3_encode.restype = I
            lib.oracle_int8_quantize_row.argtypes = [P, L, P, P]
            lib.oracle_int8_quantize_row.restype = None
            lib.oracle_append_q8.argtypes = [P, P, P, P, L, L, L, L, I, I, P, P, P, L, F, F]
            lib.oracle_append_q8.restype = L
            lib.oracle_copy_blocks_q8.argtypes = [P, P, P, P, L, L, L, L, P, L]
            lib.oracle_copy_blocks_q8.restype = L
            lib.oracle_decode_q8.argtypes = [P, I, P, P, P, P, I, D, D, L, L, L, L, P, L, P, L, L,
                                             D, P, I]
            lib.oracle_decode_q8.restype = L
            lib.oracle_swap_blocks.argtypes = [P, P, P, I, L, L, P, L, I]
            lib.oracle_swap_blocks.restype = L
            lib.oracle_prefill.argtypes = [P, P, P, I, L, L, L, L, P, P, L, P, L, L, D, P, I]
            lib.oracle_prefill.restype = L
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data


def decode_elem(raw: np.ndarray, idx: int, dtype: str) -> float:
    return _load().oracle_decode_elem(_ptr(raw), idx, _DTYPE_CODE[dtype])


def append(k_pool, v_pool, k_new, v_new, slot_mapping, dtype: str) -> int:
    nb, bs, hkv, d = k_pool.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return _load().oracle_append(_ptr(k_pool), _ptr(v_pool), nb, bs, hkv, d,
                                 _DTYPE_CODE[dtype], _ptr(k_new), _ptr(v_new),
                                 _ptr(slots), slots.shape[0])


def copy_blocks(k_pool, v_pool, pairs, dtype: str) -> int:
    nb, bs, hkv, d = k_pool.shape
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return _load().oracle_copy_blocks(_ptr(k_pool), _ptr(v_pool), nb, bs, hkv, d,
                                      _DTYPE_CODE[dtype], _ptr(pr), pr.shape[0])


def decode(q, k_pool, v_pool, dtype: str, block_tables, seq_lens, scale: float,
           num_kv_heads: int, num_threads: int = 1, return_status: bool = False):
    """fp64 attention output [B, Hq, D]; see ``oracle_decode`` in the C file."""
    B, Hq, D = q.shape
    nb, bs, hkv, d = k_pool.shape
    assert hkv == num_kv_heads and d == D
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = _load().oracle_decode(_ptr(np.ascontiguousarray(q)), _ptr(k_pool),
                               _ptr(v_pool), _DTYPE_CODE[dtype], nb, bs, hkv, D,
                               _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
                               _ptr(sl), B, Hq, float(scale), _ptr(out),
                               int(num_threads))
    if st < 0:
        raise ValueError("oracle_decode rejected its arguments")
    return (out, st) if return_status else out


# ------------------------------------------------------- 8-bit KV cache --

def _optr(a):
    return None if a is None else _ptr(a)


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def e4m3_encode(t: float) -> int:
    return _load().oracle_e4m3_encode(float(t))


def int8_quantize_row(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.shape[0], dtype=np.int8)
    sc = np.zeros(1, dtype=np.float32)
    _load().oracle_int8_quantize_row(_ptr(x), x.shape[0], _ptr(codes), _ptr(sc))
    return codes, sc[0]


def append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, in_dtype: str,
              slot_mapping, fmt: str, fp8_k_scale: float = 1.0, fp8_v_scale: float = 1.0) -> int:
    nb, bs, hkv, d = k_codes.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    r = _load().oracle_append_q8(_ptr(k_codes), _ptr(v_codes), _optr(k_scales), _optr(v_scales),
                                 nb, bs, hkv, d, _FMT_CODE[fmt], _DTYPE_CODE[in_dtype],
                                 _ptr(np.ascontiguousarray(k_new)), _ptr(np.ascontiguousarray(v_new)),
                                 _ptr(slots), slots.shape[0], float(fp8_k_scale), float(fp8_v_scale))
    if r < 0:
        raise MemoryError("oracle_append_q8")
    return r


def copy_blocks_q8(k_codes, v_codes, k_scales, v_scales, pairs) -> int:
    nb, bs, hkv, d = k_codes.shape
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return _load().oracle_copy_blocks_q8(_ptr(k_codes), _ptr(v_codes), _optr(k_scales),
                                         _optr(v_scales), nb, bs, hkv, d, _ptr(pr), pr.shape[0])


def decode_q8(q, in_dtype: str, k_codes, v_codes, k_scales, v_scales, fmt: str, block_tables,
              seq_lens, scale: float, num_kv_heads: int, fp8_k_scale: float = 1.0,
              fp8_v_scale: float = 1.0, num_threads: int = 1, return_status: bool = False):
    """fp64 attention output [B, Hq, D] over an 8-bit pool (``oracle_decode_q8``)."""
    B, Hq, D = q.shape
    nb, bs, hkv, d = k_codes.shape
    assert hkv == num_kv_heads and d == D
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = _load().oracle_decode_q8(_ptr(np.ascontiguousarray(q)), _DTYPE_CODE[in_dtype],
                                  _ptr(k_codes), _ptr(v_codes), _optr(k_scales), _optr(v_scales),
                                  _FMT_CODE[fmt], float(fp8_k_scale), float(fp8_v_scale),
                                  nb, bs, hkv, D, _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
                                  _ptr(sl), B, Hq, float(scale), _ptr(out), int(num_threads))
    if st < 0:
        raise ValueError("oracle_decode_q8 rejected its arguments")
    return (out, st) if return_status else out


# ------------------------------------------------------- swap to host ----

def swap_blocks(gpu_arrays, host_arrays, pairs, direction: int) -> int:
    """See ``oracle_swap_blocks``: arrays share their leading (block) axis."""
    assert len(gpu_arrays) == len(host_arrays)
    n = len(gpu_arrays)
    for g, h in zip(gpu_arrays, host_arrays):
        assert g.shape[1:] == h.shape[1:] and g.dtype == h.dtype
        _ptr(g), _ptr(h)
    gp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in gpu_arrays])
    hp = (ctypes.c_void_p * n)(*[a.ctypes.data for a in host_arrays])
    bb = (ctypes.c_long * n)(*[a[0].nbytes if a.shape[0] else a.itemsize * int(np.prod(a.shape[1:]))
                               for a in gpu_arrays])
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return _load().oracle_swap_blocks(gp, hp, bb, n, gpu_arrays[0].shape[0], host_arrays[0].shape[0],
                                      _ptr(pr), pr.shape[0], int(direction))


# ------------------------------------------------- paged (chunked) prefill --

def prefill(q, k_pool, v_pool, dtype: str, cu_seqlens, block_tables, seq_lens, scale: float,
            num_kv_heads: int, num_threads: int = 1, return_status: bool = False):
    """fp64 out [T, Hq, D] (see ``oracle_prefill``)."""
    T, Hq, D = q.shape
    nb, bs, hkv, d = k_pool.shape
    assert hkv == num_kv_heads and d == D
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    st = _load().oracle_prefill(_ptr(np.ascontiguousarray(q)), _ptr(k_pool), _ptr(v_pool),
                                _DTYPE_CODE[dtype], nb, bs, hkv, D, _ptr(cu), _ptr(bt),
                                bt.shape[1], _ptr(sl), sl.shape[0], Hq, float(scale), _ptr(out),
                                int(num_threads))
    if st < 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return (out, st) if return_status else out
