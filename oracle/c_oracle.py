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
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (plain -O2, no fast-math) if it is missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
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
