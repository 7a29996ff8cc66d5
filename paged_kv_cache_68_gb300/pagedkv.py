"""Python binding of ``libpagedkv`` (the C ABI in ``include/pagedkv.h``).

Argument marshalling only: torch tensors are used for device memory and
streams, and every step of the hot path runs in the library's CUDA kernels.
There is no fallback: if the library cannot be built or loaded, or a call
fails, an exception is raised.

The module-level functions carry the C names (``kv_pool_create``,
``kv_pool_create_quantized``,
``kv_append``, ``copy_blocks``, ``kv_swap_blocks``, ``paged_attention_workspace_size``,
``paged_attention_decode``, ``paged_attention_cascade_workspace_size``,
``paged_attention_decode_cascade``, ``paged_attention_prefill``,
``paged_attention_decode_noalloc``,
``kv_pool_get_error``, ``kv_pool_clear_error``, ``kv_pool_destroy``);
``KVPool`` bundles them for convenience.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

KV_OK, KV_EINVAL, KV_EUNSUPPORTED, KV_ECUDA, KV_ERANGE, KV_ENOWORKSPACE = range(6)
KV_DEVERR_SLOT_RANGE = 0x1
KV_DEVERR_BLOCK_RANGE = 0x2
KV_DEVERR_PAIR_RANGE = 0x4
KV_DEVERR_SEQ_RANGE = 0x8
KV_DEVERR_TIMEOUT = 0x10
KV_DEVERR_GROUP_RANGE = 0x20
KV_DEVERR_QUERY_RANGE = 0x40

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
KV_FP8_E4M3, KV_INT8 = 3, 4
CACHE_CODE = {"fp8_e4m3": KV_FP8_E4M3, "int8": KV_INT8}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = load()
        msg = lib.kv_strerror(status).decode()
        cuda = lib.kv_last_cuda_error().decode()
        super().__init__(f"{what}: {msg}" + (f" ({cuda})" if status == KV_ECUDA and cuda else ""))
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load(build: bool = True) -> ctypes.CDLL:
    """Load ``libpagedkv.so`` (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build:
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"libpagedkv is not built ({_build.LIB_PATH} missing)")
        lib = ctypes.CDLL(_build.LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "kv_pool_create": ([I, I, I, I, I, P, P, ctypes.POINTER(P)], I),
            "kv_pool_create_quantized": ([I, I, I, I, I, I, P, P, P, P, F, F, ctypes.POINTER(P)], I),
            "kv_pool_destroy": ([P], I),
            "kv_append": ([P, P, P, P, I, P], I),
            "copy_blocks": ([P, P, I, P], I),
            "paged_attention_workspace_size": ([P, I, I, ctypes.POINTER(S)], I),
            "paged_attention_decode_launches": ([P, I, I, ctypes.POINTER(I)], I),
            "paged_attention_decode": ([P, P, P, P, I, P, I, I, F, I, P, S, P], I),
            "paged_attention_cascade_workspace_size": ([P, I, I, I, ctypes.POINTER(S)], I),
            "paged_attention_decode_cascade": ([P, P, P, P, I, P, I, I, F, I, P, P, P, I, P, S, P], I),
            "kv_swap_blocks": ([P, P, P, P, P, I, P, I, I, P], I),
            "paged_attention_prefill": ([P, P, P, P, I, I, P, I, P, I, I, F, I, P], I),
            "kv_pool_set_wait_limit": ([P, ctypes.c_ulonglong], I),
            "kv_pool_get_error": ([P, ctypes.POINTER(I)], I),
            "kv_pool_clear_error": ([P], I),
            "kv_strerror": ([I], ctypes.c_char_p),
            "kv_last_cuda_error": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = args, res
        _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != KV_OK:
        raise PagedKVError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


# -- the C entry points, by name -----------------------------------------------

def kv_pool_create(k_pool: torch.Tensor, v_pool: torch.Tensor) -> ctypes.c_void_p:
    """Describe pools [num_blocks, block_size, num_kv_heads, head_dim]."""
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or k_pool.dim() != 4:
        raise ValueError("k_pool and v_pool must be equal-shaped 4-D tensors")
    if k_pool.dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported pool dtype {k_pool.dtype}")
    n, bs, hkv, d = k_pool.shape
    h = ctypes.c_void_p()
    _check(load().kv_pool_create(n, bs, hkv, d, DTYPE_CODE[k_pool.dtype],
                                 _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), ctypes.byref(h)),
           "kv_pool_create")
    return h


def kv_pool_create_quantized(k_codes: torch.Tensor, v_codes: torch.Tensor, dtype, cache: str,
                             k_scales: Optional[torch.Tensor] = None,
                             v_scales: Optional[torch.Tensor] = None, k_scale: float = 1.0,
                             v_scale: float = 1.0) -> ctypes.c_void_p:
    """Describe an 8-bit pool: uint8 codes [num_blocks, block_size, num_kv_heads,
    head_dim]; ``cache`` "fp8_e4m3" (per-pool scales k_scale, v_scale) or
    "int8" (fp32 scales [num_blocks, num_kv_heads, block_size]); ``dtype`` the
    16-bit type of q, out and new K/V rows."""
    if k_codes.shape != v_codes.shape or k_codes.dim() != 4:
        raise ValueError("k_codes and v_codes must be equal-shaped 4-D tensors")
    if cache not in CACHE_CODE:
        raise ValueError(f"unknown cache format {cache!r}")
    n, bs, hkv, d = k_codes.shape
    ks = vs = None
    if cache == "int8":
        for t, name in ((k_scales, "k_scales"), (v_scales, "v_scales")):
            if t is None or tuple(t.shape) != (n, hkv, bs):
                raise ValueError(f"{name} must be [num_blocks, num_kv_heads, block_size]")
        ks, vs = _dev(k_scales, "k_scales", torch.float32), _dev(v_scales, "v_scales", torch.float32)
    h = ctypes.c_void_p()
    _check(load().kv_pool_create_quantized(
        n, bs, hkv, d, CACHE_CODE[cache], DTYPE_CODE[dtype], _dev(k_codes, "k_codes", torch.uint8),
        _dev(v_codes, "v_codes", torch.uint8), ks, vs, float(k_scale), float(v_scale),
        ctypes.byref(h)), "kv_pool_create_quantized")
    return h


def kv_pool_destroy(handle) -> None:
    _check(load().kv_pool_destroy(handle), "kv_pool_destroy")


def kv_append(handle, k_new, v_new, slot_mapping, dtype, stream=None) -> None:
    t = int(slot_mapping.shape[0])
    _check(load().kv_append(handle, _dev(k_new, "k_new", dtype), _dev(v_new, "v_new", dtype),
                            _dev(slot_mapping, "slot_mapping", torch.int64), t, _stream(stream)),
           "kv_append")


def copy_blocks(handle, pairs, stream=None) -> None:
    n = int(pairs.shape[0]) if pairs.numel() else 0
    ptr = _dev(pairs, "pairs", torch.int32) if n else None
    _check(load().copy_blocks(handle, ptr, n, _stream(stream)), "copy_blocks")


KV_SWAP_OUT, KV_SWAP_IN = 0, 1


def _host(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous pinned host tensor")
    return t.data_ptr()


def kv_swap_blocks(handle, host_k, host_v, pairs, direction: int, host_k_scales=None,
                   host_v_scales=None, stream=None) -> None:
    """Move whole blocks between the pool and pinned host pools of the same
    layout: pairs int32 [P, 2] = (pool block, host block), on the device."""
    n = int(pairs.shape[0]) if pairs.numel() else 0
    ptr = _dev(pairs, "pairs", torch.int32) if n else None
    hs = lambda t, nm: None if t is None else _host(t, nm)
    _check(load().kv_swap_blocks(handle, _host(host_k, "host_k"), _host(host_v, "host_v"),
                                 hs(host_k_scales, "host_k_scales"),
                                 hs(host_v_scales, "host_v_scales"), int(host_k.shape[0]), ptr, n,
                                 int(direction), _stream(stream)), "kv_swap_blocks")


def paged_attention_decode_launches(handle, batch: int, num_q_heads: int) -> int:
    out = ctypes.c_int()
    _check(load().paged_attention_decode_launches(handle, batch, num_q_heads, ctypes.byref(out)),
           "paged_attention_decode_launches")
    return int(out.value)


def paged_attention_workspace_size(handle, batch: int, num_q_heads: int) -> int:
    out = ctypes.c_size_t()
    _check(load().paged_attention_workspace_size(handle, batch, num_q_heads, ctypes.byref(out)),
           "paged_attention_workspace_size")
    return int(out.value)


def paged_attention_decode(handle, q, out, block_tables, seq_lens, scale: float,
                           num_kv_heads: int, workspace, dtype, stream=None) -> None:
    b, hq, _ = q.shape
    _check(load().paged_attention_decode(
        handle, _dev(q, "q", dtype), _dev(out, "out", dtype),
        _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), int(b), int(hq), float(scale), int(num_kv_heads),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "paged_attention_decode")


def paged_attention_cascade_workspace_size(handle, batch: int, num_q_heads: int,
                                           num_groups: int) -> int:
    out = ctypes.c_size_t()
    _check(load().paged_attention_cascade_workspace_size(handle, batch, num_q_heads, num_groups,
                                                         ctypes.byref(out)),
           "paged_attention_cascade_workspace_size")
    return int(out.value)


def paged_attention_decode_cascade(handle, q, out, block_tables, seq_lens, scale: float,
                                   num_kv_heads: int, group_first, group_size,
                                   group_shared_blocks, workspace, dtype, stream=None) -> None:
    b, hq, _ = q.shape
    k = int(group_first.numel())
    gp = lambda t, n: _dev(t, n, torch.int32) if k else None
    _check(load().paged_attention_decode_cascade(
        handle, _dev(q, "q", dtype), _dev(out, "out", dtype),
        _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), int(b), int(hq), float(scale), int(num_kv_heads),
        gp(group_first, "group_first"), gp(group_size, "group_size"),
        gp(group_shared_blocks, "group_shared_blocks"), k,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "paged_attention_decode_cascade")


def paged_attention_prefill(handle, q, out, cu_seqlens, max_query_len: int, block_tables,
                            seq_lens, scale: float, num_kv_heads: int, dtype,
                            stream=None) -> None:
    """q, out [T, Hq, D]; cu_seqlens int32 [B + 1]; seq_lens int32 [B]
    (context after the chunk's append); block_tables int32 [B, max_blocks]."""
    t, hq, _ = q.shape
    b = int(seq_lens.numel())
    _check(load().paged_attention_prefill(
        handle, _dev(q, "q", dtype), _dev(out, "out", dtype),
        _dev(cu_seqlens, "cu_seqlens", torch.int32), int(t), int(max_query_len),
        _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens", torch.int32), b, int(hq), float(scale), int(num_kv_heads),
        _stream(stream)), "paged_attention_prefill")


def kv_pool_set_wait_limit(handle, limit_ns: int) -> None:
    """Limit of one pipeline wait in the decode kernels (default and largest
    2 s; 0 makes every wait that is not already satisfied give up)."""
    _check(load().kv_pool_set_wait_limit(handle, int(limit_ns)), "kv_pool_set_wait_limit")


def kv_pool_get_error(handle) -> int:
    bits = ctypes.c_int()
    st = load().kv_pool_get_error(handle, ctypes.byref(bits))
    if st not in (KV_OK, KV_ERANGE):
        _check(st, "kv_pool_get_error")
    return int(bits.value)


def kv_pool_clear_error(handle) -> None:
    _check(load().kv_pool_clear_error(handle), "kv_pool_clear_error")


# -- convenience wrapper ------------------------------------------------------------

class KVPool:
    """A KV block pool (two caller-owned tensors) plus its library handle."""

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, *, cache: Optional[str] = None,
                 dtype=None, k_scales: Optional[torch.Tensor] = None,
                 v_scales: Optional[torch.Tensor] = None, k_scale: float = 1.0,
                 v_scale: float = 1.0):
        """A 16-bit or fp32 pool (k_pool, v_pool of that type), or with
        ``cache`` set an 8-bit pool: uint8 codes, ``dtype`` the 16-bit type of
        q / out / new rows, and the scales ``kv_pool_create_quantized`` takes."""
        self.k_pool, self.v_pool = k_pool, v_pool
        self.cache = cache
        self.k_scales, self.v_scales = k_scales, v_scales
        self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim = k_pool.shape
        if cache is None:
            self.dtype = k_pool.dtype
            self.handle = kv_pool_create(k_pool, v_pool)
        else:
            self.dtype = dtype
            self.handle = kv_pool_create_quantized(k_pool, v_pool, dtype, cache, k_scales,
                                                   v_scales, k_scale, v_scale)
        self._ws: Optional[torch.Tensor] = None

    def close(self) -> None:
        if self.handle is not None:
            kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, k_new, v_new, slot_mapping, stream=None) -> None:
        kv_append(self.handle, k_new, v_new, slot_mapping, self.dtype, stream)

    def copy_blocks(self, pairs, stream=None) -> None:
        copy_blocks(self.handle, pairs, stream)

    def host_pool(self, num_host_blocks: int):
        """Pinned host arrays of this pool's layout for swapped-out blocks:
        (k, v, k_scales, v_scales); the scales are None unless INT8."""
        shape = (num_host_blocks, self.block_size, self.num_kv_heads, self.head_dim)
        k = torch.empty(shape, dtype=self.k_pool.dtype, pin_memory=True)
        v = torch.empty(shape, dtype=self.k_pool.dtype, pin_memory=True)
        ks = vs = None
        if self.cache == "int8":
            sshape = (num_host_blocks, self.num_kv_heads, self.block_size)
            ks = torch.empty(sshape, dtype=torch.float32, pin_memory=True)
            vs = torch.empty(sshape, dtype=torch.float32, pin_memory=True)
        return k, v, ks, vs

    def swap_out(self, host, pairs, stream=None) -> None:
        """host = host_pool(...); pairs (pool block, host block) on the device."""
        kv_swap_blocks(self.handle, host[0], host[1], pairs, KV_SWAP_OUT, host[2], host[3], stream)

    def swap_in(self, host, pairs, stream=None) -> None:
        kv_swap_blocks(self.handle, host[0], host[1], pairs, KV_SWAP_IN, host[2], host[3], stream)

    def workspace(self, batch: int, num_q_heads: int) -> torch.Tensor:
        """A cached device workspace large enough for (batch, num_q_heads)."""
        need = paged_attention_workspace_size(self.handle, batch, num_q_heads)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.k_pool.device)
        return self._ws

    def decode(self, q, block_tables, seq_lens, scale: float, out=None, workspace=None,
               stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        if workspace is None:
            workspace = self.workspace(q.shape[0], q.shape[1])
        paged_attention_decode(self.handle, q, out, block_tables, seq_lens, scale,
                               self.num_kv_heads, workspace, self.dtype, stream)
        return out

    def decode_cascade(self, q, block_tables, seq_lens, scale: float, groups, out=None,
                       workspace=None, stream=None) -> torch.Tensor:
        """Decode with shared-prefix groups: ``groups`` int32 [K, 3] on the
        device, rows (first member, members, shared leading blocks)."""
        if out is None:
            out = torch.empty_like(q)
        groups = groups.reshape(-1, 3)
        k = int(groups.shape[0])
        if workspace is None:
            need = paged_attention_cascade_workspace_size(self.handle, q.shape[0], q.shape[1], k)
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(need, dtype=torch.uint8, device=self.k_pool.device)
            workspace = self._ws
        cols = [groups[:, i].contiguous() for i in range(3)]
        paged_attention_decode_cascade(self.handle, q, out, block_tables, seq_lens, scale,
                                       self.num_kv_heads, cols[0], cols[1], cols[2], workspace,
                                       self.dtype, stream)
        return out

    def prefill(self, q, cu_seqlens, max_query_len: int, block_tables, seq_lens, scale: float,
                out=None, stream=None) -> torch.Tensor:
        """Chunked prefill attention of the flattened queries ``q`` [T, Hq, D]."""
        if out is None:
            out = torch.empty_like(q)
        paged_attention_prefill(self.handle, q, out, cu_seqlens, max_query_len, block_tables,
                                seq_lens, scale, self.num_kv_heads, self.dtype, stream)
        return out

    def set_wait_limit(self, limit_ns: int) -> None:
        kv_pool_set_wait_limit(self.handle, limit_ns)

    def get_error(self) -> int:
        return kv_pool_get_error(self.handle)

    def clear_error(self) -> None:
        kv_pool_clear_error(self.handle)


def paged_attention_decode_noalloc(handle, q, out, block_tables, seq_lens, scale: float,
                                   num_kv_heads: int, dtype, stream=None) -> None:
    """Decode without a workspace argument, for callers that cannot allocate
    device memory (an engine that reserved the device for its KV pool, a
    plug-in whose host framework owns the allocator): the library's built-in
    32 MiB scratch array is used.  Calls that overlap on the GPU race on that
    array; the first call on a device should precede any stream capture."""
    fn = load().paged_attention_decode_noalloc
    if fn.restype is not ctypes.c_int:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [P, P, P, P, I, P, I, I, F, I, P]
        fn.restype = I
    b, hq, _ = q.shape
    _check(fn(handle, _dev(q, "q", dtype), _dev(out, "out", dtype),
              _dev(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
              _dev(seq_lens, "seq_lens", torch.int32), int(b), int(hq), float(scale),
              int(num_kv_heads), _stream(stream)), "paged_attention_decode_noalloc")
