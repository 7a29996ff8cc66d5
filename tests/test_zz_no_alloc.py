"""paged_attention_decode_noalloc (GPU): the decode entry point for callers
that cannot allocate device memory -- e.g. an engine that has reserved the
whole device for its KV pool and forbids allocation in the decode loop, or a
plug-in whose host framework owns the allocator.  It runs the same kernels
with the same work split as paged_attention_decode (which takes a
caller-allocated workspace), so on two calls in a row that share its built-in
scratch array its output must be bit-identical to that call's, and within
the parity tolerance of the oracle.  The scratch keeps what the last call
left there; a call after one of another shape must not be misled by it.  A
call whose need exceeds the array's fixed size is refused before anything is
enqueued.

Kept in a file that pytest collects last."""

import ctypes

import numpy as np
import pytest
import torch

from parity import check_attention, oracle_step
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20      # the built-in array's size, as the header states


def _noalloc_fn():
    fn = pagedkv.load().paged_attention_decode_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, I, P, I, I, F, I, P]
    fn.restype = I
    return fn


def _case(w):
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone())
    q = tv(w.q)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev))
    pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
    return pool, q, tables, lens


def _noalloc(fn, pool, q, tables, lens, w):
    out = torch.empty_like(q)
    st = fn(pool.handle, q.data_ptr(), out.data_ptr(), tables.data_ptr(), int(tables.shape[1]),
            lens.data_ptr(), w.batch, w.num_q_heads, float(w.scale), w.num_kv_heads,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pagedkv.KV_OK, pagedkv.load().kv_strerror(st)
    return out


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_matches_workspace_decode_on_two_calls():
    fn = _noalloc_fn()
    cases = [wl.llama3_8b_gqa(5, batch=48, median=400, hi=3000),
             wl.opt13b_mha(6, batch=6, lo=1, hi=900)]
    for i, w in enumerate(cases):                       # two calls in a row
        _, _, ref = oracle_step(w)
        pool, q, tables, lens = _case(w)
        try:
            want = pool.decode(q, tables, lens, w.scale)  # caller-allocated workspace
            got = _noalloc(fn, pool, q, tables, lens, w)
            torch.cuda.synchronize()
            assert pool.get_error() == 0
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
                f"call {i}: not bit-identical to paged_attention_decode"
            check_attention(wl.value_to_numpy(got, w.dtype), ref, w.dtype, f"call {i}")
        finally:
            pool.close()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_after_a_call_of_another_shape():
    """A larger batch leaves its claim counter and partials in the scratch,
    where the next, smaller call's sit."""
    fn = _noalloc_fn()
    big = wl.llama3_8b_gqa(34, batch=200, median=200, hi=1200)
    small = wl.llama3_8b_gqa(35, batch=40, median=300, hi=2000)
    _, _, ref = oracle_step(small)
    for rep in range(2):
        for w in (big, small):
            pool, q, tables, lens = _case(w)
            try:
                got = _noalloc(fn, pool, q, tables, lens, w)
                torch.cuda.synchronize()
                assert pool.get_error() == 0
                if w is small:
                    check_attention(wl.value_to_numpy(got, w.dtype), ref, w.dtype,
                                    f"after a larger call #{rep}")
            finally:
                pool.close()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_refuses_a_need_beyond_its_array():
    """1,024 KV heads x 4,096 sequences need more than the 32 MiB array (their
    piece counters alone take 64 MiB): KV_ENOWORKSPACE, before anything is
    read or enqueued, and the pool stays usable."""
    fn = _noalloc_fn()
    hkv, batch = 1024, 4096
    k = torch.zeros((1, 16, hkv, 128), dtype=torch.bfloat16, device="cuda")
    pool = pagedkv.KVPool(k, k.clone())
    try:
        need = pagedkv.paged_attention_workspace_size(pool.handle, batch, hkv)
        assert need > SCRATCH_BYTES, need
        small = torch.zeros(64, dtype=torch.int32, device="cuda")   # never read
        st = fn(pool.handle, small.data_ptr(), small.data_ptr(), small.data_ptr(), 1,
                small.data_ptr(), batch, hkv, 0.088, hkv,
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == pagedkv.KV_ENOWORKSPACE, pagedkv.load().kv_strerror(st)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
    finally:
        pool.close()
