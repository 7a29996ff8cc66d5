"""paged_attention_decode_noalloc (GPU): the decode entry point for callers
that cannot allocate device memory -- e.g. an engine that has reserved the
whole device for its KV pool and forbids allocation in the decode loop, or a
plug-in whose host framework owns the allocator.  It must give the output of
paged_attention_decode (which takes a caller-allocated workspace) within the
tolerance of the parity tests, on two calls in a row that share its built-in
scratch array.

Kept in a file that pytest collects last."""

import ctypes

import numpy as np
import pytest
import torch

from parity import check_attention
from oracle import np_oracle
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


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
    pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
    return pool, q, tables, lens


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_matches_workspace_decode_on_two_calls():
    fn = _noalloc_fn()
    cases = [wl.llama3_8b_gqa(5, batch=48, median=400, hi=3000),
             wl.opt13b_mha(6, batch=6, lo=1, hi=900)]
    for i, w in enumerate(cases):                       # two calls in a row
        pool, q, tables, lens = _case(w)
        try:
            ref = pool.decode(q, tables, lens, w.scale)  # caller-allocated workspace
            out = torch.empty_like(q)
            st = fn(pool.handle, q.data_ptr(), out.data_ptr(), tables.data_ptr(),
                    int(tables.shape[1]), lens.data_ptr(), w.batch, w.num_q_heads,
                    float(w.scale), w.num_kv_heads,
                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == pagedkv.KV_OK, pagedkv.load().kv_strerror(st)
            torch.cuda.synchronize()
            assert pool.get_error() == 0
            ref_raw = wl.value_to_numpy(ref, w.dtype)
            got_raw = wl.value_to_numpy(out, w.dtype)
            check_attention(got_raw, np_oracle.to_f64(ref_raw, w.dtype), w.dtype, f"call {i}")
        finally:
            pool.close()
