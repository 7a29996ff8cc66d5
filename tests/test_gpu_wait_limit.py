"""GPU: the decode kernels' bounded waits give up, report and return.

Every pipeline wait of the decode kernels is bounded, so that a fault cannot
hang the GPU: on expiry the kernel sets KV_DEVERR_TIMEOUT, stops loading,
lets the copies already in flight land and returns.  Here the limit is set to
0 ns with valid inputs, so a wait that finds its tile not yet landed gives
up at once (at these sizes the kernels stream from HBM and many waits do);
nothing is broken on purpose and every copy completes.  The call must return, the stream synchronise, the timeout bit be
set; a normal call on the same pool afterwards must match the oracle."""

import numpy as np
import pytest
import torch

from parity import check_attention, oracle_step
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _inputs(w):
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone())
    pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev))
    pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
    q = tv(w.q)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    return pool, q, tables, lens


def _expire_then_recover(w, decode):
    _, _, ref = oracle_step(w)
    pool, q, tables, lens = _inputs(w)
    try:
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        pool.set_wait_limit(0)
        decode(pool, q, tables, lens)
        torch.cuda.synchronize()                      # the kernels returned
        bits = pool.get_error()
        assert bits & pagedkv.KV_DEVERR_TIMEOUT, f"no timeout reported ({bits:#x})"
        pool.clear_error()
        pool.set_wait_limit(2_000_000_000)
        out = decode(pool, q, tables, lens)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        return check_attention(wl.value_to_numpy(out, w.dtype), ref, w.dtype, "after recovery")
    finally:
        pool.close()


def test_plain_decode_wait_gives_up():
    w = wl.llama3_8b_gqa(41, batch=64, median=700, hi=3000)
    _expire_then_recover(w, lambda pool, q, t, l: pool.decode(q, t, l, w.scale))


def test_long_context_decode_wait_gives_up():
    w = wl.long_context(42, batch=2, lo=20000, hi=30000, block_size=16)
    _expire_then_recover(w, lambda pool, q, t, l: pool.decode(q, t, l, w.scale))


def test_cascade_decode_wait_gives_up():
    w = wl.shared_prefix(43, prompts=6, prompt_len=2000, n=4, max_divergent=200)
    groups = torch.from_numpy(np.ascontiguousarray(w.groups, dtype=np.int32)).to("cuda")
    _expire_then_recover(w, lambda pool, q, t, l: pool.decode_cascade(q, t, l, w.scale, groups))


def test_prefill_wait_gives_up():
    """The tensor-core prefill kernel (TMA producers, MMA issuers, softmax
    warps, TMEM): with the limit at 0 its roles give up, the MMA issuers still
    wait (with the full limit) for the products already issued before TMEM is
    freed, and the call returns with the timeout bit set; then a normal call
    matches the oracle."""
    from parity import oracle_prefill_step
    w = wl.chunked_prefill(44, batch=6, chunk=256, max_prefix=2000, decodes=4)
    _, _, ref, rows = oracle_prefill_step(w)
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone())
    try:
        q = tv(w.q)
        tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
        lens = torch.from_numpy(w.seq_lens).to(dev)
        cu = torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)).to(dev)
        mq = int(np.diff(w.cu_seqlens).max())
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        pool.set_wait_limit(0)
        pool.prefill(q, cu, mq, tables, lens, w.scale, out=torch.zeros_like(q))
        torch.cuda.synchronize()                      # the kernel returned
        bits = pool.get_error()
        assert bits & pagedkv.KV_DEVERR_TIMEOUT, f"no timeout reported ({bits:#x})"
        pool.clear_error()
        pool.set_wait_limit(2_000_000_000)
        out = pool.prefill(q, cu, mq, tables, lens, w.scale, out=torch.zeros_like(q))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        check_attention(wl.value_to_numpy(out, w.dtype)[rows], ref, w.dtype, "after recovery")
    finally:
        pool.close()
