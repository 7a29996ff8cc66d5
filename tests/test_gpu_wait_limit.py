"""GPU: the decode and prefill kernels' bounded waits give up, report and return.

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

from oracle import np_oracle
from parity import TORCH_DTYPE, _t, check_attention, oracle_step, oracle_step_q8
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


# -- 8-bit pools: the same form for the kernels with code rings and scales ------

def _q8_pool(w, p, dev):
    kc, vc = _t(p.k_codes, dev).clone(), _t(p.v_codes, dev).clone()
    ks = None if p.k_scales is None else _t(p.k_scales, dev).clone()
    vs = None if p.v_scales is None else _t(p.v_scales, dev).clone()
    return pagedkv.KVPool(kc, vc, cache=p.cache, dtype=TORCH_DTYPE[w.dtype], k_scales=ks,
                          v_scales=vs, k_scale=p.k_scale, v_scale=p.v_scale)


def _q8_expire_then_recover(w, cache, call, ref, rows=None):
    """Append the step's tokens (quantising), run `call(pool)` with the wait
    limit at 0 (timeout bit expected), then again with the full limit: the
    output (rows `rows`, or all) must match `ref`."""
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    p = wl.q8_pools(w, cache, 7)
    pool = _q8_pool(w, p, dev)
    try:
        if w.pairs is not None and len(w.pairs):
            pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev))
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        pool.set_wait_limit(0)
        call(pool)
        torch.cuda.synchronize()                      # the kernels returned
        bits = pool.get_error()
        assert bits & pagedkv.KV_DEVERR_TIMEOUT, f"no timeout reported ({bits:#x})"
        pool.clear_error()
        pool.set_wait_limit(2_000_000_000)
        out = call(pool)
        torch.cuda.synchronize()
        assert pool.get_error() == 0
        got = wl.value_to_numpy(out, w.dtype)
        return check_attention(got if rows is None else got[rows], ref(p), w.dtype,
                               f"{cache}: after recovery")
    finally:
        pool.close()


def _decode_args(w):
    dev = torch.device("cuda")
    q = wl.value_to_torch(w.q, w.dtype, dev)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    return q, tables, lens


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_decode_wait_gives_up(cache):
    """The 8-bit split kernel: code tiles by TMA, INT8 scales by bulk copy, all
    counted on the stages' barriers and drained after the give-up.  The full
    Llama-3-8B-shaped step: with INT8's three stages per warp a smaller step
    can find every tile landed by the time it is waited for."""
    w = wl.llama3_8b_gqa(45)
    q, tables, lens = _decode_args(w)
    _q8_expire_then_recover(w, cache, lambda pool: pool.decode(q, tables, lens, w.scale),
                            lambda p: oracle_step_q8(w, p)[4])


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_cascade_wait_gives_up(cache):
    """The 8-bit shared-prefix pass (a producer warp, attending warps that
    keep walking their pieces after the give-up, so the named barriers between
    them stay matched) and the split kernel behind it."""
    w = wl.shared_prefix(46, prompts=4, prompt_len=2000, n=4, max_divergent=200)
    q, tables, lens = _decode_args(w)
    groups = torch.from_numpy(np.ascontiguousarray(w.groups, dtype=np.int32)).to("cuda")
    _q8_expire_then_recover(w, cache,
                            lambda pool: pool.decode_cascade(q, tables, lens, w.scale, groups),
                            lambda p: oracle_step_q8(w, p)[4])


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_prefill_wait_gives_up(cache):
    """The 8-bit prefill: code rings, two converter warps per side (the helper
    waits on the same stages and the producer on the helper), the INT8 scale
    ring and the converted query tiles."""
    w = wl.chunked_prefill(47, batch=6, chunk=256, max_prefix=2000, decodes=4)
    dev = torch.device("cuda")
    q = wl.value_to_torch(w.q, w.dtype, dev)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)).to(dev)
    mq = int(np.diff(w.cu_seqlens).max())

    def ref(p):
        h = wl.on_host(w)
        host = lambda a: None if a is None else np.ascontiguousarray(
            a.cpu().numpy() if isinstance(a, torch.Tensor) else a).copy()
        kc, vc, ks, vs = host(p.k_codes), host(p.v_codes), host(p.k_scales), host(p.v_scales)
        from oracle import c_oracle
        c_oracle.append_q8(kc, vc, ks, vs, h.k_new, h.v_new, h.dtype, h.slot_mapping, p.cache,
                           p.k_scale, p.v_scale)
        return np_oracle.prefill_q8(h.q, h.dtype, kc, vc, ks, vs, p.cache, h.cu_seqlens,
                                    h.block_tables, h.seq_lens, h.scale, h.num_kv_heads,
                                    fp8_k_scale=p.k_scale, fp8_v_scale=p.v_scale)

    _q8_expire_then_recover(
        w, cache, lambda pool: pool.prefill(q, cu, mq, tables, lens, w.scale, out=torch.zeros_like(q)),
        ref)
