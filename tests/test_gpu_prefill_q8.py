"""GPU parity of paged (chunked) prefill on 8-bit pools (FP8 E4M3 with
per-pool scales, INT8 with per-token-head scales): the quantising kv_append of
the chunks, then paged_attention_prefill through the C ABI, against the
oracle's fp64 prefill over the dequantised codes ("Part 3: single node",
random-liu.github.io, ch. 10: stored 8-bit, turned back into wider numbers
when read; ch. 13 sec. 1-2: a chunk's queries attend causally over the cached
prefix and the chunk).  The codes convert exactly, so the 16-bit attention
tolerance applies.  Cases span several 64-token KV tiles and 128-row query
tiles with ragged tails, every GQA group, block sizes 16-128, bf16 and f16
queries, decode requests mixed in."""

import numpy as np
import pytest
import torch

from oracle import c_oracle, np_oracle
from parity import ORACLE_THREADS, TORCH_DTYPE, _t, assert_q8_pools_equal, check_attention
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CACHES = [("fp8_e4m3", 1.0, 1.0), ("fp8_e4m3", 0.25, 3.0), ("int8", 1.0, 1.0)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _step(seed, prefix, chunks, *, dtype="bf16", hq=32, hkv=8, bs=16):
    return wl.chunked_prefill_step("q8 prefill", seed, prefix, chunks, dtype=dtype, num_q_heads=hq,
                                   num_kv_heads=hkv, head_dim=128, block_size=bs)


def _gpu(w, p, device="cuda"):
    tv = lambda a: wl.value_to_torch(a, w.dtype, device)
    kc, vc = _t(p.k_codes, device).clone(), _t(p.v_codes, device).clone()
    ks = None if p.k_scales is None else _t(p.k_scales, device).clone()
    vs = None if p.v_scales is None else _t(p.v_scales, device).clone()
    pool = pagedkv.KVPool(kc, vc, cache=p.cache, dtype=TORCH_DTYPE[w.dtype], k_scales=ks,
                          v_scales=vs, k_scale=p.k_scale, v_scale=p.v_scale)
    try:
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(device))
        q = tv(w.q)
        out = torch.zeros_like(q)
        cu = torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)).to(device)
        mq = int(np.diff(w.cu_seqlens).max())
        pool.prefill(q, cu, mq, torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device),
                     torch.from_numpy(w.seq_lens).to(device), w.scale, out=out)
        torch.cuda.synchronize()
        err = pool.get_error()
    finally:
        pool.close()
    host = lambda t: None if t is None else t.cpu().numpy()
    return host(kc), host(vc), host(ks), host(vs), wl.value_to_numpy(out, w.dtype), err


def _oracle(w, p):
    h = wl.on_host(w)
    host = lambda a: None if a is None else np.ascontiguousarray(
        a.cpu().numpy() if isinstance(a, torch.Tensor) else a).copy()
    kc, vc, ks, vs = host(p.k_codes), host(p.v_codes), host(p.k_scales), host(p.v_scales)
    c_oracle.append_q8(kc, vc, ks, vs, h.k_new, h.v_new, h.dtype, h.slot_mapping, p.cache,
                       p.k_scale, p.v_scale)
    out = np_oracle.prefill_q8(h.q, h.dtype, kc, vc, ks, vs, p.cache, h.cu_seqlens,
                               h.block_tables, h.seq_lens, h.scale, h.num_kv_heads,
                               fp8_k_scale=p.k_scale, fp8_v_scale=p.v_scale)
    return kc, vc, ks, vs, out


def _check(w, cache, sk=1.0, sv=1.0, seed=9, what=""):
    p = wl.q8_pools(w, cache, seed, sk, sv)
    gk, gv, gks, gvs, out, err = _gpu(w, p)
    rk, rv, rks, rvs, ref = _oracle(w, p)
    assert err == 0, f"{what}: device error bits {err:#x}"
    assert_q8_pools_equal((gk, gv, gks, gvs), (rk, rv, rks, rvs), what)
    return check_attention(out, ref, w.dtype, what)


@pytest.mark.parametrize("cache,sk,sv", CACHES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_q8_prefill_llama(cache, sk, sv, dtype):
    """Llama-3-8B-shaped GQA: chunks after cached prefixes (ragged KV tiles),
    a fresh prompt, decode requests."""
    w = _step(1, [0, 100, 300, 37, 0], [150, 1, 130, 200, 1], dtype=dtype)
    print(_check(w, cache, sk, sv, what=f"{cache} {dtype}"))


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("hq,hkv,bs", [(16, 16, 32), (16, 8, 64), (64, 8, 128), (8, 1, 16)])
def test_q8_prefill_groups_and_block_sizes(cache, hq, hkv, bs):
    w = _step(2, [70, 0, 260], [40, 129, 3], hq=hq, hkv=hkv, bs=bs)
    print(_check(w, cache, what=f"{cache} {hq}/{hkv} bs{bs}"))


def test_q8_prefill_int8_v_scales_zero_then_jump():
    """INT8 V scales zero over a request's first block and 100x larger on a
    later one: P is weighed by each token's own V scale."""
    w = _step(3, [200, 90], [60, 30])
    p = wl.q8_pools(w, "int8", 4)
    vs = np.array(p.v_scales.cpu().numpy() if isinstance(p.v_scales, torch.Tensor)
                  else p.v_scales, copy=True)
    bt = np.asarray(w.block_tables)
    vs[bt[0, 0]] = 0.0
    vs[bt[0, 5]] *= 100.0
    p.v_scales = vs
    gk, gv, gks, gvs, out, err = _gpu(w, p)
    rk, rv, rks, rvs, ref = _oracle(w, p)
    assert err == 0
    print(check_attention(out, ref, w.dtype, "int8 v scales"))
