"""Shared helpers for the GPU parity tests: run one decode step through the
C ABI, run the same step through the CPU oracle, compare.

Tolerances (spec bar, written here once):
  * append / copy: the whole K and V pools must match the oracle byte for byte;
  * attention, fp32: max |gpu - oracle| <= 1e-5;
  * attention, fp16 / bf16: max |gpu - oracle| <= 2e-3 per element and
    max |gpu - oracle| / max |oracle| <= 1e-2.  A bf16 output with
    |oracle| >= 1 cannot meet 2e-3 (half a bf16 ulp there is 3.9e-3), so such
    elements must instead lie within one bf16 ulp of the oracle; they are
    counted and reported.
"""

from __future__ import annotations

import os

import numpy as np
import torch

from oracle import c_oracle, np_oracle
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ORACLE_THREADS = max(1, (os.cpu_count() or 2) - 1)


def gpu_step(w: wl.Workload, device="cuda", return_pools=True):
    """copy_blocks -> kv_append -> paged_attention_decode through the C ABI.

    Returns (k_pool, v_pool, out, error_bits); pools/out as raw host arrays.
    """
    tv = lambda a: wl.value_to_torch(a, w.dtype, device)
    k, v = tv(w.k_pool).clone(), tv(w.v_pool).clone()
    q, kn, vn = tv(w.q), tv(w.k_new), tv(w.v_new)
    slots = torch.from_numpy(w.slot_mapping).to(device)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device)
    lens = torch.from_numpy(w.seq_lens).to(device)
    pairs = torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(device)
    pool = pagedkv.KVPool(k, v)
    try:
        pool.copy_blocks(pairs)
        pool.append(kn, vn, slots)
        out = pool.decode(q, tables, lens, w.scale)
        torch.cuda.synchronize()
        err = pool.get_error()
    finally:
        pool.close()
    res_out = wl.value_to_numpy(out, w.dtype)
    if not return_pools:
        return None, None, res_out, err
    return wl.value_to_numpy(k, w.dtype), wl.value_to_numpy(v, w.dtype), res_out, err


def oracle_step(w: wl.Workload, seqs=None):
    """The same step on the CPU oracle; attention only for `seqs` if given."""
    h = wl.on_host(w)
    k, v = h.k_pool.copy(), h.v_pool.copy()
    assert c_oracle.copy_blocks(k, v, h.pairs, h.dtype) == 0
    assert c_oracle.append(k, v, h.k_new, h.v_new, h.slot_mapping, h.dtype) == 0
    sel = np.arange(h.batch) if seqs is None else np.asarray(seqs)
    out = c_oracle.decode(np.ascontiguousarray(h.q[sel]), k, v, h.dtype,
                          np.ascontiguousarray(h.block_tables[sel]),
                          np.ascontiguousarray(h.seq_lens[sel]), h.scale, h.num_kv_heads,
                          num_threads=ORACLE_THREADS)
    return k, v, out


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - 7)


def check_same_attention(a_raw: np.ndarray, b_raw: np.ndarray, dtype: str, what: str = ""):
    """Two device results of the same attention (e.g. cascade and plain
    decode), each within the tolerance of the exact value: they may differ by
    twice the per-element bound -- 2e-3 each below |out| = 1, and for bf16
    outputs of |out| >= 1 one ulp each (both are rounded once to bf16)."""
    a, b = np_oracle.to_f64(a_raw, dtype), np_oracle.to_f64(b_raw, dtype)
    lim = np.full(a.shape, 4e-3)
    if dtype == "bf16":
        big = np.maximum(np.abs(a), np.abs(b)) >= 1.0
        lim[big] = np.maximum(lim[big], 2.0 * bf16_ulp(np.maximum(np.abs(a), np.abs(b))[big]))
    diff = np.abs(a - b)
    assert (diff <= lim).all(), f"{what}: results differ by {diff.max():.3e}"
    return float(diff.max())


def check_attention(out_raw: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    got = np_oracle.to_f64(out_raw, dtype)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if dtype == "f32":
        assert err.max() <= 1e-5, f"{what}: max abs err {err.max():.3e} > 1e-5"
        return {"max_abs": float(err.max()), "exempt": 0}
    scale = max(float(np.abs(ref).max()), 1e-30)
    rel = float(err.max()) / scale
    assert rel <= 1e-2, f"{what}: max rel err {rel:.3e} > 1e-2"
    exempt = (np.abs(ref) >= 1.0) if dtype == "bf16" else np.zeros_like(ref, dtype=bool)
    bad = (err > 2e-3) & ~exempt
    assert not bad.any(), f"{what}: {int(bad.sum())} elements over 2e-3 (max {err[~exempt].max():.3e})"
    if exempt.any():
        assert (err[exempt] <= bf16_ulp(ref[exempt])).all(), f"{what}: |out|>=1 element beyond 1 ulp"
    return {"max_abs": float(err.max()), "max_rel": rel, "exempt": int(exempt.sum())}


def assert_pools_equal(got_k, got_v, ref_k, ref_v, what=""):
    assert got_k.shape == ref_k.shape
    assert got_k.tobytes() == ref_k.tobytes(), f"{what}: K pool differs from the oracle"
    assert got_v.tobytes() == ref_v.tobytes(), f"{what}: V pool differs from the oracle"


# -- 8-bit pools -------------------------------------------------------------------

def _t(a, device):
    return a.to(device) if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a)).to(device)


def gpu_step_q8(w: wl.Workload, p: wl.Q8Pools, device="cuda", return_pools=True, groups=None):
    """copy_blocks -> kv_append (quantising) -> decode on an 8-bit pool (cascade
    decode over `groups` [first, size, shared blocks] rows when given).
    Returns (k_codes, v_codes, k_scales, v_scales, out, error_bits) on the host."""
    tv = lambda a: wl.value_to_torch(a, w.dtype, device)
    kc, vc = _t(p.k_codes, device).clone(), _t(p.v_codes, device).clone()
    ks = None if p.k_scales is None else _t(p.k_scales, device).clone()
    vs = None if p.v_scales is None else _t(p.v_scales, device).clone()
    pool = pagedkv.KVPool(kc, vc, cache=p.cache, dtype=TORCH_DTYPE[w.dtype], k_scales=ks,
                          v_scales=vs, k_scale=p.k_scale, v_scale=p.v_scale)
    try:
        pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(device))
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(device))
        tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device)
        lens = torch.from_numpy(w.seq_lens).to(device)
        if groups is None:
            out = pool.decode(tv(w.q), tables, lens, w.scale)
        else:
            g = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).to(device)
            out = pool.decode_cascade(tv(w.q), tables, lens, w.scale, g)
        torch.cuda.synchronize()
        err = pool.get_error()
    finally:
        pool.close()
    res = wl.value_to_numpy(out, w.dtype)
    if not return_pools:
        return None, None, None, None, res, err
    host = lambda t: None if t is None else t.cpu().numpy()
    return host(kc), host(vc), host(ks), host(vs), res, err


def oracle_step_q8(w: wl.Workload, p: wl.Q8Pools, seqs=None):
    """The same step on the C oracle: returns (codes and scales after the
    append, attention output for `seqs` or every sequence)."""
    h = wl.on_host(w)
    host = lambda a: None if a is None else np.ascontiguousarray(
        a.cpu().numpy() if isinstance(a, torch.Tensor) else a).copy()
    kc, vc, ks, vs = host(p.k_codes), host(p.v_codes), host(p.k_scales), host(p.v_scales)
    assert c_oracle.copy_blocks_q8(kc, vc, ks, vs, h.pairs) == 0
    c_oracle.append_q8(kc, vc, ks, vs, h.k_new, h.v_new, h.dtype, h.slot_mapping, p.cache,
                       p.k_scale, p.v_scale)
    sel = np.arange(h.batch) if seqs is None else np.asarray(seqs, dtype=np.int64)
    out = c_oracle.decode_q8(np.ascontiguousarray(h.q[sel]), h.dtype, kc, vc, ks, vs, p.cache,
                             np.ascontiguousarray(h.block_tables[sel]),
                             np.ascontiguousarray(h.seq_lens[sel]), h.scale, h.num_kv_heads,
                             p.k_scale, p.v_scale, num_threads=ORACLE_THREADS)
    return kc, vc, ks, vs, out


def assert_q8_pools_equal(got, want, what=""):
    for g, r, name in zip(got, want, ("k codes", "v codes", "k scales", "v scales")):
        if r is None:
            assert g is None, f"{what}: {name}"
            continue
        if r.dtype == np.uint8:
            bad = np.flatnonzero(g.reshape(-1) != r.reshape(-1))
            assert bad.size == 0, f"{what}: {name} differ at {bad.size} bytes, first {bad[:5]}"
        else:
            ok = (g.view(np.uint32) == r.view(np.uint32)) | (np.isnan(g) & np.isnan(r))
            assert ok.all(), f"{what}: {name} differ at {np.flatnonzero(~ok.reshape(-1))[:5]}"


# -- paged (chunked) prefill -----------------------------------------------------

def gpu_prefill_step(w: wl.Workload, device="cuda", max_query_len=None, return_pools=True):
    """kv_append of the chunks' K/V -> paged_attention_prefill through the C ABI.
    Returns (k_pool, v_pool, out, error_bits) as raw host arrays."""
    tv = lambda a: wl.value_to_torch(a, w.dtype, device)
    k, v = tv(w.k_pool).clone(), tv(w.v_pool).clone()
    q, kn, vn = tv(w.q), tv(w.k_new), tv(w.v_new)
    slots = torch.from_numpy(w.slot_mapping).to(device)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device)
    lens = torch.from_numpy(w.seq_lens).to(device)
    cu = torch.from_numpy(np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)).to(device)
    mq = int(np.diff(w.cu_seqlens).max()) if max_query_len is None else max_query_len
    pool = pagedkv.KVPool(k, v)
    try:
        pool.append(kn, vn, slots)
        out = torch.zeros_like(q)
        pool.prefill(q, cu, mq, tables, lens, w.scale, out=out)
        torch.cuda.synchronize()
        err = pool.get_error()
    finally:
        pool.close()
    res = wl.value_to_numpy(out, w.dtype)
    if not return_pools:
        return None, None, res, err
    return wl.value_to_numpy(k, w.dtype), wl.value_to_numpy(v, w.dtype), res, err


def oracle_prefill_step(w: wl.Workload, requests=None):
    """The same step on the C oracle.  Returns (k_pool, v_pool, out, rows):
    `out` holds the rows of `requests` (every request if None), `rows` their
    indices in the flattened query stream."""
    h = wl.on_host(w)
    k, v = h.k_pool.copy(), h.v_pool.copy()
    assert c_oracle.append(k, v, h.k_new, h.v_new, h.slot_mapping, h.dtype) == 0
    cu = np.asarray(h.cu_seqlens, dtype=np.int64)
    reqs = np.arange(h.batch) if requests is None else np.asarray(requests)
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in reqs] + [np.zeros(0, np.int64)])
    sub_cu = np.concatenate([[0], np.cumsum([cu[b + 1] - cu[b] for b in reqs])]).astype(np.int32)
    out = c_oracle.prefill(np.ascontiguousarray(h.q[rows]), k, v, h.dtype, sub_cu,
                           np.ascontiguousarray(h.block_tables[reqs]),
                           np.ascontiguousarray(h.seq_lens[reqs]), h.scale, h.num_kv_heads,
                           num_threads=ORACLE_THREADS)
    return k, v, out, rows
