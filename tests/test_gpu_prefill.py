"""GPU parity of paged (chunked) prefill: kv_append of the chunks, then
paged_attention_prefill through the C ABI, against the CPU oracle (GB300,
sm_103a).  Cases span several KV tiles of 128 tokens, several query tiles and
ragged tails of both, every GQA group size, block sizes 8-128, fp16 and bf16,
decode requests mixed in, and the degenerate inputs."""

import numpy as np
import pytest
import torch

from parity import (assert_pools_equal, check_attention, gpu_prefill_step, gpu_step,
                    oracle_prefill_step, TORCH_DTYPE)
from oracle import np_oracle
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _step(name, seed, prefix, chunks, *, dtype="bf16", hq=32, hkv=8, bs=16):
    return wl.chunked_prefill_step(name, seed, prefix, chunks, dtype=dtype, num_q_heads=hq,
                                   num_kv_heads=hkv, head_dim=128, block_size=bs)


def _check(w, what, requests=None, max_query_len=None):
    gk, gv, out, err = gpu_prefill_step(w, max_query_len=max_query_len)
    rk, rv, ref, rows = oracle_prefill_step(w, requests)
    assert err == 0, f"{what}: device error bits {err:#x}"
    assert_pools_equal(gk, gv, rk, rv, what)
    return check_attention(out[rows], ref, w.dtype, what)


# -- the chunked-prefill step at sizes the oracle finishes in seconds ------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_llama3_chunked_prefill_small(seed):
    """A fresh prompt (no prefix), prefixes inside and across KV tiles, chunks of
    1 to 300 queries (ragged query tiles), bf16, GQA group 4."""
    w = _step("small", seed, [0, 5, 130, 300, 1000, 17], [37, 128, 1, 300, 64, 200])
    _check(w, f"llama3 chunked seed {seed}")


def test_llama3_chunked_prefill_workload_small():
    w = wl.chunked_prefill(0, batch=4, chunk=256, max_prefix=1200, decodes=6)
    _check(w, "chunked_prefill workload, small")


@pytest.mark.parametrize("dtype,hq,hkv,bs", [
    ("f16", 8, 8, 16),      # MHA (group 1), the OPT-13B kind
    ("bf16", 16, 8, 32),    # group 2
    ("f16", 32, 4, 8),      # group 8, block size 8
    ("bf16", 8, 2, 64),     # group 4, block size 64
    ("bf16", 16, 4, 128),   # one block per KV tile
])
def test_shapes_groups_and_block_sizes(dtype, hq, hkv, bs):
    w = _step(f"{dtype} {hq}/{hkv} bs{bs}", 3, [0, 77, 400], [150, 33, 129], dtype=dtype,
              hq=hq, hkv=hkv, bs=bs)
    _check(w, f"{dtype} hq{hq} hkv{hkv} bs{bs}")


def test_full_size_workload_sampled():
    """The benchmark's workload (16 requests x 256-token chunks after cached
    prefixes of U[0, 3840] tokens): every request's K/V bit-exact, attention of
    four requests (shortest, longest and two others) against the oracle."""
    w = wl.chunked_prefill(0)
    pre = w.seq_lens - np.diff(w.cu_seqlens)
    order = np.argsort(pre)
    reqs = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 3})
    _check(w, "chunked_prefill full size", requests=reqs)


# -- agreement with decode, edge cases ---------------------------------------------------

def test_one_query_per_request_matches_decode():
    """C_b = 1 for every request is a decode step: prefill and decode kernels
    agree within the tolerance, and both match the oracle."""
    w = _step("decode-like", 4, [0, 15, 16, 127, 128, 700, 2000], [1] * 7)
    _, _, out_p, err = gpu_prefill_step(w, return_pools=False)
    assert err == 0
    _, _, ref, rows = oracle_prefill_step(w)
    check_attention(out_p[rows], ref, w.dtype, "prefill C=1")
    _, _, out_d, err = gpu_step(w, return_pools=False)
    assert err == 0
    check_attention(out_d, ref, w.dtype, "decode")


def test_empty_requests_and_queries_without_context():
    """Requests with no queries are skipped; a chunk longer than the context
    (C_b > L_b) has queries at negative positions, whose output is 0."""
    w = _step("empty", 5, [10, 0, 40, 0], [20, 0, 5, 3])
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[3] = 1                       # 3 queries, context of 1: positions -2, -1, 0
    gk, gv, out, err = gpu_prefill_step(w)
    rk, rv, ref, rows = oracle_prefill_step(w)
    assert err == 0
    check_attention(out[rows], ref, w.dtype, "empty / negative positions")
    lo = int(w.cu_seqlens[3])
    assert not np.any(np_oracle.to_f64(out[lo:lo + 2], w.dtype)), \
        "queries at negative positions must be 0"


def test_repeated_calls_are_bit_identical():
    w = _step("repeat", 6, [333, 50], [200, 90])
    outs = [gpu_prefill_step(w, return_pools=False)[2] for _ in range(2)]
    assert outs[0].tobytes() == outs[1].tobytes()


def test_query_count_past_max_query_len_sets_error():
    w = _step("maxq", 7, [10, 20], [40, 100])
    _, _, out, err = gpu_prefill_step(w, max_query_len=64, return_pools=False)
    assert err & pagedkv.KV_DEVERR_QUERY_RANGE
    # the first request fits and is still computed
    _, _, ref, rows = oracle_prefill_step(w, requests=[0])
    check_attention(out[rows], ref, w.dtype, "request within max_query_len")


def test_bad_block_id_and_overlong_seq_set_errors():
    w = _step("bad", 8, [100, 50], [20, 10])
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 2] = w.num_blocks + 5
    _, _, _, err = gpu_prefill_step(w, return_pools=False)
    assert err & pagedkv.KV_DEVERR_BLOCK_RANGE
    w2 = _step("long", 9, [100], [20])
    w2.seq_lens = np.array([w2.block_tables.shape[1] * 16 + 5], np.int32)
    _, _, _, err = gpu_prefill_step(w2, return_pools=False)
    assert err & pagedkv.KV_DEVERR_SEQ_RANGE


def test_host_argument_errors():
    dev = "cuda"
    k = torch.zeros(8, 16, 2, 128, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    pool = pagedkv.KVPool(k, v)
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, 4], dtype=torch.int32, device=dev)
    tables = torch.zeros(1, 8, dtype=torch.int32, device=dev)
    lens = torch.tensor([4], dtype=torch.int32, device=dev)
    try:
        for kw, status in [({"scale": 0.0}, pagedkv.KV_EINVAL), ({"scale": -1.0}, pagedkv.KV_EINVAL),
                           ({"max_query_len": 0}, pagedkv.KV_EINVAL),
                           ({"max_query_len": 5}, pagedkv.KV_EINVAL)]:
            args = {"scale": 0.1, "max_query_len": 4}
            args.update(kw)
            with pytest.raises(pagedkv.PagedKVError) as ei:
                pool.prefill(q, cu, args["max_query_len"], tables, lens, args["scale"])
            assert ei.value.status == status
        with pytest.raises(pagedkv.PagedKVError) as ei:        # group of 3
            pagedkv.paged_attention_prefill(pool.handle, q[:, :6].contiguous(), q[:, :6].clone(),
                                            cu, 4, tables, lens, 0.1, 2, torch.bfloat16)
        assert ei.value.status == pagedkv.KV_EUNSUPPORTED
    finally:
        pool.close()
    k32 = torch.zeros(8, 16, 2, 128, dtype=torch.float32, device=dev)
    pool32 = pagedkv.KVPool(k32, k32.clone())
    try:
        q32 = torch.zeros(4, 8, 128, dtype=torch.float32, device=dev)
        with pytest.raises(pagedkv.PagedKVError) as ei:
            pool32.prefill(q32, cu, 4, tables, lens, 0.1)
        assert ei.value.status == pagedkv.KV_EUNSUPPORTED
    finally:
        pool32.close()


def test_many_requests_keep_grid_order_and_ties():
    """More requests than the launch order ranks (257 > 256): the grid's own
    order is used; a batch with many equal costs exercises the ranking's
    tie-break.  Both match the oracle on sampled requests."""
    rng = np.random.default_rng(11)
    pre = rng.integers(0, 300, size=257)
    chk = rng.integers(1, 40, size=257)
    w = _step("257 requests", 11, pre, chk)
    _check(w, "257 requests", requests=[0, 1, 128, 255, 256])
    w2 = _step("ties", 12, [64] * 12 + [200, 7], [30] * 12 + [65, 1])
    _check(w2, "equal costs")
