"""GPU parity of kv_swap_blocks: blocks moved to a pinned host pool and back
through the C ABI equal the oracle's swap byte for byte, and decode after a
swap round trip into other physical blocks gives the same bits."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import c_oracle, np_oracle
from parity import TORCH_DTYPE
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl
from paged_kv_cache_68_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _np(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _pool(w, cache):
    dev = torch.device("cuda")
    if cache is None:
        tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
        return pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone()), None
    p = wl.q8_pools(w, cache, 5)
    t = lambda a: (a.clone() if isinstance(a, torch.Tensor)
                   else torch.from_numpy(np.ascontiguousarray(a))).to(dev)
    pool = pagedkv.KVPool(t(p.k_codes), t(p.v_codes), cache=cache, dtype=TORCH_DTYPE[w.dtype],
                          k_scales=None if p.k_scales is None else t(p.k_scales),
                          v_scales=None if p.v_scales is None else t(p.v_scales))
    return pool, p


def _arrays(pool):
    return [a for a in (pool.k_pool, pool.v_pool, pool.k_scales, pool.v_scales) if a is not None]


@pytest.mark.parametrize("cache", [None, "fp8_e4m3", "int8"])
def test_swap_out_and_in_match_the_oracle(cache):
    w = wl.build_step("swap", 2, [40, 7, 100, 33, 16], dtype="bf16", num_q_heads=16,
                      num_kv_heads=4, head_dim=128, block_size=16, pool_factor=2.5)
    dev = torch.device("cuda")
    pool, _ = _pool(w, cache)
    try:
        host = pool.host_pool(12)
        for a in host:
            if a is not None:
                a.view(torch.uint8).fill_(0xAB)
        gpu0 = [_np(a) for a in _arrays(pool)]
        host0 = [_np(a) for a in host if a is not None]
        tables = w.block_tables
        out_pairs = np.array([[int(tables[2, j]), j] for j in range(7)] + [[int(tables[0, 1]), 9]],
                             np.int32)
        pool.swap_out(host, torch.from_numpy(out_pairs).to(dev))
        torch.cuda.synchronize()
        g_ref = [a.copy() for a in gpu0]
        h_ref = [a.copy() for a in host0]
        assert c_oracle.swap_blocks(g_ref, h_ref, out_pairs, np_oracle.SWAP_OUT) == 0
        for got, ref in zip([a for a in host if a is not None], h_ref):
            assert _np(got).tobytes() == ref.tobytes()
        # in: host blocks 0..6 -> the spare GPU blocks, 9 -> another spare
        used = set(int(b) for b in tables.reshape(-1) if b >= 0)
        spare = [b for b in range(w.num_blocks) if b not in used]
        in_pairs = np.array([[spare[j], j] for j in range(7)] + [[spare[8], 9]], np.int32)
        pool.swap_in(host, torch.from_numpy(in_pairs).to(dev))
        torch.cuda.synchronize()
        assert c_oracle.swap_blocks(g_ref, h_ref, in_pairs, np_oracle.SWAP_IN) == 0
        for got, ref in zip(_arrays(pool), g_ref):
            assert _np(got).tobytes() == ref.tobytes()
        assert pool.get_error() == 0
    finally:
        pool.close()


@pytest.mark.parametrize("cache", [None, "int8"])
def test_decode_after_a_block_manager_swap_round_trip_is_bit_identical(cache):
    """A group preempted by the block manager: swap out, the freed GPU blocks
    reused and overwritten, swap back into different blocks; decode through
    the new tables gives the same bits as before."""
    rng = np.random.default_rng(4)
    bs, hkv, d, hq = 16, 8, 128, 32
    bm = BlockManager(64, bs, free_order=rng.permutation(64).tolist(), num_cpu_blocks=32)
    lens = [90, 33, 47, 150]
    for s, L in enumerate(lens):
        bm.allocate_prompt(s, L)
    width = max(len(t) for t in bm.tables.values()) + 1
    tab = lambda: np.array([bm.tables[s] + [-1] * (width - len(bm.tables[s])) for s in range(4)],
                           np.int32)
    w = wl.build_step("swap-bm", 6, [1] * 4, dtype="bf16", num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d, block_size=bs, num_blocks=64)
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    k = torch.randn((64, bs, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((64, bs, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    if cache is None:
        pool = pagedkv.KVPool(k, v)
    else:
        w.k_pool, w.v_pool = k, v
        pool, _ = _pool(w, cache)
    try:
        q = torch.randn((4, hq, d), generator=g, device=dev).to(torch.bfloat16)
        lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
        before = pool.decode(q, torch.from_numpy(tab()).to(dev), lens_t, 0.088).clone()
        host = pool.host_pool(32)
        pairs = bm.swap_out([1, 3])
        pool.swap_out(host, torch.tensor(pairs, dtype=torch.int32, device=dev))
        bm.allocate_prompt(9, 200)                     # reuses the freed blocks ...
        for blk in bm.tables[9]:                       # ... and overwrites them
            for a in _arrays(pool):
                a[blk].view(torch.uint8).fill_(0x7F)
        bm.free_seq(9)
        back = bm.swap_in([1, 3])
        pool.swap_in(host, torch.tensor(back, dtype=torch.int32, device=dev))
        bm.check_invariant()
        after = pool.decode(q, torch.from_numpy(tab()).to(dev), lens_t, 0.088)
        torch.cuda.synchronize()
        assert torch.equal(before.view(torch.int16), after.view(torch.int16))
        assert pool.get_error() == 0
    finally:
        pool.close()


def test_swap_errors():
    w = wl.build_step("swap-err", 3, [20], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                      head_dim=128, block_size=16)
    dev = torch.device("cuda")
    pool, _ = _pool(w, None)
    try:
        host = pool.host_pool(4)
        pool.swap_out(host, torch.tensor([[0, 7], [1, 1]], dtype=torch.int32, device=dev))
        assert pool.get_error() & pagedkv.KV_DEVERR_PAIR_RANGE
        pool.clear_error()
        with pytest.raises(ValueError):                  # pageable host memory
            pagedkv.kv_swap_blocks(pool.handle, torch.empty(host[0].shape, dtype=host[0].dtype),
                                   host[1], torch.zeros((1, 2), dtype=torch.int32, device=dev),
                                   pagedkv.KV_SWAP_OUT)
        lib = pagedkv.load()
        pageable = np.zeros(host[0].numel() // 2 + 64, np.uint16)
        ptr = (pageable.ctypes.data + 15) // 16 * 16
        # the pair names a host block past the pool, so even a launch would
        # touch no host memory; the call must refuse before that
        pr = torch.tensor([[0, 99]], dtype=torch.int32, device=dev)
        st = lib.kv_swap_blocks(pool.handle, ctypes.c_void_p(ptr), ctypes.c_void_p(host[1].data_ptr()),
                                None, None, 4, ctypes.c_void_p(pr.data_ptr()), 1, 0, None)
        assert st == pagedkv.KV_EINVAL
        st = lib.kv_swap_blocks(pool.handle, ctypes.c_void_p(host[0].data_ptr()),
                                ctypes.c_void_p(host[1].data_ptr()), None, None, 4,
                                ctypes.c_void_p(pr.data_ptr()), 1, 2, None)
        assert st == pagedkv.KV_EINVAL                   # bad direction
        assert pool.get_error() == 0
    finally:
        pool.close()
