"""Swap to host, CPU side (no GPU): the oracle's swap copy against its pins,
and the block manager's CPU block allocator ("Lecture 3", sec. 5.2: a
preempted request's blocks go to CPU memory through a CPU block allocator and
come back on resume; the swap space needed is bounded by the GPU pool)."""

import numpy as np
import pytest

from oracle import c_oracle as co
from oracle import np_oracle as npo
from paged_kv_cache_68_gb300 import workloads as wl
from paged_kv_cache_68_gb300.block_manager import BlockManager, OutOfBlocks


def _pools(rng, nb, bs=4, hkv=2, d=8, scales=False):
    k = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
    v = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
    arrs = [k, v]
    if scales:
        arrs += [rng.random((nb, hkv, bs)).astype(np.float32) for _ in range(2)]
    return arrs


@pytest.mark.parametrize("scales", [False, True])
def test_swap_numpy_and_c_agree_and_count_bad_pairs(c_oracle, scales):
    rng = np.random.default_rng(1)
    gpu = _pools(rng, 10, scales=scales)
    host = [np.zeros((6,) + a.shape[1:], a.dtype) for a in gpu]
    pairs = [[3, 0], [7, 5], [9, 2], [10, 1], [2, 6]]
    res = []
    for impl in (npo, co):
        g = [a.copy() for a in gpu]
        h = [a.copy() for a in host]
        assert impl.swap_blocks(g, h, pairs, npo.SWAP_OUT) == 2
        g2 = [np.full_like(a, np.nan) for a in g]
        assert impl.swap_blocks(g2, h, [[0, 0], [1, 5], [4, 2]], npo.SWAP_IN) == 0
        res.append((h, g2))
    (h1, g1), (h2, g2) = res
    for a, b in zip(h1 + g1, h2 + g2):
        assert np.array_equal(a, b, equal_nan=True)


def test_swap_out_then_in_equals_copy_blocks(c_oracle):
    """Out to host block h, in to GPU block g' == the pinned copy g -> g'."""
    rng = np.random.default_rng(2)
    k, v = _pools(rng, 12)
    hk, hv = np.zeros((4,) + k.shape[1:], k.dtype), np.zeros((4,) + v.shape[1:], v.dtype)
    ref_k, ref_v = k.copy(), v.copy()
    assert co.copy_blocks(ref_k, ref_v, [[2, 8], [5, 9]], "f32") == 0
    assert co.swap_blocks([k, v], [hk, hv], [[2, 3], [5, 0]], npo.SWAP_OUT) == 0
    assert co.swap_blocks([k, v], [hk, hv], [[8, 3], [9, 0]], npo.SWAP_IN) == 0
    assert np.array_equal(k, ref_k) and np.array_equal(v, ref_v)


def test_decode_is_unchanged_by_a_swap_round_trip(c_oracle):
    """Attention reads blocks through the table, so moving a preempted
    sequence's blocks out and back into other physical blocks changes nothing
    ("Lecture 3", sec. 3.2: the kernel sees only physical block numbers)."""
    w = wl.build_step("swap", 3, [13, 30, 7], dtype="f32", num_q_heads=4, num_kv_heads=2,
                      head_dim=16, block_size=4, pool_factor=3.0)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    co.append(k, v, w.k_new, w.v_new, w.slot_mapping, "f32")
    before = co.decode(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 2)
    # sequence 1 leaves: its blocks go to host, its GPU blocks are reused
    table1 = [int(b) for b in w.block_tables[1] if b >= 0]
    hk = np.zeros((len(table1),) + k.shape[1:], k.dtype)
    hv = np.zeros_like(hk)
    assert co.swap_blocks([k, v], [hk, hv], [[b, i] for i, b in enumerate(table1)], npo.SWAP_OUT) == 0
    k[table1] = np.nan
    v[table1] = np.nan
    used = set(int(b) for b in w.block_tables.reshape(-1) if b >= 0)
    fresh = [b for b in range(k.shape[0]) if b not in used][:len(table1)]
    assert co.swap_blocks([k, v], [hk, hv], [[b, i] for i, b in enumerate(fresh)], npo.SWAP_IN) == 0
    tables = w.block_tables.copy()
    tables[1, :len(fresh)] = fresh
    after = co.decode(w.q, k, v, "f32", tables, w.seq_lens, w.scale, 2)
    assert np.array_equal(before, after)


# --- the CPU block allocator -------------------------------------------------------

def test_swap_group_round_trip_keeps_counts_and_tables():
    bm = BlockManager(16, 4, num_cpu_blocks=8)
    bm.allocate_prompt(0, 10)                       # 3 blocks
    bm.fork(0, 1)
    bm.append_slot(1)                               # 1 copies its last block (shared)
    bm.allocate_prompt(2, 5)
    before = {s: list(bm.tables[s]) for s in (0, 1)}
    pairs = bm.swap_out([0, 1])
    bm.check_invariant()
    assert sorted(p[0] for p in pairs) == sorted(set(before[0] + before[1]))
    assert len(pairs) == 4 and bm.num_free() == 16 - 2
    with pytest.raises(ValueError):
        bm.append_slot(0)
    back = bm.swap_in([0, 1])
    bm.check_invariant()
    cpu_of = {g: c for g, c in pairs}
    gpu_of = {c: g for g, c in back}
    for s in (0, 1):
        assert bm.tables[s] == [gpu_of[cpu_of[b]] for b in before[s]]
    assert bm.ref[bm.tables[0][0]] == 2             # the shared prompt blocks stay shared
    assert not bm.swapped


def test_swap_refuses_blocks_shared_outside_the_group():
    bm = BlockManager(8, 4, num_cpu_blocks=8)
    bm.allocate_prompt(0, 8)
    bm.fork(0, 1)
    with pytest.raises(ValueError):
        bm.swap_out([0])
    bm.check_invariant()


def test_swap_space_and_gpu_space_run_out_all_or_nothing():
    bm = BlockManager(8, 4, num_cpu_blocks=2)
    bm.allocate_prompt(0, 12)                       # 3 blocks > 2 swap blocks
    with pytest.raises(OutOfBlocks):
        bm.swap_out([0])
    bm.check_invariant()
    bm2 = BlockManager(4, 4, num_cpu_blocks=4)
    bm2.allocate_prompt(0, 16)
    bm2.swap_out([0])
    bm2.allocate_prompt(1, 5)                       # takes 2 of the freed blocks
    with pytest.raises(OutOfBlocks):
        bm2.swap_in([0])
    bm2.check_invariant()
    bm2.free_seq(0)                                 # a swapped sequence can be dropped
    bm2.check_invariant()
    assert len(bm2.cpu_free) == 4


def test_swapping_everything_fits_a_swap_space_the_size_of_the_pool():
    """The swap space needed is bounded by the GPU pool: every sequence out at
    once fits num_cpu_blocks = num_blocks."""
    rng = np.random.default_rng(3)
    bm = BlockManager(40, 4, free_order=rng.permutation(40).tolist(), num_cpu_blocks=40)
    sid = 0
    while bm.num_free() >= 3:
        bm.allocate_prompt(sid, int(rng.integers(1, 12)))
        sid += 1
    used = 40 - bm.num_free()
    pairs = bm.swap_out(list(range(sid)))
    assert len(pairs) == used and bm.num_free() == 40
    bm.check_invariant()
