"""GPU parity: copy_blocks, kv_append and paged_attention_decode through the C
ABI against the CPU oracle, on every decode-step configuration and its edge
cases (GB300, sm_103a)."""

import numpy as np
import pytest
import torch

from parity import assert_pools_equal, check_attention, gpu_step, oracle_step, TORCH_DTYPE
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _full_check(w, what, seqs=None):
    gk, gv, out, err = gpu_step(w)
    rk, rv, ref = oracle_step(w, seqs)
    assert err == 0, f"{what}: device error bits {err:#x}"
    assert_pools_equal(gk, gv, rk, rv, what)
    sel = slice(None) if seqs is None else np.asarray(seqs)
    return check_attention(out[sel], ref, w.dtype, what)


# -- the configurations, at sizes the oracle finishes in seconds -----------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32(seed):
    _full_check(wl.tiny(seed), f"tiny seed {seed}")


@pytest.mark.parametrize("seed", [0, 1])
def test_opt13b_mha_small(seed):
    _full_check(wl.opt13b_mha(seed, batch=8, lo=1, hi=700), f"opt13b small {seed}")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_llama3_gqa_small(seed):
    _full_check(wl.llama3_8b_gqa(seed, batch=24, median=200, hi=1500), f"llama3 small {seed}")


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_long_context_small(bs):
    _full_check(wl.long_context(0, batch=3, lo=3000, hi=9000, block_size=bs), f"long bs{bs}")


@pytest.mark.parametrize("prompt_len", [2000, 2008])
def test_shared_prefix_small(prompt_len):
    w = wl.shared_prefix(0, prompts=3, prompt_len=prompt_len, n=4, max_divergent=40)
    _full_check(w, f"shared prefix {prompt_len}")


def test_shared_prefix_fresh_fork_copies():
    """First decode step after a fork with a partial last prompt block: three
    copy-on-write copies per prompt go through copy_blocks in this step."""
    w = wl.shared_prefix(0, prompts=4, prompt_len=2008, n=4, divergent=np.zeros(16, np.int64))
    assert w.pairs.shape == (12, 2)
    _full_check(w, "fresh fork")


@pytest.mark.parametrize("batch,median,hi,launches", [(256, 48, 400, 1), (96, 48, 400, 2),
                                                      (4, 1500, 6000, 2)])
def test_both_merge_paths(batch, median, hi, launches):
    """A (sequence, KV head) cut across warp ranges is merged in the split
    kernel when the pairs are many (one launch) and by a second kernel when
    there are fewer (two launches: one warp per pair for some hundreds of
    pairs, four warps sharing a pair's partials for a few pairs): each
    against the oracle, at sizes that reach each path."""
    w = wl.llama3_8b_gqa(11, batch=batch, median=median, hi=hi)
    k = torch.empty(tuple(w.k_pool.shape), dtype=TORCH_DTYPE[w.dtype], device="cuda")
    pool = pagedkv.KVPool(k, k.clone())
    try:
        n = pagedkv.paged_attention_decode_launches(pool.handle, w.batch, w.num_q_heads)
    finally:
        pool.close()
    assert n == launches
    _full_check(w, f"merge path ({launches} launches)")


def test_max_batch_of_short_and_empty_sequences():
    """4,096 sequences (the largest batch) of 0-41 tokens, one in twenty empty:
    thousands of short pieces per warp range, and (b, g) pairs with no units."""
    rng = np.random.default_rng(21)
    ctx = rng.integers(0, 41, size=4096)
    w = wl.build_step("max batch", 21, ctx, dtype="bf16", num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=16)
    lens = np.asarray(w.seq_lens).copy()
    lens[rng.random(4096) < 0.05] = 0
    w.seq_lens = lens.astype(np.int32)
    print(_full_check(w, "max batch, short and empty"))


def test_long_contexts_with_an_empty_sequence():
    """The merge kernel's path (few (b, g) pairs, each cut across many warp
    ranges) with a zero-length sequence among the long ones."""
    w = wl.long_context(5, batch=3, lo=3000, hi=9000, block_size=16)
    lens = np.asarray(w.seq_lens).copy()
    lens[1] = 0
    w.seq_lens = lens.astype(np.int32)
    print(_full_check(w, "long contexts, one empty"))


# -- full sizes, in the launch configuration the benchmark times --------------------

@pytest.mark.slow
def test_llama3_gqa_full():
    w = wl.llama3_8b_gqa(0, device="cuda")
    print(_full_check(w, "llama3 full"))


@pytest.mark.slow
def test_opt13b_mha_full():
    w = wl.opt13b_mha(0, device="cuda")
    print(_full_check(w, "opt13b full"))


@pytest.mark.slow
def test_shared_prefix_full():
    w = wl.shared_prefix(0, device="cuda")
    print(_full_check(w, "shared prefix full"))
    w = wl.shared_prefix(0, prompt_len=2008, device="cuda")
    print(_full_check(w, "shared prefix 2008 full"))


@pytest.mark.slow
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_long_context_full_sampled(bs):
    """Full-size long-context step; the oracle checks 3 of the 8 sequences."""
    w = wl.long_context(0, block_size=bs, device="cuda")
    print(_full_check(w, f"long full bs{bs}", seqs=[0, 3, 7]))


# -- edge cases ---------------------------------------------------------------------

@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("f32", 8, 8, 64, 4), ("f32", 8, 2, 128, 16), ("f16", 4, 4, 64, 16), ("f16", 16, 2, 128, 8),
    ("bf16", 16, 8, 128, 16), ("bf16", 16, 2, 64, 32), ("bf16", 8, 1, 128, 1), ("f16", 8, 4, 64, 5),
    # tensor-core path: 16-bit, head_dim 128, groups of 4 / 8, block sizes 8 (two blocks
    # per tile), 16 and 32
    ("bf16", 16, 2, 128, 16), ("bf16", 32, 4, 128, 32), ("f16", 32, 8, 128, 16),
    ("f16", 16, 2, 128, 32), ("bf16", 32, 8, 128, 8),
])
def test_shapes_groups_and_block_sizes(dtype, hq, hkv, d, bs):
    ctx = [0, 1, bs - 1, bs, 2 * bs - 1, 3 * bs, 97, 300]
    w = wl.build_step("shapes", 3, [max(0, c) for c in ctx], dtype=dtype, num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=d, block_size=bs)
    _full_check(w, f"{dtype} {hq}/{hkv} d{d} bs{bs}")


def test_seq_len_one_returns_v0():
    w = wl.build_step("one", 4, [0, 0, 0], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                      head_dim=128, block_size=16)
    _, _, out, err = gpu_step(w)
    assert err == 0
    vn = np.repeat(w.v_new, 4, axis=1)           # each query head sees its kv head's row
    assert np.array_equal(out, vn)


def test_zero_length_sequence_gives_zeros():
    w = wl.build_step("zero", 5, [10, 20], dtype="f16", num_q_heads=4, num_kv_heads=4,
                      head_dim=64, block_size=16)
    w.seq_lens = np.array([0, 21], np.int32)
    _, _, out, err = gpu_step(w)
    assert err == 0
    assert np.all(out[0] == 0) and np.isfinite(out[1].astype(np.float32)).all()


def test_placement_permutation_gives_identical_bits():
    """Scattered and contiguous placement of the same tokens: bit-identical
    output (the work split depends only on the lengths)."""
    a = wl.llama3_8b_gqa(7, batch=16, median=300, hi=2000)
    b = wl.llama3_8b_gqa(7, batch=16, median=300, hi=2000, placement="identity")
    # same tokens, same values, different physical blocks: rebuild b's pools from a's rows
    bs = a.block_size
    ka, va = a.k_pool.reshape(-1, 8, 128), a.v_pool.reshape(-1, 8, 128)
    kb, vb = wl.nan_fill(b.k_pool.shape, "bf16"), wl.nan_fill(b.v_pool.shape, "bf16")
    for s in range(a.batch):
        L = int(a.seq_lens[s]) - 1
        pos = np.arange(L)
        ra = a.block_tables[s][pos // bs] * bs + pos % bs
        rb = b.block_tables[s][pos // bs] * bs + pos % bs
        kb.reshape(-1, 8, 128)[rb] = ka[ra]
        vb.reshape(-1, 8, 128)[rb] = va[ra]
    b.k_pool, b.v_pool, b.q, b.k_new, b.v_new = kb, vb, a.q, a.k_new, a.v_new
    _, _, oa, _ = gpu_step(a, return_pools=False)
    _, _, ob, _ = gpu_step(b, return_pools=False)
    assert np.array_equal(oa, ob)


def test_empty_copy_list_and_all_padding_slots():
    w = wl.tiny(0)
    w.slot_mapping = np.full_like(w.slot_mapping, -1)
    gk, gv, _, err = gpu_step(w)
    assert err == 0
    assert gk.tobytes() == w.k_pool.tobytes() and gv.tobytes() == w.v_pool.tobytes()


def _pool_on_gpu(w):
    k = wl.value_to_torch(w.k_pool, w.dtype, "cuda").clone()
    v = wl.value_to_torch(w.v_pool, w.dtype, "cuda").clone()
    return pagedkv.KVPool(k, v)


def test_out_of_range_slot_sets_error_and_is_skipped():
    w = wl.tiny(1)
    slots = w.slot_mapping.copy()
    slots[2] = w.num_blocks * w.block_size + 5
    pool = _pool_on_gpu(w)
    try:
        pool.append(wl.value_to_torch(w.k_new, "f32", "cuda"), wl.value_to_torch(w.v_new, "f32", "cuda"),
                    torch.from_numpy(slots).cuda())
        assert pool.get_error() & pagedkv.KV_DEVERR_SLOT_RANGE
        ref = w.k_pool.copy()
        for i in (0, 1, 3):
            ref[slots[i] // 4, slots[i] % 4] = w.k_new[i]
        assert pool.k_pool.cpu().numpy().tobytes() == ref.tobytes()
        pool.clear_error()
        assert pool.get_error() == 0
    finally:
        pool.close()


def test_out_of_range_pair_sets_error():
    w = wl.tiny(2)
    pool = _pool_on_gpu(w)
    try:
        pool.copy_blocks(torch.tensor([[0, 1], [3, 64]], dtype=torch.int32, device="cuda"))
        assert pool.get_error() & pagedkv.KV_DEVERR_PAIR_RANGE
        k = pool.k_pool.cpu().numpy()
        assert np.array_equal(k[1], w.k_pool[0], equal_nan=True)
    finally:
        pool.close()


def test_bad_block_id_and_overlong_seq_set_errors_and_skip():
    w = wl.tiny(3)
    from oracle import c_oracle
    k, v = np.nan_to_num(w.k_pool, nan=0.5), np.nan_to_num(w.v_pool, nan=0.25)
    c_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping, "f32")
    bt = w.block_tables.copy()
    bt[1, 2] = 9999
    lens = w.seq_lens.copy()
    lens[3] = bt.shape[1] * w.block_size + 40          # longer than its table
    ref, st = c_oracle.decode(w.q, k, v, "f32", bt, lens, w.scale, 4, return_status=True)
    assert st > 0
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    pool = pagedkv.KVPool(kt, vt)
    try:
        out = pool.decode(torch.from_numpy(w.q).cuda(), torch.from_numpy(bt).cuda(),
                          torch.from_numpy(lens).cuda(), w.scale)
        bits = pool.get_error()
        assert bits & pagedkv.KV_DEVERR_BLOCK_RANGE and bits & pagedkv.KV_DEVERR_SEQ_RANGE
        check_attention(out.cpu().numpy(), ref, "f32", "bad ids")
    finally:
        pool.close()


def test_host_argument_errors():
    w = wl.tiny(0)
    pool = _pool_on_gpu(w)
    try:
        q = wl.value_to_torch(w.q, "f32", "cuda")
        tables = torch.from_numpy(w.block_tables).cuda()
        lens = torch.from_numpy(w.seq_lens).cuda()
        ws = pool.workspace(4, 4)
        with pytest.raises(pagedkv.PagedKVError) as e:        # wrong kv heads
            pagedkv.paged_attention_decode(pool.handle, q, torch.empty_like(q), tables, lens, 0.1,
                                           2, ws, torch.float32)
        assert e.value.status == pagedkv.KV_EINVAL
        with pytest.raises(pagedkv.PagedKVError) as e:        # workspace too small
            pagedkv.paged_attention_decode(pool.handle, q, torch.empty_like(q), tables, lens, 0.1,
                                           4, ws[:16], torch.float32)
        assert e.value.status == pagedkv.KV_ENOWORKSPACE
        q3 = torch.zeros(4, 12, 64, device="cuda")             # group 3
        with pytest.raises(pagedkv.PagedKVError) as e:
            pool.decode(q3, tables, lens, 0.1, workspace=ws)
        assert e.value.status == pagedkv.KV_EUNSUPPORTED
    finally:
        pool.close()


def test_repeated_calls_are_deterministic():
    w = wl.llama3_8b_gqa(3, batch=32, median=500, hi=4000)
    _, _, o1, _ = gpu_step(w, return_pools=False)
    _, _, o2, _ = gpu_step(w, return_pools=False)
    assert np.array_equal(o1, o2)
