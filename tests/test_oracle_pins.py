"""Pins of the CPU oracle against things other than itself (no GPU).

Each pin names what fixes the expected value: a closed form, a library
routine, an invariant the pages state, or the other (independently written)
oracle.  Both oracles -- numpy and plain C -- go through every pin.
"""

import math

import numpy as np
import pytest
import torch

from oracle import np_oracle
from paged_kv_cache_68_gb300 import workloads as wl

DTYPES = ["f32", "f16", "bf16"]


def _both(c_oracle):
    return [("numpy", lambda *a, **k: np_oracle.decode(*a, **k)),
            ("c", lambda *a, **k: c_oracle.decode(*a, **k)),
            ("c4", lambda *a, **k: c_oracle.decode(*a, num_threads=4, **k))]


def _pool(n_blocks, bs, hkv, d, dtype, fill=np.nan):
    return wl.nan_fill((n_blocks, bs, hkv, d), dtype)


def _set_rows(pool, table, values_f32, dtype):
    """Write float32 rows [L, Hkv, D] into pool positions 0..L-1 of `table`."""
    bs = pool.shape[1]
    for t in range(values_f32.shape[0]):
        pool[table[t // bs], t % bs] = wl.from_f32(values_f32[t], dtype)


# --- element decoding: brute force against library conversions --------------

def test_f16_decoder_all_bit_patterns(c_oracle):
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([c_oracle.decode_elem(bits, i, "f16") for i in range(1 << 16)])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    assert np.array_equal(np_oracle.to_f64(bits.view(np.float16), "f16"), want, equal_nan=True)


def test_bf16_decoder_all_bit_patterns(c_oracle):
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([c_oracle.decode_elem(bits, i, "bf16") for i in range(1 << 16)])
    assert np.array_equal(got, want, equal_nan=True)
    assert np.array_equal(np_oracle.to_f64(bits, "bf16"), want, equal_nan=True)


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(100_000, dtype=np.float32) * 7
    mine = wl.from_f32(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


# --- closed forms on hand-worked cases ----------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
def test_one_token_returns_v0_exactly(c_oracle, dtype):
    """seq_len 1: the softmax weight is exactly 1, so out = v_0."""
    rng = np.random.default_rng(3)
    bs, hkv, d = 4, 2, 8
    pool_k, pool_v = _pool(6, bs, hkv, d, dtype), _pool(6, bs, hkv, d, dtype)
    table = np.array([[5, -1]], dtype=np.int32)
    kv = rng.standard_normal((2, 1, hkv, d), dtype=np.float32)
    _set_rows(pool_k, table[0], kv[0], dtype)
    _set_rows(pool_v, table[0], kv[1], dtype)
    q = wl.from_f32(rng.standard_normal((1, 4, d), dtype=np.float32), dtype)
    want = np_oracle.to_f64(pool_v[5, 0], dtype)            # [Hkv, D]
    for name, f in _both(c_oracle):
        out = f(q, pool_k, pool_v, dtype, table, np.array([1], np.int32), 0.3, hkv)
        assert np.array_equal(out[0, :2], np.repeat(want[:1], 2, 0)), name
        assert np.array_equal(out[0, 2:], np.repeat(want[1:], 2, 0)), name


def test_two_tokens_sigmoid_form(c_oracle):
    """Two positions: w_0 = 1 / (1 + exp(s_1 - s_0)), w_1 = 1 - w_0.

    q = (2, 0, 0, 0), k_0 = (1, 0, 0, 0), k_1 = (0, 1, 0, 0), scale 0.5:
    s_0 = 1, s_1 = 0.  v_0 = (4, 0, 0, 2), v_1 = (0, 8, 0, 2).
    """
    bs, d = 4, 4
    pk, pv = _pool(3, bs, 1, d, "f32"), _pool(3, bs, 1, d, "f32")
    table = np.array([[2]], dtype=np.int32)
    pk[2, 0, 0], pk[2, 1, 0] = [1, 0, 0, 0], [0, 1, 0, 0]
    pv[2, 0, 0], pv[2, 1, 0] = [4, 0, 0, 2], [0, 8, 0, 2]
    q = np.array([[[2, 0, 0, 0]]], dtype=np.float32)
    w0 = 1.0 / (1.0 + math.exp(-1.0))
    want = np.array([4 * w0, 8 * (1 - w0), 0.0, 2.0])
    for name, f in _both(c_oracle):
        out = f(q, pk, pv, "f32", table, np.array([2], np.int32), 0.5, 1)
        np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-14, err_msg=name)


def test_three_tokens_across_blocks(c_oracle):
    """Scores (a, 0, b) with e^a = 2, e^b = 5: weights 2/8, 1/8, 5/8.

    Block size 2 so the three positions straddle two physical blocks listed
    out of order in the table (logical 0 -> physical 3, logical 1 -> 0).
    """
    bs, d = 2, 2
    pk, pv = _pool(4, bs, 1, d, "f32"), _pool(4, bs, 1, d, "f32")
    table = np.array([[3, 0]], dtype=np.int32)
    a, b = np.float32(math.log(2.0)), np.float32(math.log(5.0))
    pk[3, 0, 0], pk[3, 1, 0], pk[0, 0, 0] = [a, 0], [0, 0], [b, 0]
    pv[3, 0, 0], pv[3, 1, 0], pv[0, 0, 0] = [8, 0], [0, 8], [8, 8]
    q = np.array([[[1, 0]]], dtype=np.float32)
    ea, eb = math.exp(float(a)), math.exp(float(b))     # the stored (rounded) scores
    z = ea + 1 + eb
    want = np.array([8 * (ea + eb) / z, 8 * (1 + eb) / z])
    for name, f in _both(c_oracle):
        out = f(q, pk, pv, "f32", table, np.array([3], np.int32), 1.0, 1)
        np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-13, err_msg=name)
        np.testing.assert_allclose(out[0, 0], [8 * 7 / 8, 8 * 6 / 8], rtol=0, atol=1e-6)


@pytest.mark.parametrize("dtype", DTYPES)
def test_q_zero_gives_mean_of_v(c_oracle, dtype):
    """q = 0: every score is 0, the weights are uniform, out = mean_t v_t."""
    w = wl.tiny(seed=5) if dtype == "f32" else wl.build_step(
        "t", 5, [9, 30, 1], dtype=dtype, num_q_heads=6, num_kv_heads=3, head_dim=32, block_size=8)
    q = np.zeros_like(w.q)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    group = w.num_q_heads // w.num_kv_heads
    for name, f in _both(c_oracle):
        out = f(q, k, v, w.dtype, w.block_tables, w.seq_lens, w.scale, w.num_kv_heads)
        for b in range(w.batch):
            V = np_oracle.to_f64(np_oracle.gather_kv(v, w.block_tables[b], int(w.seq_lens[b])), w.dtype)
            want = np.repeat(V.mean(axis=0), group, axis=0)
            np.testing.assert_allclose(out[b], want, rtol=0, atol=1e-13, err_msg=name)


def test_gqa_contiguous_grouping(c_oracle):
    """V of kv head g is the constant g + 1, so out[h] = h // group + 1 exactly
    ([RL-Part3] ch. 9 sec. 1: query heads form groups of consecutive heads)."""
    w = wl.build_step("g", 7, [5, 40], dtype="f32", num_q_heads=8, num_kv_heads=2,
                      head_dim=16, block_size=4)
    v = w.v_pool.copy()
    for g in range(2):
        v[:, :, g, :] = np.where(np.isnan(v[:, :, g, :]), np.nan, g + 1)
    vn = np.ones_like(w.v_new)
    vn[:, 1] = 2
    k = w.k_pool.copy()
    np_oracle.append(k, v, w.k_new, vn, w.slot_mapping)
    for name, f in _both(c_oracle):
        out = f(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 2)
        for h in range(8):
            np.testing.assert_allclose(out[:, h], h // 4 + 1, rtol=0, atol=1e-13,
                                       err_msg=f"{name} head {h}")


def test_seq_len_zero_gives_zeros(c_oracle):
    w = wl.build_step("z", 2, [0, 3], dtype="bf16", num_q_heads=2, num_kv_heads=1,
                      head_dim=8, block_size=4)
    lens = np.array([0, 4], np.int32)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    for name, f in _both(c_oracle):
        out = f(w.q, k, v, "bf16", w.block_tables, lens, w.scale, 1)
        assert np.all(out[0] == 0) and np.all(np.isfinite(out[1])), name


# --- reductions to a library routine -----------------------------------------------

@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("f32", 4, 4, 64, 4), ("f16", 8, 8, 32, 16),
                                               ("bf16", 8, 2, 64, 8), ("bf16", 16, 2, 128, 32)])
def test_identity_table_equals_torch_sdpa(c_oracle, dtype, hq, hkv, d, bs):
    """With each sequence contiguous in the pool, paged attention is dense
    attention: compare with torch's scaled_dot_product_attention in fp64
    ([CS349D-L3] sec. 3.2: mathematically the same as contiguous attention)."""
    w = wl.build_step("id", 11, [1, 7, 16, 33, 100], dtype=dtype, num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=d, block_size=bs, placement="identity")
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        start = int(w.block_tables[b, 0])
        # identity placement: the sequence's rows are one contiguous run
        kk = np_oracle.to_f64(k.reshape(-1, hkv, d)[start * bs:start * bs + L], dtype)
        vv = np_oracle.to_f64(v.reshape(-1, hkv, d)[start * bs:start * bs + L], dtype)
        qq = torch.from_numpy(np_oracle.to_f64(w.q[b], dtype))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, torch.from_numpy(kk).permute(1, 0, 2)[None], torch.from_numpy(vv).permute(1, 0, 2)[None],
            scale=w.scale, enable_gqa=True)[0, :, 0, :].numpy()
        for name, f in _both(c_oracle):
            out = f(w.q[b:b + 1], k, v, dtype, w.block_tables[b:b + 1], w.seq_lens[b:b + 1],
                    w.scale, hkv)
            np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12, err_msg=name)


# --- invariants the pages state -----------------------------------------------------

def _permute_physical(w, perm):
    """Move physical block i to perm[i]; remap tables and slots accordingly."""
    k = np.empty_like(w.k_pool)
    v = np.empty_like(w.v_pool)
    k[perm], v[perm] = w.k_pool, w.v_pool
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    bs = w.block_size
    slots = perm[w.slot_mapping // bs] * bs + w.slot_mapping % bs
    return k, v, bt, slots


@pytest.mark.parametrize("dtype", DTYPES)
def test_placement_permutation_invariance(c_oracle, dtype):
    """Any permutation of physical placement gives bit-identical outputs
    ([CS349D-L3] sec. 3.2: same tokens for sequential or shuffled blocks)."""
    w = wl.build_step("p", 21, [3, 16, 17, 64, 70], dtype=dtype, num_q_heads=8,
                      num_kv_heads=4, head_dim=32, block_size=8)
    k0, v0 = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k0, v0, w.k_new, w.v_new, w.slot_mapping)
    perm = np.random.default_rng(0).permutation(w.num_blocks)
    k1, v1, bt1, sl1 = _permute_physical(w, perm)
    np_oracle.append(k1, v1, w.k_new, w.v_new, sl1)
    for name, f in _both(c_oracle):
        o0 = f(w.q, k0, v0, dtype, w.block_tables, w.seq_lens, w.scale, 4)
        o1 = f(w.q, k1, v1, dtype, bt1, w.seq_lens, w.scale, 4)
        assert np.array_equal(o0, o1), name


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lse_merge_of_block_pieces_equals_whole(c_oracle, dtype):
    """Attention over a sequence cut at block boundaries into pieces, each piece
    attended on its own (a table of just its blocks) and the pieces combined by
    log-sum-exp weights (the combine of the split decode, [11868-L24] sec. 3.2:
    partial softmaxes merge exactly through their maxima and sums), equals the
    attention over the whole sequence.  The per-piece log-sum-exp of the
    scores is taken here from the gathered K in numpy; the outputs come from
    the oracles."""
    w = wl.build_step("lse", 11, [1, 37, 64, 150], dtype=dtype, num_q_heads=8, num_kv_heads=2,
                      head_dim=32, block_size=8)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    group = w.num_q_heads // w.num_kv_heads
    q = np_oracle.to_f64(w.q, dtype)
    bs = w.block_size
    for name, f in _both(c_oracle):
        whole = f(w.q, k, v, dtype, w.block_tables, w.seq_lens, w.scale, w.num_kv_heads)
        for b in range(w.batch):
            L = int(w.seq_lens[b])
            nb = -(-L // bs)
            cuts = sorted({0, nb // 3, (2 * nb) // 3, nb})
            outs, lses = [], []
            for j0, j1 in zip(cuts[:-1], cuts[1:]):
                if j1 == j0:
                    continue
                row = np.full((1, w.block_tables.shape[1]), -1, np.int32)
                row[0, :j1 - j0] = w.block_tables[b, j0:j1]
                n = min(L, j1 * bs) - j0 * bs
                outs.append(f(w.q[b:b + 1], k, v, dtype, row, np.array([n], np.int32), w.scale,
                              w.num_kv_heads)[0])
                K = np_oracle.to_f64(np_oracle.gather_kv(k, row[0], n), dtype)   # [n, Hkv, D]
                lse = np.empty(w.num_q_heads)
                for h in range(w.num_q_heads):
                    sc = w.scale * (K[:, h // group, :] @ q[b, h])
                    lse[h] = sc.max() + np.log(np.exp(sc - sc.max()).sum())
                lses.append(lse)
            lses = np.array(lses)                                    # [pieces, Hq]
            wts = np.exp(lses - lses.max(axis=0))
            merged = (wts[:, :, None] * np.array(outs)).sum(axis=0) / wts.sum(axis=0)[:, None]
            np.testing.assert_allclose(merged, whole[b], rtol=0, atol=1e-12,
                                       err_msg=f"{name} b={b}")


def test_shared_blocks_equal_private_copies(c_oracle):
    """Samples whose tables share refcounted prefix blocks give the same output
    as samples holding private copies of those blocks ([CS349D-L3] sec. 4.1:
    sharing only stores the duplicate data once)."""
    w = wl.shared_prefix(seed=4, prompts=2, prompt_len=40, n=3, max_divergent=9)
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.copy_blocks(k, v, w.pairs)
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    # private layout: every sample's blocks copied to fresh ids
    B, width = w.block_tables.shape
    used = [(b, j) for b in range(B) for j in range(width) if w.block_tables[b, j] >= 0]
    kp = np.concatenate([k, np.empty((len(used),) + k.shape[1:], k.dtype)])
    vp = np.concatenate([v, np.empty((len(used),) + v.shape[1:], v.dtype)])
    bt = np.full_like(w.block_tables, -1)
    for i, (b, j) in enumerate(used):
        kp[w.num_blocks + i], vp[w.num_blocks + i] = k[w.block_tables[b, j]], v[w.block_tables[b, j]]
        bt[b, j] = w.num_blocks + i
    assert len(set(bt[bt >= 0].tolist())) == len(used)
    shared = len(set(w.block_tables[w.block_tables >= 0].tolist()))
    assert shared < len(used)
    for name, f in _both(c_oracle):
        o_sh = f(w.q, k, v, "bf16", w.block_tables, w.seq_lens, w.scale, 8)
        o_pr = f(w.q, kp, vp, "bf16", bt, w.seq_lens, w.scale, 8)
        assert np.array_equal(o_sh, o_pr), name


def test_unwritten_rows_never_read(c_oracle):
    """Rows past the end of the last block and table entries past the last
    block hold NaN / -1; outputs stay finite ([CS349D-L3] sec. 3.2: only the
    written rows of the last block take part)."""
    w = wl.build_step("u", 8, [1, 2, 5, 13], dtype="f16", num_q_heads=2, num_kv_heads=2,
                      head_dim=16, block_size=8, table_width=6)
    assert (w.block_tables == -1).any()
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    for name, f in _both(c_oracle):
        assert np.isfinite(f(w.q, k, v, "f16", w.block_tables, w.seq_lens, w.scale, 2)).all(), name


# --- the two oracles against each other ------------------------------------------------

@pytest.mark.parametrize("builder", [
    lambda: wl.tiny(0),
    lambda: wl.opt13b_mha(1, batch=3, lo=1, hi=300),
    lambda: wl.llama3_8b_gqa(2, batch=6, median=60, hi=400),
    lambda: wl.long_context(3, batch=2, lo=500, hi=900, block_size=32),
    lambda: wl.shared_prefix(4, prompts=2, prompt_len=41, n=4, max_divergent=20),
])
def test_numpy_and_c_oracles_agree(c_oracle, builder):
    w = builder()
    k1, v1 = w.k_pool.copy(), w.v_pool.copy()
    k2, v2 = w.k_pool.copy(), w.v_pool.copy()
    assert np_oracle.copy_blocks(k1, v1, w.pairs) == 0
    assert c_oracle.copy_blocks(k2, v2, w.pairs, w.dtype) == 0
    assert np_oracle.append(k1, v1, w.k_new, w.v_new, w.slot_mapping) == 0
    assert c_oracle.append(k2, v2, w.k_new, w.v_new, w.slot_mapping, w.dtype) == 0
    assert k1.tobytes() == k2.tobytes() and v1.tobytes() == v2.tobytes()
    o1 = np_oracle.decode(w.q, k1, v1, w.dtype, w.block_tables, w.seq_lens, w.scale, w.num_kv_heads)
    o2, st = c_oracle.decode(w.q, k2, v2, w.dtype, w.block_tables, w.seq_lens, w.scale,
                             w.num_kv_heads, num_threads=3, return_status=True)
    assert st == 0
    assert np.isfinite(o1).all()
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


# --- append and copy: definitions and error counting ------------------------------------

def test_append_writes_rows_at_slots(c_oracle):
    w = wl.tiny(9)
    for impl in ("numpy", "c"):
        k, v = w.k_pool.copy(), w.v_pool.copy()
        bad = (np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping) if impl == "numpy"
               else c_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping, "f32"))
        assert bad == 0
        bs = w.block_size
        for i, s in enumerate(w.slot_mapping):
            assert np.array_equal(k[s // bs, s % bs], w.k_new[i])
            assert np.array_equal(v[s // bs, s % bs], w.v_new[i])
        changed = ~((k == w.k_pool) | (np.isnan(k) & np.isnan(w.k_pool))).all(axis=(2, 3))
        assert changed.sum() == len(w.slot_mapping)


def test_append_skips_padding_and_counts_out_of_range(c_oracle):
    w = wl.tiny(1)
    slots = w.slot_mapping.copy()
    slots[0] = -1
    slots[1] = w.num_blocks * w.block_size          # one past the end
    for impl in ("numpy", "c"):
        k, v = w.k_pool.copy(), w.v_pool.copy()
        bad = (np_oracle.append(k, v, w.k_new, w.v_new, slots) if impl == "numpy"
               else c_oracle.append(k, v, w.k_new, w.v_new, slots, "f32"))
        assert bad == 1
        ref_k = w.k_pool.copy()
        bs = w.block_size
        for i in (2, 3):
            ref_k[slots[i] // bs, slots[i] % bs] = w.k_new[i]
        assert ref_k.tobytes() == k.tobytes()


def test_copy_blocks_definition(c_oracle):
    rng = np.random.default_rng(0)
    k0 = rng.standard_normal((10, 4, 2, 8), dtype=np.float32)
    v0 = rng.standard_normal((10, 4, 2, 8), dtype=np.float32)
    pairs = np.array([[1, 7], [3, 2], [1, 9]], np.int32)
    for impl in ("numpy", "c"):
        k, v = k0.copy(), v0.copy()
        bad = (np_oracle.copy_blocks(k, v, pairs) if impl == "numpy"
               else c_oracle.copy_blocks(k, v, pairs, "f32"))
        assert bad == 0
        for blk in range(10):
            src = {7: 1, 2: 3, 9: 1}.get(blk, blk)
            assert np.array_equal(k[blk], k0[src]) and np.array_equal(v[blk], v0[src])
        k, v = k0.copy(), v0.copy()
        badpairs = np.array([[1, 10], [-1, 2], [4, 5]], np.int32)
        bad = (np_oracle.copy_blocks(k, v, badpairs) if impl == "numpy"
               else c_oracle.copy_blocks(k, v, badpairs, "f32"))
        assert bad == 2 and np.array_equal(k[5], k0[4]) and np.array_equal(k[2], k0[2])


def test_c_oracle_counts_invalid_table_entries(c_oracle):
    w = wl.tiny(2)
    bt = w.block_tables.copy()
    bt[1, 0] = w.num_blocks + 3
    k, v = w.k_pool.copy(), w.v_pool.copy()
    c_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping, "f32")
    out, st = c_oracle.decode(w.q, k, v, "f32", bt, w.seq_lens, w.scale, 4, return_status=True)
    assert st > 0 and np.isfinite(out).all()
    out2, st2 = c_oracle.decode(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 4,
                                return_status=True)
    assert st2 == 0
    assert np.array_equal(out[[0, 2, 3]], out2[[0, 2, 3]])
