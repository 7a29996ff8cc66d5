"""Seeded workload generators: determinism and the configured shapes (no GPU)."""

import numpy as np

from paged_kv_cache_68_gb300 import workloads as wl


def test_tiny_config_shape():
    w = wl.tiny(0)
    assert w.num_blocks == 64 and w.block_size == 4 and w.dtype == "f32"
    assert w.seq_lens.tolist() == [7, 18, 34, 51]
    assert w.q.shape == (4, 4, 64) and w.k_new.shape == (4, 4, 64)
    assert w.scale == 1.0 / 8.0
    assert w.info["blocks_used"] == 2 + 5 + 9 + 13
    used = w.block_tables[w.block_tables >= 0]
    assert len(set(used.tolist())) == used.size


def test_generation_is_deterministic():
    a, b = wl.opt13b_mha(3, batch=4, lo=10, hi=40), wl.opt13b_mha(3, batch=4, lo=10, hi=40)
    for f in ("k_pool", "v_pool", "q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens"):
        assert np.array_equal(getattr(a, f), getattr(b, f), equal_nan=True), f
    c = wl.opt13b_mha(4, batch=4, lo=10, hi=40)
    assert not np.array_equal(a.q, c.q)


def test_unwritten_rows_are_nan_and_slots_are_empty():
    w = wl.llama3_8b_gqa(1, batch=8, median=40, hi=200)
    kf = w.k_pool.reshape(-1, 8, 128)
    # the append's slots hold NaN (bf16 0x7FC0) until kv_append runs
    assert np.all(kf[w.slot_mapping] == 0x7FC0)
    nan_rows = int(np.all(kf == 0x7FC0, axis=(1, 2)).sum())
    assert nan_rows == kf.shape[0] - int((w.seq_lens - 1).sum())


def test_lognormal_lengths_clip_and_pool_factor():
    ctx = wl.llama3_context_lens(np.random.default_rng(0), 256)
    assert ctx.min() >= 16 and ctx.max() <= 8192
    assert 0.5 < np.median(ctx) / 1024 < 2.0
    w = wl.llama3_8b_gqa(0, batch=16, median=64, hi=300)
    assert np.array_equal(w.seq_lens - 1, wl.llama3_context_lens(np.random.default_rng(0), 16, 64, 1.0, 16, 300))
    need = sum(-(-int(L) // 16) for L in w.seq_lens)
    assert w.num_blocks == int(np.ceil(1.5 * need))


def test_long_context_block_sizes():
    for bs in (8, 16, 32):
        w = wl.long_context(0, batch=2, lo=100, hi=300, block_size=bs)
        assert w.block_size == bs and w.k_pool.shape[1] == bs
        assert all(len([x for x in row if x >= 0]) == -(-int(L) // bs)
                   for row, L in zip(w.block_tables, w.seq_lens))


def test_kv_bytes_per_token_match_the_pages_model_sizes():
    """Per token and layer, K + V take 4 KiB for the Llama-3-8B shape (8 KV heads
    x 128 dims x 2 bytes x 2) and 20 KiB for the OPT-13B shape (40 heads).  Over
    32 and 40 layers that is 128 KiB per token and 2 MiB per 16-token block
    ([11868-L24] reference answer 1) and 800 KiB per token and 12.5 MiB per
    block ([CS349D-L3] exercise 1)."""
    llama = wl.llama3_8b_gqa(0, batch=2, median=40, hi=100)
    opt = wl.opt13b_mha(0, batch=2, lo=10, hi=40)
    for w, layers, per_token, per_block in ((llama, 32, 128 << 10, 2 << 20),
                                            (opt, 40, 800 << 10, 25 << 19)):
        row = w.num_kv_heads * w.head_dim * w.elem_bytes * 2
        assert row * layers == per_token
        assert row * layers * w.block_size == per_block
        assert w.block_size == 16
