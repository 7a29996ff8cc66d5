"""Host block manager against the pages' worked examples (no GPU)."""

import numpy as np
import pytest

from conftest import golden
from oracle import np_oracle
from paged_kv_cache_68_gb300 import workloads as wl
from paged_kv_cache_68_gb300.block_manager import BlockManager, OutOfBlocks


def test_cs349d_demo1_block_tables():
    """Two requests, block size 8, 12 shuffled physical blocks: the printed
    tables, last-block fill and free counts at prefill and decode 1/5/12."""
    g = golden("cs349d_demo1_block_tables.json")
    bm = BlockManager(g["num_blocks"], g["block_size"], free_order=g["free_order"])
    bm.allocate_prompt("A", g["prefill"]["A"])
    bm.allocate_prompt("B", g["prefill"]["B"])
    done = 0
    for row in g["rows"]:
        while done < row["decode_steps"]:
            bm.append_slot("A")
            bm.append_slot("B")
            bm.check_invariant()
            done += 1
        for s in ("A", "B"):
            assert bm.lens[s] == row[f"{s}_tokens"], row["step"]
            assert bm.table(s) == row[f"{s}_table"], row["step"]
            fill = bm.lens[s] - (len(bm.table(s)) - 1) * g["block_size"]
            assert fill == row[f"{s}_last_fill"], row["step"]
        assert bm.num_free() == row["free"], row["step"]
    for s in g["slots"]:
        assert bm.slot_of(s["seq"], s["position"]) == s["slot"]


def test_cs349d_demo1_append_slots():
    """The slot handed out for A's 21st token (position 20) is 36 and for
    B's 25th token (position 24) is 8."""
    g = golden("cs349d_demo1_block_tables.json")
    bm = BlockManager(g["num_blocks"], g["block_size"], free_order=g["free_order"])
    bm.allocate_prompt("A", 20)
    bm.allocate_prompt("B", 24)
    assert bm.append_slot("A") == (36, None)
    assert bm.append_slot("B") == (8, None)


@pytest.mark.parametrize("case", golden("kwkr_manager_cases.json")["cases"], ids=lambda c: c["name"])
def test_kwkr_manager_cases(case):
    """The toy KVCacheManager's three test cases: on-demand blocks, gathering
    the scattered cache truncated at the sequence length, and OOM."""
    bm = BlockManager(case["num_blocks"], case["block_size"], pop="front")
    if "expect_error" in case:
        with pytest.raises(RuntimeError, match=case["expect_error"]):
            bm.allocate_prompt(0, case["prompt"])
        return
    bm.allocate_prompt(0, case["prompt"])
    assert len(bm.table(0)) == case["after_prefill"]["table_len"]
    if "free" in case["after_prefill"]:
        assert bm.num_free() == case["after_prefill"]["free"]
    for dec in case["decodes"]:
        while bm.lens[0] < dec["to_len"]:
            bm.append_slot(0)
        assert len(bm.table(0)) == dec["table_len"]
        if "free" in dec:
            assert bm.num_free() == dec["free"]
    pool = np.zeros((case["num_blocks"], case["block_size"], 1, case["head_dim"]), np.float32)
    for blk, val in zip(bm.table(0), case["fill"]):
        pool[blk] = val
    cache = np_oracle.gather_kv(pool, np.asarray(bm.table(0)), bm.lens[0])[:, 0]
    assert list(cache.shape) == case["gather_shape"]
    for r in case["gather_rows"]:
        assert np.all(cache[r["rows"][0]:r["rows"][1]] == r["value"])


def test_out_of_blocks_on_decode():
    bm = BlockManager(2, 4)
    bm.allocate_prompt(0, 8)
    with pytest.raises(OutOfBlocks, match="OOM"):
        bm.append_slot(0)


def _parallel_sampling(prompt_len, n, out_len, bs):
    """Prefill once, fork n - 1 samples, decode out_len tokens per sample
    step by step; return (blocks in use, copies made)."""
    bm = BlockManager(10_000, bs)
    bm.allocate_prompt(0, prompt_len)
    for i in range(1, n):
        bm.fork(0, i)
    for _ in range(out_len):
        for s in range(n):
            bm.append_slot(s)
            bm.check_invariant()
    return bm.num_blocks - bm.num_free(), bm.copies_made


def test_cs349d_ex2_parallel_sampling_blocks():
    """Prompt 62, n = 4, 40 output tokens, bs 8: 31 blocks shared vs 52
    private (40.4% saved), 3 copy-on-write copies; the granularity-free
    closed form gives 45.6%."""
    g = golden("cs349d_ex2_cow.json")
    used, copies = _parallel_sampling(g["prompt_len"], g["n"], g["output_len"], g["block_size"])
    assert used == g["blocks_shared"]
    assert copies == g["cow_copies"]
    private = g["n"] * -(-(g["prompt_len"] + g["output_len"]) // g["block_size"])
    assert private == g["blocks_private"]
    assert round(1 - used / private, 3) == g["saved_fraction"]
    n, lp, lo = g["n"], g["prompt_len"], g["output_len"]
    assert round((n - 1) * lp / (n * (lp + lo)), 3) == g["closed_form_saving"]


@pytest.mark.parametrize("case", golden("l24_answer4_cow_count.json")["cases"],
                         ids=lambda c: f"L{c['prompt_len']}_bs{c['block_size']}")
def test_l24_cow_count_rule(case):
    """n - 1 copies when the last prompt block is partial, 0 when full."""
    _, copies = _parallel_sampling(case["prompt_len"], case["n"], 3, case["block_size"])
    assert copies == case["copies"]


def test_refcount_invariant_random_ops():
    """[S06]: after every operation the number of tables holding a block
    equals its reference count (random fork / append / free sequence)."""
    rng = np.random.default_rng(0)
    bm = BlockManager(200, 4, free_order=rng.permutation(200).tolist(), pop="back")
    live, nxt = [], 0
    for _ in range(2000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                bm.allocate_prompt(nxt, int(rng.integers(0, 30)))
                live.append(nxt)
                nxt += 1
            elif op == 1:
                bm.fork(live[rng.integers(len(live))], nxt)
                live.append(nxt)
                nxt += 1
            elif op == 2:
                bm.append_slot(live[rng.integers(len(live))])
            else:
                bm.free_seq(live.pop(rng.integers(len(live))))
        except OutOfBlocks:
            pass
        bm.check_invariant()


def test_beam_fork_and_free_releases_only_at_zero():
    bm = BlockManager(20, 4)
    bm.allocate_prompt(0, 10)
    bm.fork(0, 1)
    bm.fork(1, 2)
    shared = bm.table(0)
    bm.free_seq(1)
    assert all(bm.ref[b] == 2 for b in shared) and bm.num_free() == 17
    bm.free_seq(0)
    bm.free_seq(2)
    assert bm.num_free() == 20
    bm.check_invariant()


def test_shared_prefix_workload_copy_counts():
    """2000-token prompts are whole blocks at bs 16: no copies; 2008-token
    prompts: n - 1 copies per prompt across history and step."""
    w0 = wl.shared_prefix(seed=0, prompts=4, prompt_len=2000, n=4, max_divergent=8)
    assert w0.info["history_copies"] == 0 and w0.pairs.shape == (0, 2)
    w1 = wl.shared_prefix(seed=0, prompts=4, prompt_len=2008, n=4, max_divergent=8)
    assert w1.info["history_copies"] + w1.info["step_copies"] == 4 * 3
    w2 = wl.shared_prefix(seed=0, prompts=4, prompt_len=2008, n=4,
                          divergent=np.zeros(16, np.int64))
    assert w2.info["history_copies"] == 0 and w2.pairs.shape == (12, 2)
    dsts = w2.pairs[:, 1]
    assert len(set(dsts.tolist())) == len(dsts) and not set(dsts) & set(w2.pairs[:, 0])


def test_expected_waste_is_under_one_block_and_independent_of_length():
    """Only a sequence's last block holds unused slots: [S06] "how to choose the
    block size" puts the expected waste at half a block per request, whatever
    its length.  Over every length residue the mean is exactly (bs - 1) / 2
    slots, the same for short and long sequences; growing a sequence token by
    token keeps it below one block."""
    for bs in (1, 4, 8, 16, 32):
        for base in (0, 10 * bs, 1000 * bs):
            m = BlockManager(num_blocks=4096, block_size=bs)
            waste = []
            for i, n in enumerate(range(base + 1, base + bs + 1)):
                m.allocate_prompt(i, n)
                waste.append(len(m.table(i)) * bs - n)
                m.free_seq(i)
            assert sum(waste) * 2 == (bs - 1) * bs, (bs, base)
        m = BlockManager(num_blocks=64, block_size=bs)
        m.allocate_prompt(0, 1)
        for _ in range(3 * bs):
            m.append_slot(0)
            assert 0 <= len(m.table(0)) * bs - m.lens[0] < bs
        m.check_invariant()
