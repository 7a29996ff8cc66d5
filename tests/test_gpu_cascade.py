"""GPU parity of cascade (shared-prefix) decode: the same result as plain
decode and as the CPU oracle, with each shared block read once per group."""

import numpy as np
import pytest
import torch

from parity import check_attention, check_same_attention, oracle_step
from oracle import np_oracle
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _run(w, groups, cascade=True):
    """copy -> append -> decode (cascade or plain); returns out (raw), error bits."""
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone())
    try:
        pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev))
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
        q = tv(w.q)
        tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
        lens = torch.from_numpy(w.seq_lens).to(dev)
        if cascade:
            g = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).to(dev)
            out = pool.decode_cascade(q, tables, lens, w.scale, g)
        else:
            out = pool.decode(q, tables, lens, w.scale)
        torch.cuda.synchronize()
        return wl.value_to_numpy(out, w.dtype), pool.get_error()
    finally:
        pool.close()


def _check(w, groups, what):
    out, err = _run(w, groups)
    assert err == 0, f"{what}: device error bits {err:#x}"
    _, _, ref = oracle_step(w)
    rep = check_attention(out, ref, w.dtype, what)
    plain, _ = _run(w, groups, cascade=False)
    check_same_attention(out, plain, w.dtype, f"{what}: cascade vs plain decode")
    return rep


@pytest.mark.parametrize("prompt_len", [2000, 2008])
def test_shared_prefix_cascade(prompt_len):
    w = wl.shared_prefix(1, prompts=3, prompt_len=prompt_len, n=4, max_divergent=60)
    assert (w.groups[:, 2] >= 125).all()
    _check(w, w.groups, f"cascade p{prompt_len}")


def test_fresh_fork_cascade():
    w = wl.shared_prefix(2, prompts=4, prompt_len=136, n=4, divergent=np.zeros(16, np.int64))
    assert w.pairs.shape == (12, 2)
    _check(w, w.groups, "fresh fork cascade")


@pytest.mark.parametrize("bs", [16, 32])
def test_cascade_block_sizes(bs):
    w = wl.shared_prefix(3, prompts=2, prompt_len=700, n=4, max_divergent=90, block_size=bs)
    _check(w, w.groups, f"cascade bs{bs}")


def test_cascade_large_groups_and_ungrouped_sequences():
    """Groups of 6 (two sub-groups at group size 4), a group whose sharing is
    turned off (0 blocks), and sequences outside every group."""
    w = wl.shared_prefix(4, prompts=3, prompt_len=500, n=6, max_divergent=40)
    g = w.groups.copy()
    g[1, 2] = 0                           # decoded plainly
    g = g[[0, 1]]                         # the third prompt's samples are ungrouped
    _check(w, g, "large groups")


def test_cascade_group8_and_members_without_suffix():
    """Query/KV head ratio 8 (two members per sub-group); two sequences whose
    whole context is shared (nothing left for the per-sequence pass)."""
    base = wl.build_step("g8", 5, [300, 300, 411, 77], dtype="bf16", num_q_heads=16,
                         num_kv_heads=2, head_dim=128, block_size=16)
    w = base
    # make sequence 1 an exact copy of sequence 0 (same table, same length)
    w.block_tables[1] = w.block_tables[0]
    w.seq_lens[1] = w.seq_lens[0]
    w.slot_mapping[1] = -1                  # its append would duplicate sequence 0's
    shared = int(-(-int(w.seq_lens[0]) // 16))
    groups = np.array([[0, 2, shared]], np.int32)
    _check(w, groups, "group 8, empty suffix")


@pytest.mark.parametrize("dtype,hq,hkv,bs,n", [("f16", 16, 16, 16, 4),   # MHA (OPT-13B kind)
                                               ("bf16", 16, 8, 32, 6),   # ratio 2
                                               ("f16", 8, 8, 32, 17)])   # two sub-groups of 16
def test_cascade_group_ratios_1_and_2(dtype, hq, hkv, bs, n):
    """Query/KV head ratios 1 and 2: a prefix tile holds 16 and 8 members'
    query rows; 17 samples of one prompt at ratio 1 fill a sub-group and
    spill one member into a second."""
    w = wl.shared_prefix(8, prompts=3, prompt_len=600, n=n, max_divergent=50, block_size=bs,
                         num_q_heads=hq, num_kv_heads=hkv, dtype=dtype)
    assert (w.groups[:, 2] >= 600 // bs).all()
    _check(w, w.groups, f"cascade {dtype} {hq}/{hkv} bs{bs} n{n}")


def test_cascade_rejects_overlapping_groups_but_stays_correct():
    w = wl.shared_prefix(6, prompts=2, prompt_len=300, n=4, max_divergent=20)
    g = w.groups.copy()
    g[1, 0] = 2                           # overlaps group 0
    out, err = _run(w, g)
    assert err & pagedkv.KV_DEVERR_GROUP_RANGE
    _, _, ref = oracle_step(w)
    check_attention(out, ref, w.dtype, "bad groups")


def test_cascade_unsupported_shape_runs_plain_decode():
    w = wl.shared_prefix(7, prompts=2, prompt_len=100, n=4, max_divergent=10, block_size=8)
    _check(w, w.groups, "bs8 falls back to plain decode")


@pytest.mark.slow
def test_shared_prefix_cascade_full():
    for pl in (2000, 2008):
        w = wl.shared_prefix(0, prompt_len=pl, device="cuda")
        print(_check(w, w.groups, f"cascade full p{pl}"))
