"""GPU parity of cascade (shared-prefix) decode on 8-bit pools (FP8 E4M3 with
per-pool scales, INT8 with per-token-head scales).

Forked samples share their prompt's blocks ("Lecture 3", semidirectx.com
CS349D notes, sec. 4.1); the cascade reads each shared block once per group
and folds that partial into each member's log-sum-exp merge ("Lecture 24",
semidirectx.com CMU 11-868 notes, sec. 3.2).  The 8-bit codes convert
exactly, so the result must meet the 16-bit attention tolerance against the
oracle's fp64 attention over the dequantised values, and lie close to the
plain 8-bit decode's.  On block size 16 the prefix pass takes two blocks per
unit: an odd shared block count leaves the last shared block to the second
pass."""

import numpy as np
import pytest
import torch

from oracle import np_oracle
from parity import check_attention, check_same_attention, gpu_step_q8, oracle_step_q8
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CACHES = [("fp8_e4m3", 1.0, 1.0), ("fp8_e4m3", 0.25, 3.0), ("int8", 1.0, 1.0)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _check(w, cache, groups, sk=1.0, sv=1.0, seed=5, what="", p=None):
    p = p if p is not None else wl.q8_pools(w, cache, seed, sk, sv)
    gk, gv, gks, gvs, out, err = gpu_step_q8(w, p, groups=groups)
    assert err == 0, f"{what}: device error bits {err:#x}"
    _, _, _, _, ref = oracle_step_q8(w, p)
    rep = check_attention(out, ref, w.dtype, what)
    _, _, _, _, plain, err2 = gpu_step_q8(w, p, return_pools=False)
    assert err2 == 0
    check_same_attention(out, plain, w.dtype, f"{what}: cascade vs plain decode")
    return rep


@pytest.mark.parametrize("cache,sk,sv", CACHES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_q8_cascade_llama(cache, sk, sv, dtype):
    """Llama-3-8B-shaped GQA, block size 16: 2000-token prompts share 125
    blocks (62 two-block units + one block left to the second pass)."""
    w = wl.shared_prefix(41, prompts=3, prompt_len=2000, n=4, max_divergent=60, dtype=dtype)
    assert (w.groups[:, 2] == 125).all()
    print(_check(w, cache, w.groups, sk, sv, what=f"{cache} {dtype}"))


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("prompt_len,bs", [(2008, 16), (1000, 32), (136, 16), (31, 16)])
def test_q8_cascade_prompt_lengths(cache, prompt_len, bs):
    """A partly filled last shared block (copy-on-write), one block per unit
    at block size 32, a short prompt, and a prompt of one partial block (no
    whole unit to share: plain decode)."""
    w = wl.shared_prefix(42, prompts=2, prompt_len=prompt_len, n=4, max_divergent=50,
                         block_size=bs)
    print(_check(w, cache, w.groups, what=f"{cache} p{prompt_len} bs{bs}"))


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_cascade_fresh_fork(cache):
    """Every member still shares its whole context: the second pass attends
    only each member's own last block."""
    w = wl.shared_prefix(43, prompts=4, prompt_len=136, n=4, divergent=np.zeros(16, np.int64))
    print(_check(w, cache, w.groups, what=f"{cache} fresh fork"))


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("dtype,hq,hkv,bs,n", [
    ("f16", 16, 16, 16, 4),        # group 1: 16 members per sub-group
    ("bf16", 16, 8, 32, 6),        # group 2: 8 members per sub-group
    ("bf16", 64, 8, 16, 6),        # group 8: two members per sub-group
])
def test_q8_cascade_group_ratios(cache, dtype, hq, hkv, bs, n):
    w = wl.shared_prefix(44, prompts=2, prompt_len=600, n=n, max_divergent=40, block_size=bs,
                         num_q_heads=hq, num_kv_heads=hkv, dtype=dtype)
    print(_check(w, cache, w.groups, what=f"{cache} {dtype} {hq}/{hkv} bs{bs} n{n}"))


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_cascade_sub_groups_and_unused_groups(cache):
    """Groups of 6 at group size 4 (two sub-groups), a group whose sharing is
    turned off (0 blocks) and sequences outside every group."""
    w = wl.shared_prefix(45, prompts=3, prompt_len=500, n=6, max_divergent=40)
    g = w.groups.copy()
    g[1, 2] = 0
    g = g[[0, 1]]                                   # the third prompt's samples: ungrouped
    print(_check(w, cache, g, what=f"{cache} sub-groups"))


def test_q8_cascade_int8_v_scales_zero_then_jump():
    """INT8 V scales zero over the first two shared blocks and 100x larger on a
    later one: both passes weigh P by each token's V scale over the largest met
    so far, which starts at zero and rises mid-prefix."""
    w = wl.shared_prefix(46, prompts=2, prompt_len=900, n=4, max_divergent=30)
    p = wl.q8_pools(w, "int8", 12)
    vs = np.array(p.v_scales.cpu().numpy() if isinstance(p.v_scales, torch.Tensor)
                  else p.v_scales, copy=True)                  # [N, Hkv, bs]
    bt = np.asarray(w.block_tables)
    for first, size, blocks in np.asarray(w.groups):
        vs[bt[first, 0]] = 0.0
        vs[bt[first, 1]] = 0.0
        vs[bt[first, blocks // 2]] *= 100.0
    p.v_scales = vs
    print(_check(w, "int8", w.groups, what="int8 v scales", p=p))


def _effective(w, member, first, covered):
    """The workload with `member`'s first `covered` table entries replaced by
    those of `first` (the blocks the shared-prefix pass attends for it)."""
    h = wl.on_host(w)
    t = np.array(h.block_tables, copy=True)
    t[member, :covered] = t[first, :covered]
    h.block_tables = t
    return h


@pytest.mark.parametrize("cache", ["bf16", "fp8_e4m3", "int8"])
def test_cascade_second_pass_skips_exactly_the_prefix(cache):
    """The prefix pass attends the shared blocks through the group's first
    member's table; the second pass must start after them.  Member 1's shared
    entries are pointed at the other prompt's blocks: its cascade output must
    be attention over the first member's prefix and its own suffix (which
    plain decode of the same tables is not), so a second pass that re-read
    the prefix, or skipped a different count, fails.  40 full blocks of 16
    are shared: whole units for both the 16-bit (one block per unit) and the
    8-bit (two) second pass."""
    w = wl.shared_prefix(47, prompts=2, prompt_len=640, n=4, max_divergent=40)
    assert (np.asarray(w.groups)[:, 2] == 40).all()
    h = wl.on_host(w)
    t = np.array(h.block_tables, copy=True)
    t[1, :40] = t[4, :40]                      # member 1 now reads prompt 1's blocks
    h.block_tables = t
    eff = _effective(h, 1, 0, 40)              # what the cascade must attend for member 1
    if cache == "bf16":
        dev = torch.device("cuda")
        tv = lambda a: wl.value_to_torch(a, h.dtype, dev)
        outs = []
        for cascade in (True, False):
            pool = pagedkv.KVPool(tv(h.k_pool).clone(), tv(h.v_pool).clone())
            try:
                pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(h.pairs, dtype=np.int32)).to(dev))
                pool.append(tv(h.k_new), tv(h.v_new), torch.from_numpy(h.slot_mapping).to(dev))
                tables = torch.from_numpy(np.ascontiguousarray(h.block_tables)).to(dev)
                lens = torch.from_numpy(h.seq_lens).to(dev)
                if cascade:
                    g = torch.from_numpy(np.ascontiguousarray(h.groups, dtype=np.int32)).to(dev)
                    out = pool.decode_cascade(tv(h.q), tables, lens, h.scale, g)
                else:
                    out = pool.decode(tv(h.q), tables, lens, h.scale)
                torch.cuda.synchronize()
                assert pool.get_error() == 0
                outs.append(wl.value_to_numpy(out, h.dtype))
            finally:
                pool.close()
        from parity import oracle_step
        _, _, ref = oracle_step(eff)
        got, plain = outs
    else:
        p = wl.q8_pools(h, cache, 8)
        _, _, _, _, got, err = gpu_step_q8(h, p, return_pools=False, groups=h.groups)
        assert err == 0
        _, _, _, _, plain, err = gpu_step_q8(h, p, return_pools=False)
        assert err == 0
        _, _, _, _, ref = oracle_step_q8(eff, p)
    check_attention(got, ref, h.dtype, f"{cache} cascade with member 1's prefix from member 0")
    g64 = np_oracle.to_f64(got, h.dtype)[1]
    p64 = np_oracle.to_f64(plain, h.dtype)[1]
    assert np.abs(g64 - p64).max() > 1e-2, "member 1's output does not depend on the prefix pass"
