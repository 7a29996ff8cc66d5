"""GPU: the decode's workspace may hold anything before a call.

The split kernel counts the pieces of each (sequence, KV head) cut across warp
ranges and the warp completing the count merges their partials by
log-sum-exp ("Lecture 24", semidirectx.com CMU 11-868 notes, sec. 3.2: the
merge must combine exactly the partials of one sequence).  A count read from
leftover memory would merge too early or never; each call's counters carry a
fresh random 64-bit tag, and a counter of another tag counts as zero.  Here
the workspace is filled with patterns that look like live counts -- int32
words 0, 1, ..., 4095 repeating (what a reused block table or length array
leaves), 64-bit words (e << 32) | j for small e and j, and the previous
call's own counters -- before every call, and the output must still match
the oracle: plain and cascade decode (the built-in-scratch call is covered in
the file collected last)."""

import numpy as np
import pytest
import torch

from parity import check_attention, oracle_step
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _fill(ws: torch.Tensor, pattern: str) -> None:
    n = ws.numel() // 8 * 8
    if pattern == "int32_ramp":
        words = torch.arange(n // 4, dtype=torch.int64, device=ws.device) % 4096
        ws[:n].view(torch.int32).copy_(words.to(torch.int32))
    elif pattern == "tagged64":
        i = torch.arange(n // 8, dtype=torch.int64, device=ws.device)
        e, j = (i // 7) % 64, i % 7
        ws[:n].view(torch.int64).copy_((e << 32) | j)
    else:
        ws.fill_(0xff)


def _inputs(w):
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(tv(w.k_pool).clone(), tv(w.v_pool).clone())
    pool.copy_blocks(torch.from_numpy(np.ascontiguousarray(w.pairs, dtype=np.int32)).to(dev))
    pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
    q = tv(w.q)
    tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    return pool, q, tables, lens


PATTERNS = ["int32_ramp", "tagged64", "ones"]


@pytest.mark.parametrize("w_fn", [
    lambda: wl.llama3_8b_gqa(31, batch=40, median=300, hi=2000),      # merged in the split kernel
    lambda: wl.long_context(32, batch=3, lo=3000, hi=9000, block_size=16),   # merge kernel
], ids=["split-merge", "merge-kernel"])
def test_plain_decode_with_stale_workspace(w_fn):
    w = w_fn()
    _, _, ref = oracle_step(w)
    pool, q, tables, lens = _inputs(w)
    try:
        ws = pool.workspace(w.batch, w.num_q_heads)
        for pat in PATTERNS:
            for rep in range(2):
                _fill(ws, pat)
                out = pool.decode(q, tables, lens, w.scale, workspace=ws)
                torch.cuda.synchronize()
                assert pool.get_error() == 0
                check_attention(wl.value_to_numpy(out, w.dtype), ref, w.dtype, f"{pat} #{rep}")
    finally:
        pool.close()


def test_cascade_decode_with_stale_workspace():
    w = wl.shared_prefix(33, prompts=3, prompt_len=1000, n=4, max_divergent=60)
    _, _, ref = oracle_step(w)
    pool, q, tables, lens = _inputs(w)
    try:
        groups = torch.from_numpy(np.ascontiguousarray(w.groups, dtype=np.int32)).to("cuda")
        need = pagedkv.paged_attention_cascade_workspace_size(pool.handle, w.batch, w.num_q_heads,
                                                               int(groups.shape[0]))
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        for pat in PATTERNS:
            for rep in range(2):
                _fill(ws, pat)
                out = pool.decode_cascade(q, tables, lens, w.scale, groups, workspace=ws)
                torch.cuda.synchronize()
                assert pool.get_error() == 0
                check_attention(wl.value_to_numpy(out, w.dtype), ref, w.dtype,
                                f"cascade {pat} #{rep}")
    finally:
        pool.close()
