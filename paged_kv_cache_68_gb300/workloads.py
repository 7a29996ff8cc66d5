"""Seeded synthetic decode-step workloads.

Every workload is one decode step of one layer: (1) the copy-on-write block
copies planned for this step, (2) the slot-mapped append of each sequence's
new K/V row, (3) PagedAttention decode of one query token per sequence over
its whole context including the new token.

This module only draws inputs; it holds none of the kernels' arithmetic.  It
is shared by the CUDA-side tests and benchmark and, as plain numpy arrays, by
the oracle.  Draw order for a seed is fixed: context lengths, placement
permutation, K rows, V rows, q, new K rows, new V rows (per-config extras are
documented on each builder).

Conventions (readings of the pages where they are silent):

* pool layout [num_blocks, block_size, Hkv, D], separate K and V pools;
* context lengths are drawn *before* the step; the step appends one token at
  position L and attends over L + 1 tokens (``seq_lens`` = L + 1);
* pool size is 1.5x the blocks the batch needs after the append, placed by a
  seeded random permutation of the physical ids (first-in first-out);
* rows never written (unused blocks, rows past the end of a last block, the
  new token's slot before the append) hold NaN, and block-table entries past
  a sequence's last block hold -1, so any read of them shows up;
* values are N(0, 1) drawn in float32 and rounded to the storage type
  (round to nearest even).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

from .block_manager import BlockManager

DTYPES = ("f32", "f16", "bf16")
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    k_pool: np.ndarray          # [N, bs, Hkv, D] raw, state before the step
    v_pool: np.ndarray
    q: np.ndarray               # [B, Hq, D] raw
    k_new: np.ndarray           # [T, Hkv, D] raw
    v_new: np.ndarray
    slot_mapping: np.ndarray    # int64 [T]
    block_tables: np.ndarray    # int32 [B, max_blocks_per_seq], -1 padded
    seq_lens: np.ndarray        # int32 [B], after the append
    pairs: np.ndarray           # int32 [P, 2] (src, dst), this step's copies
    info: Dict[str, float] = field(default_factory=dict)
    # sequences sharing prefix blocks: int32 [K, 3] (first member, members,
    # shared leading blocks), or None
    groups: Optional[np.ndarray] = None
    # chunked prefill: int32 [B + 1] query boundaries in the flattened q /
    # k_new / v_new / slot_mapping (None: one query per sequence)
    cu_seqlens: Optional[np.ndarray] = None

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    def kv_bytes(self) -> int:
        """K and V bytes attention must read: exact tokens, not padded blocks."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * 2 * self.elem_bytes

    def attention_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode: K/V + q + out + tables + lengths."""
        bs = self.block_size
        tbl = int(sum(-(-int(L) // bs) for L in self.seq_lens)) * 4
        qo = 2 * int(np.prod(tuple(self.q.shape))) * self.elem_bytes
        return self.kv_bytes() + qo + tbl + 4 * self.batch

    def append_bytes(self) -> int:
        n = int((self.slot_mapping >= 0).sum())
        return n * self.num_kv_heads * self.head_dim * self.elem_bytes * 2 * 2 + 8 * n

    def copy_bytes(self) -> int:
        blk = self.block_size * self.num_kv_heads * self.head_dim * self.elem_bytes
        return int(self.pairs.shape[0]) * blk * 2 * 2

    def step_bytes(self) -> int:
        return self.attention_bytes() + self.append_bytes() + self.copy_bytes()

    def attention_flops(self) -> int:
        """QK and PV multiply-adds (x2) over every (query, visible token) pair."""
        if self.cu_seqlens is None:
            return int(self.seq_lens.astype(np.int64).sum()) * self.num_q_heads * self.head_dim * 4
        pairs = 0
        for b in range(self.batch):
            C = int(self.cu_seqlens[b + 1] - self.cu_seqlens[b])
            L = int(self.seq_lens[b])
            # query i sees L - C + i + 1 tokens
            pairs += C * (L - C + 1) + C * (C - 1) // 2
        return pairs * self.num_q_heads * self.head_dim * 4


# -- element helpers ---------------------------------------------------------

def nan_fill(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.full(shape, np.nan, dtype=np.float32)
    if dtype == "f16":
        return np.full(shape, np.nan, dtype=np.float16)
    return np.full(shape, 0x7FC0, dtype=np.uint16)


def from_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage type (nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    u = x.view(np.uint32)
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def randn(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return from_f32(rng.standard_normal(shape, dtype=np.float32), dtype)


def _token_rows(table: List[int], n_tokens: int, bs: int) -> np.ndarray:
    """Pool rows (in the [N * bs] view) of positions 0..n_tokens-1."""
    t = np.asarray(table, dtype=np.int64)
    pos = np.arange(n_tokens, dtype=np.int64)
    return t[pos // bs] * bs + pos % bs


def _tables_array(bm: BlockManager, seq_ids: List[int], width: Optional[int]) -> np.ndarray:
    w = max([len(bm.tables[s]) for s in seq_ids] + [1])
    w = max(w, width or 0)
    out = np.full((len(seq_ids), w), -1, dtype=np.int32)
    for i, s in enumerate(seq_ids):
        t = bm.tables[s]
        out[i, :len(t)] = t
    return out


def _fill_rows(rng, pool_flat: np.ndarray, rows: np.ndarray, dtype: str):
    """pool_flat[rows] = N(0,1), drawn in chunks of about 2M values (bounded,
    reused host temporaries)."""
    inner = pool_flat.shape[1:]
    chunk = max(1, (1 << 21) // max(1, int(np.prod(inner))))
    for i in range(0, rows.shape[0], chunk):
        r = rows[i:i + chunk]
        pool_flat[r] = randn(rng, (r.shape[0],) + inner, dtype)


class _HostValues:
    """Values drawn with the numpy generator into host arrays (raw storage)."""

    def __init__(self, rng: np.random.Generator, dtype: str):
        self.rng, self.dtype = rng, dtype

    def nan(self, shape):
        return nan_fill(shape, self.dtype)

    def randn(self, shape):
        return randn(self.rng, shape, self.dtype)

    def fill_rows(self, pool, rows: np.ndarray):
        n = pool.shape[0] * pool.shape[1]
        _fill_rows(self.rng, pool.reshape(n, *pool.shape[2:]), rows, self.dtype)

    def set_rows(self, pool, rows: np.ndarray, values):
        pool.reshape(-1, *pool.shape[2:])[rows] = values


class _DeviceValues:
    """Values drawn on a CUDA device with a seeded torch generator: the same
    structure (lengths, placement, tables, slots) as the host backend, other
    N(0, 1) values, and no host copy of the pool.  Used for full-size runs."""

    def __init__(self, seed: int, dtype: str, device: str):
        import torch
        self.torch, self.device = torch, torch.device(device)
        self.tdtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(0x5EED0000 + int(seed))

    def nan(self, shape):
        return self.torch.full(tuple(shape), float("nan"), dtype=self.tdtype, device=self.device)

    def randn(self, shape):
        return self.torch.randn(tuple(shape), generator=self.gen, device=self.device,
                                dtype=self.torch.float32).to(self.tdtype)

    def fill_rows(self, pool, rows: np.ndarray):
        flat = pool.view(-1, *pool.shape[2:])
        idx = self.torch.from_numpy(np.ascontiguousarray(rows, dtype=np.int64)).to(self.device)
        chunk = 1 << 18
        for i in range(0, idx.shape[0], chunk):
            r = idx[i:i + chunk]
            flat[r] = self.randn((r.shape[0],) + tuple(pool.shape[2:]))

    def set_rows(self, pool, rows: np.ndarray, values):
        idx = self.torch.from_numpy(np.ascontiguousarray(rows, dtype=np.int64)).to(self.device)
        pool.view(-1, *pool.shape[2:])[idx] = values


def _values(seed: int, rng: np.random.Generator, dtype: str, device: Optional[str]):
    return _HostValues(rng, dtype) if device in (None, "cpu") else _DeviceValues(seed, dtype, device)


# -- generic independent-sequence step ------------------------------------------

def build_step(name: str, seed: int, context_lens, *, dtype: str, num_q_heads: int,
               num_kv_heads: int, head_dim: int, block_size: int,
               num_blocks: Optional[int] = None, pool_factor: float = 1.5,
               scale: Optional[float] = None, placement: str = "random",
               rng: Optional[np.random.Generator] = None,
               table_width: Optional[int] = None, device: Optional[str] = None) -> Workload:
    """One decode step over independent sequences with the given context lengths.

    ``placement``: "random" (seeded permutation of physical ids) or
    "identity" (ids in allocation order, i.e. each sequence contiguous).
    ``device``: None/"cpu" draws values into host numpy arrays; "cuda[:i]"
    draws them on that device into torch tensors (see ``_DeviceValues``).
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    B, bs = ctx.shape[0], block_size
    need = int(sum(-(-(int(L) + 1) // bs) for L in ctx))
    N = num_blocks if num_blocks is not None else max(need, int(math.ceil(pool_factor * need)))
    if N < need:
        raise ValueError(f"pool of {N} blocks cannot hold the {need} blocks needed")
    if placement == "random":
        order = rng.permutation(N).tolist()
    elif placement == "identity":
        # each sequence's blocks, the append's block included, consecutive ids
        nb_after = [-(-(int(L) + 1) // bs) for L in ctx]
        start = np.concatenate([[0], np.cumsum(nb_after)]).astype(np.int64)
        order = [int(start[b]) + j for b in range(B) for j in range(-(-int(ctx[b]) // bs))]
        order += [int(start[b]) + nb_after[b] - 1 for b in range(B)
                  if -(-int(ctx[b]) // bs) < nb_after[b]]
        order += list(range(int(start[-1]), N))
    else:
        raise ValueError(f"unknown placement {placement!r}")
    bm = BlockManager(N, bs, free_order=order)
    for b in range(B):
        bm.allocate_prompt(b, int(ctx[b]))
    inner = (num_kv_heads, head_dim)
    val = _values(seed, rng, dtype, device)
    k_pool = val.nan((N, bs) + inner)
    v_pool = val.nan((N, bs) + inner)
    rows = np.concatenate([_token_rows(bm.tables[b], int(ctx[b]), bs) for b in range(B)]
                          + [np.zeros(0, np.int64)])
    val.fill_rows(k_pool, rows)
    val.fill_rows(v_pool, rows)
    q = val.randn((B, num_q_heads, head_dim))
    k_new = val.randn((B,) + inner)
    v_new = val.randn((B,) + inner)
    slots, pairs = [], []
    for b in range(B):
        slot, cow = bm.append_slot(b)
        slots.append(slot)
        if cow:
            pairs.append(cow)
    bm.check_invariant()
    seq_lens = (ctx + 1).astype(np.int32)
    w = Workload(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=N,
        scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        k_pool=k_pool, v_pool=v_pool, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=np.asarray(slots, dtype=np.int64),
        block_tables=_tables_array(bm, list(range(B)), table_width),
        seq_lens=seq_lens, pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    w.info = {"seed": seed, "tokens": int(seq_lens.sum()), "mean_len": float(seq_lens.mean()) if B else 0.0,
              "max_len": int(seq_lens.max()) if B else 0, "blocks_used": N - bm.num_free(),
              "placement": placement}
    return w


# -- the five decode-step configurations ---------------------------------------

def tiny(seed: int = 0, device: Optional[str] = None) -> Workload:
    """4 sequences of {6, 17, 33, 50} tokens, 4 = 4 heads, D 64, bs 4, pool of
    64 blocks, fp32, scale 1/8; one appended token each."""
    return build_step("tiny", seed, [6, 17, 33, 50], dtype="f32", num_q_heads=4,
                      num_kv_heads=4, head_dim=64, block_size=4, num_blocks=64,
                      scale=1.0 / 8.0, device=device)


def opt13b_mha(seed: int = 0, batch: int = 64, lo: int = 128, hi: int = 2048,
               block_size: int = 16, device: Optional[str] = None) -> Workload:
    """OPT-13B-shaped MHA step: 40 = 40 heads, D 128, fp16, bs 16, batch 64,
    context ~ U[lo, hi] (integers, inclusive)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_step("opt13b_mha", seed, ctx, dtype="f16", num_q_heads=40, num_kv_heads=40,
                      head_dim=128, block_size=block_size, rng=rng, device=device)


def llama3_context_lens(rng: np.random.Generator, batch: int = 256, median: float = 1024.0,
                        sigma: float = 1.0, lo: int = 16, hi: int = 8192) -> np.ndarray:
    """clip(round(lognormal(ln median, sigma)), lo, hi): the first draw of the
    Llama-3-8B-shaped step."""
    return np.clip(np.rint(rng.lognormal(math.log(median), sigma, size=batch)), lo, hi).astype(np.int64)


def llama3_8b_gqa(seed: int = 0, batch: int = 256, median: float = 1024.0,
                  sigma: float = 1.0, lo: int = 16, hi: int = 8192,
                  block_size: int = 16, placement: str = "random",
                  device: Optional[str] = None) -> Workload:
    """Llama-3-8B-shaped GQA step: 32 query / 8 KV heads, D 128, bf16, bs 16,
    batch 256, context = clip(round(lognormal(ln median, sigma)), lo, hi)."""
    rng = np.random.default_rng(seed)
    ctx = llama3_context_lens(rng, batch, median, sigma, lo, hi)
    return build_step("llama3_8b_gqa", seed, ctx, dtype="bf16", num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=block_size, rng=rng, placement=placement,
                      device=device)


def long_context(seed: int = 0, batch: int = 8, lo: int = 32768, hi: int = 131072,
                 block_size: int = 16, device: Optional[str] = None) -> Workload:
    """Long-context step: 32 query / 8 KV heads, D 128, bf16, batch 8,
    context ~ U[lo, hi]; block size 8, 16 or 32."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_step(f"long_context_bs{block_size}", seed, ctx, dtype="bf16", num_q_heads=32,
                      num_kv_heads=8, head_dim=128, block_size=block_size, rng=rng,
                      device=device)


def chunked_prefill_step(name: str, seed: int, prefix_lens, chunk_lens, *, dtype: str,
                         num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                         pool_factor: float = 1.5, scale: Optional[float] = None,
                         rng: Optional[np.random.Generator] = None,
                         device: Optional[str] = None) -> Workload:
    """One chunked-prefill step: request b has prefix_lens[b] tokens cached
    and a chunk of chunk_lens[b] new tokens (1 = a decode request).  The step
    appends the chunk's K/V through its slots (blocks taken on demand, as
    decode does) and attends each of its chunk_lens[b] queries causally over
    the prefix and the chunk.  Draw order: placement permutation, cached K
    rows, cached V rows, q, new K rows, new V rows."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    pre = np.asarray(prefix_lens, dtype=np.int64)
    chk = np.asarray(chunk_lens, dtype=np.int64)
    B, bs = pre.shape[0], block_size
    need = int(sum(-(-int(pre[b] + chk[b]) // bs) for b in range(B)))
    N = max(need, int(math.ceil(pool_factor * need)))
    bm = BlockManager(N, bs, free_order=rng.permutation(N).tolist())
    for b in range(B):
        bm.allocate_prompt(b, int(pre[b]))
    inner = (num_kv_heads, head_dim)
    val = _values(seed, rng, dtype, device)
    k_pool = val.nan((N, bs) + inner)
    v_pool = val.nan((N, bs) + inner)
    rows = np.concatenate([_token_rows(bm.tables[b], int(pre[b]), bs) for b in range(B)]
                          + [np.zeros(0, np.int64)])
    val.fill_rows(k_pool, rows)
    val.fill_rows(v_pool, rows)
    T = int(chk.sum())
    q = val.randn((T, num_q_heads, head_dim))
    k_new = val.randn((T,) + inner)
    v_new = val.randn((T,) + inner)
    slots = []
    for b in range(B):
        for _ in range(int(chk[b])):
            slot, cow = bm.append_slot(b)
            assert cow is None
            slots.append(slot)
    bm.check_invariant()
    seq_lens = (pre + chk).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(chk)]).astype(np.int32)
    w = Workload(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=N,
        scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        k_pool=k_pool, v_pool=v_pool, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=np.asarray(slots, dtype=np.int64),
        block_tables=_tables_array(bm, list(range(B)), None),
        seq_lens=seq_lens, pairs=np.zeros((0, 2), np.int32), cu_seqlens=cu)
    w.info = {"seed": seed, "tokens": int(seq_lens.sum()), "query_tokens": T,
              "max_query_len": int(chk.max()) if B else 0}
    return w


def chunked_prefill(seed: int = 0, batch: int = 16, chunk: int = 256, max_prefix: int = 3840,
                    decodes: int = 0, block_size: int = 16,
                    device: Optional[str] = None) -> Workload:
    """Chunked prefill, Llama-3-8B GQA shape (bf16, bs 16): ``batch`` requests
    with a chunk of ``chunk`` prompt tokens each after a cached prefix of
    U[0, max_prefix] tokens (the earlier chunks of the same prompt), plus
    ``decodes`` decode requests (one query, lognormal context as the
    Llama-3-8B step) packed into the same batch."""
    rng = np.random.default_rng(seed)
    pre = rng.integers(0, max_prefix, size=batch, endpoint=True)
    chk = np.full(batch, chunk, np.int64)
    if decodes:
        pre = np.concatenate([pre, llama3_context_lens(rng, decodes)])
        chk = np.concatenate([chk, np.ones(decodes, np.int64)])
    return chunked_prefill_step("chunked_prefill", seed, pre, chk, dtype="bf16", num_q_heads=32,
                                num_kv_heads=8, head_dim=128, block_size=block_size, rng=rng,
                                device=device)


def shared_prefix(seed: int = 0, prompts: int = 32, prompt_len: int = 2000, n: int = 4,
                  max_divergent: int = 256, block_size: int = 16,
                  divergent: Optional[np.ndarray] = None, pool_factor: float = 1.5,
                  device: Optional[str] = None, num_q_heads: int = 32, num_kv_heads: int = 8,
                  dtype: str = "bf16") -> Workload:
    """Parallel sampling over shared prompts (Llama-3-8B GQA shape, bf16, by
    default; other head counts and 16-bit types for the cascade's shapes).

    Each prompt is prefilled once and forked into n samples (every prompt
    block has reference count n).  Sample s then holds d_s ~ U[0,
    max_divergent] divergent tokens, replayed one decode step at a time over
    all samples, each write into a shared block doing copy-on-write.  The
    measured step appends one token per sample; a sample still sharing a
    partial last block copies it first, and those (src, dst) pairs are this
    step's ``pairs``.  Draw order: d_s, permutation, prompt K, prompt V,
    divergent K, divergent V, q, new K, new V.
    """
    rng = np.random.default_rng(seed)
    S, bs = prompts * n, block_size
    d = (rng.integers(0, max_divergent, size=S, endpoint=True) if divergent is None
         else np.asarray(divergent, dtype=np.int64))
    per_prompt = -(-prompt_len // bs)
    priv = sum(-(-(prompt_len + int(x) + 1) // bs) - prompt_len // bs for x in d)
    need = prompts * per_prompt + priv
    N = int(math.ceil(pool_factor * need))
    bm = BlockManager(N, bs, free_order=rng.permutation(N).tolist())
    for p in range(prompts):
        bm.allocate_prompt(p * n, prompt_len)
        for i in range(1, n):
            bm.fork(p * n, p * n + i)
    for k in range(int(d.max()) if S else 0):          # history, step by step
        for s in range(S):
            if d[s] > k:
                bm.append_slot(s)
    history_copies = bm.copies_made
    bm.check_invariant()
    inner = (num_kv_heads, 128)
    val = _values(seed, rng, dtype, device)
    k_pool = val.nan((N, bs) + inner)
    v_pool = val.nan((N, bs) + inner)
    pk = val.randn((prompts, prompt_len) + inner)
    pv = val.randn((prompts, prompt_len) + inner)
    tot_div = int(d.sum())
    dk = val.randn((tot_div,) + inner)
    dv = val.randn((tot_div,) + inner)
    off = 0
    for s in range(S):
        p = s // n
        rows = _token_rows(bm.tables[s], prompt_len + int(d[s]), bs)
        val.set_rows(k_pool, rows[:prompt_len], pk[p])
        val.set_rows(v_pool, rows[:prompt_len], pv[p])
        val.set_rows(k_pool, rows[prompt_len:], dk[off:off + int(d[s])])
        val.set_rows(v_pool, rows[prompt_len:], dv[off:off + int(d[s])])
        off += int(d[s])
    q = val.randn((S, num_q_heads, 128))
    k_new = val.randn((S,) + inner)
    v_new = val.randn((S,) + inner)
    slots, pairs = [], []
    for s in range(S):
        slot, cow = bm.append_slot(s)
        slots.append(slot)
        if cow:
            pairs.append(cow)
    bm.check_invariant()
    seq_lens = np.asarray([bm.lens[s] for s in range(S)], dtype=np.int32)
    w = Workload(name=f"shared_prefix_p{prompt_len}", dtype=dtype, num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads,
                 head_dim=128, block_size=bs, num_blocks=N, scale=1.0 / math.sqrt(128),
                 k_pool=k_pool, v_pool=v_pool, q=q, k_new=k_new, v_new=v_new,
                 slot_mapping=np.asarray(slots, dtype=np.int64),
                 block_tables=_tables_array(bm, list(range(S)), None), seq_lens=seq_lens,
                 pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    groups = np.asarray([[p * n, n, bm.shared_prefix_blocks(range(p * n, p * n + n))]
                         for p in range(prompts)], dtype=np.int32).reshape(-1, 3)
    w.groups = groups
    unique_tokens = prompts * prompt_len + int(seq_lens.sum()) - S * prompt_len
    w.info = {"seed": seed, "tokens": int(seq_lens.sum()), "unique_tokens": unique_tokens,
              "history_copies": history_copies, "step_copies": len(pairs),
              "blocks_used": N - bm.num_free(), "mean_len": float(seq_lens.mean())}
    return w


CONFIGS = {
    "tiny": tiny,
    "opt13b_mha": opt13b_mha,
    "llama3_8b_gqa": llama3_8b_gqa,
    "shared_prefix": shared_prefix,
    "long_context": long_context,
}


# -- moving a workload between host arrays and device tensors --------------------

_VALUE_FIELDS = ("k_pool", "v_pool", "q", "k_new", "v_new")


def _torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def value_to_torch(a, dtype: str, device):
    """Raw host array (or tensor) -> torch tensor of the storage dtype on device."""
    import torch
    if isinstance(a, torch.Tensor):
        return a.to(device)
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def value_to_numpy(t, dtype: str) -> np.ndarray:
    """Torch tensor (any device) or host array -> raw host array (None stays None:
    an 8-bit step drops its 16-bit pools)."""
    if t is None or isinstance(t, np.ndarray):
        return t
    import torch
    t = t.detach().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def on_host(w: Workload) -> Workload:
    """A copy of ``w`` whose value arrays are host numpy arrays."""
    import copy
    h = copy.copy(w)
    for f in _VALUE_FIELDS:
        setattr(h, f, value_to_numpy(getattr(w, f), w.dtype))
    return h


# -- 8-bit pools ---------------------------------------------------------------

@dataclass
class Q8Pools:
    """An 8-bit pool of a workload's geometry: uint8 codes [N, bs, Hkv, D] and,
    for INT8, fp32 scales [N, Hkv, bs]; per-pool scales for FP8."""
    cache: str
    k_codes: object
    v_codes: object
    k_scales: object = None
    v_scales: object = None
    k_scale: float = 1.0
    v_scale: float = 1.0

    def row_bytes(self, w: "Workload") -> int:
        """Stored bytes of one token's K and V rows: one byte per element plus
        the INT8 scales (one fp32 per KV head, for K and for V)."""
        return w.num_kv_heads * w.head_dim * 2 + (8 * w.num_kv_heads if self.cache == "int8" else 0)

    def kv_bytes(self, w: "Workload") -> int:
        """Bytes attention reads for K and V (exact tokens)."""
        return int(w.seq_lens.astype(np.int64).sum()) * self.row_bytes(w)

    def attention_bytes(self, w: "Workload") -> int:
        bs = w.block_size
        tbl = int(sum(-(-int(L) // bs) for L in w.seq_lens)) * 4
        qo = 2 * int(np.prod(tuple(w.q.shape))) * w.elem_bytes
        return self.kv_bytes(w) + qo + tbl + 4 * w.batch

    def append_bytes(self, w: "Workload") -> int:
        """16-bit rows read, codes (and scales) written, slots read."""
        n = int((np.asarray(w.slot_mapping) >= 0).sum())
        return n * (w.num_kv_heads * w.head_dim * w.elem_bytes * 2 + self.row_bytes(w) + 8)

    def copy_bytes(self, w: "Workload") -> int:
        return int(w.pairs.shape[0]) * w.block_size * self.row_bytes(w) * 2

    def step_bytes(self, w: "Workload") -> int:
        return self.attention_bytes(w) + self.append_bytes(w) + self.copy_bytes(w)


def q8_pools(w: "Workload", cache: str, seed: int, k_scale: float = 1.0,
             v_scale: float = 1.0) -> Q8Pools:
    """Seeded codes for the rows ``w``'s pools hold (rows that are NaN in the
    16-bit pools stay unreadable: E4M3 NaN codes 0x7F, INT8 scales NaN).

    FP8: N(0, 1) draws cast to E4M3 by torch (values like stored K/V);
    INT8: codes round(N(0, 42)) clipped to [-127, 127], scales U(0.01, 0.04)
    per (block, head, row).  On the device of ``w`` (numpy or CUDA torch)."""
    import torch
    dev = w.k_pool.device if isinstance(w.k_pool, torch.Tensor) else torch.device("cpu")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0x0C8D0000 + int(seed))
    shape = tuple(w.k_pool.shape)
    N, bs, H, D = shape

    def filled(pool):
        t = pool if isinstance(pool, torch.Tensor) else value_to_torch(pool, w.dtype, dev)
        return ~torch.isnan(t.reshape(N, bs, H, D)[..., 0].float())     # [N, bs, H]

    out = []
    for pool in (w.k_pool, w.v_pool):
        live = filled(pool)
        if cache == "fp8_e4m3":
            x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
            codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
            codes = torch.where(live[..., None], codes, torch.full_like(codes, 0x7F))
            scales = None
        elif cache == "int8":
            x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * 42.0
            codes = x.round().clamp(-127, 127).to(torch.int8).view(torch.uint8)
            sc = torch.rand((N, H, bs), generator=gen, device=dev, dtype=torch.float32) * 0.03 + 0.01
            scales = torch.where(live.permute(0, 2, 1), sc, torch.full_like(sc, float("nan")))
        else:
            raise ValueError(f"unknown cache format {cache!r}")
        out.append((codes.contiguous(), None if scales is None else scales.contiguous()))
    if dev.type == "cpu":
        out = [(c.numpy(), None if s is None else s.numpy()) for c, s in out]
    return Q8Pools(cache, out[0][0], out[1][0], out[0][1], out[1][1],
                   k_scale if cache == "fp8_e4m3" else 1.0, v_scale if cache == "fp8_e4m3" else 1.0)
