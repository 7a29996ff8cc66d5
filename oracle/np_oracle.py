"""numpy fp64 oracle for slot-mapped append, block copy and PagedAttention decode.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Sources (cited by page title and section):

* [CS349D-L3] "Lecture 3: memory and prefix reuse in serving engines -- vLLM
  PagedAttention and SGLang RadixAttention" (semidirectx.com, CS349D notes):
  sec. 3.1 block tables and on-demand blocks; sec. 3.2 attention over scattered
  blocks (one softmax over all positions of all blocks, only the written rows
  of the last block); sec. 4.1 copy-on-write.
* [11868-L24] "Lecture 24: PagedAttention and vLLM" (semidirectx.com, CMU
  11-868 notes): sec. 3.2 paged and contiguous attention agree up to rounding.
* [RL-Part3] "Part 3: single node" (random-liu.github.io book): ch. 9 sec. 1
  grouped-query heads; ch. 11 sec. 3 block table [max_num_reqs,
  max_num_blocks_per_req]; ch. 13 sec. 1 slot_mapping, kv_cache[slot] = new_kv.
* [S06] "S06 memory and KV cache: PagedAttention" (llminference.xinbetween.com):
  "Implementation" -- pool layout [num_blocks, block_size, n_kv_heads, head_dim]
  and the gather-then-softmax attention; the kwkr.cn blog's toy
  ``KVCacheManager.get_physical_cache`` gathers the same way.

Data conventions: a pool is a numpy array [num_blocks, block_size, Hkv, D]
holding the raw elements -- float32 for "f32", float16 for "f16", uint16 bit
patterns for "bf16".  q and new K/V rows use the same representation.
"""

from __future__ import annotations

import numpy as np

KV_DTYPES = ("f32", "f16", "bf16")


def to_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw elements to float64.

    bf16 is the top half of a binary32: shift the 16 bits up and reinterpret.
    """
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(raw, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        with np.errstate(invalid="ignore"):
            return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def append(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray,
           v_new: np.ndarray, slot_mapping: np.ndarray) -> int:
    """kv_cache[slot_mapping[i]] = new_kv for every token i, in place.

    [RL-Part3] ch. 13 sec. 1: the scheduler hands the GPU one absolute slot per
    new token; a slot is block * block_size + offset ([CS349D-L3] sec. 3.1), so
    it is a row index of the pool viewed as [num_blocks * block_size, Hkv, D].
    Negative slots are padding (skipped); slots past the pool are skipped and
    counted.  Returns the count of out-of-range slots.
    """
    nb, bs = k_pool.shape[0], k_pool.shape[1]
    kflat = k_pool.reshape(nb * bs, *k_pool.shape[2:])
    vflat = v_pool.reshape(nb * bs, *v_pool.shape[2:])
    bad = 0
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        if slot >= nb * bs:
            bad += 1
            continue
        kflat[slot] = k_new[i]
        vflat[slot] = v_new[i]
    return bad


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs: np.ndarray) -> int:
    """For each (src, dst) pair in order, copy block src over block dst.

    [CS349D-L3] sec. 4.1: a write into a block whose reference count exceeds
    one first allocates a new block, copies the content, remaps the table and
    then writes; sec. 3.2: these small copies are batched into one launch.
    Pairs naming a block outside the pool are skipped and counted.
    """
    nb = k_pool.shape[0]
    bad = 0
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= src < nb and 0 <= dst < nb):
            bad += 1
            continue
        k_pool[dst] = k_pool[src].copy()
        v_pool[dst] = v_pool[src].copy()
    return bad


def gather_kv(pool: np.ndarray, table_row: np.ndarray, seq_len: int) -> np.ndarray:
    """Assemble the logically contiguous cache [seq_len, Hkv, D] of a sequence.

    Walks the block table: logical block j lives in physical block
    table_row[j]; the last block contributes only its written rows
    ([CS349D-L3] sec. 3.2; [S06] "Implementation").  Raw elements are returned
    unconverted (the kwkr.cn toy manager's get_physical_cache does the same
    concatenate-and-truncate).
    """
    nb, bs = pool.shape[0], pool.shape[1]
    nblk = -(-seq_len // bs)
    ids = [int(table_row[j]) for j in range(nblk)]
    if any(not 0 <= i < nb for i in ids):
        raise ValueError("block table names a block outside the pool")
    blocks = [pool[i] for i in ids]
    if not blocks:
        return pool[:0, 0]
    return np.concatenate(blocks, axis=0)[:seq_len]


def decode(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, dtype: str,
           block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
           num_kv_heads: int) -> np.ndarray:
    """PagedAttention decode: out[b, h] = softmax(scale * q[b, h] K^T) V.

    For each sequence b and KV head g: gather K, V of positions 0..L-1
    through the block table, decode to fp64, and for the query heads of group
    g ([RL-Part3] ch. 9 sec. 1; contiguous groups, h // (Hq / Hkv) = g)
    compute the scores, a max-subtracted softmax over all L positions, and
    the weighted sum of V.  L = 0 gives zeros.  Returns float64 [B, Hq, D].
    """
    B, Hq, D = q.shape
    if Hq % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = Hq // num_kv_heads
    qf = to_f64(q, dtype)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        K = to_f64(gather_kv(k_pool, block_tables[b], L), dtype)   # [L, Hkv, D]
        V = to_f64(gather_kv(v_pool, block_tables[b], L), dtype)
        for g in range(num_kv_heads):
            heads = slice(g * group, (g + 1) * group)
            s = scale * (qf[b, heads] @ K[:, g, :].T)                 # [group, L]
            s = s - s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w = w / w.sum(axis=1, keepdims=True)
            out[b, heads] = w @ V[:, g, :]
    return out
