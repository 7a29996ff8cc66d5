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


# ------------------------------------------------------- 8-bit KV cache --
#
# "Part 3: single node" (random-liu.github.io), ch. 10 (KV cache quantisation,
# FP8/INT8): a new token's K and V are scaled and rounded from 16 to 8 bits
# before they are stored, and the attention turns them back into wider
# numbers when it reads them (sec. 1).  INT8 maps values to integers by a scale
# and a rounding, with the scale kept per token (or per channel) to stay
# accurate (sec. 3); FP8 keeps sign, exponent and mantissa, i.e. it is a
# shorter float (sec. 3).  Readings where the chapter is silent:
#
# * FP8 is E4M3 (4 exponent bits, bias 7, 3 mantissa bits, no infinities, only
#   S.1111.111 is NaN, largest finite 448) with one scale per pool for K and
#   one for V: code = E4M3(x / scale), value = decode(code) * scale.  Values
#   round to nearest, ties to even; anything beyond 448 (infinities included)
#   saturates to +-448; NaN stays NaN (code 0x7F).
# * INT8 keeps one scale per (token, KV head), decided when the token is
#   written: amax = max |x| over the head's D elements, inv = 127 / amax and
#   scale = amax / 127 (both fp32 divisions), code = rint(x * inv) (fp32
#   product, ties to even) clipped to [-127, 127]; value = code * scale.  An
#   all-zero row has scale 0 and codes 0; a row holding a NaN or an infinity
#   gets scale NaN and codes 0.
# * Every quantisation decision is taken in fp32 (the precision the CUDA
#   kernel takes it in); dequantisation and the attention are fp64.
# * Layout: codes [num_blocks, block_size, Hkv, D] (one byte each, the 16-bit
#   pool layout), INT8 scales [num_blocks, Hkv, block_size] fp32.

KV_CACHE_FORMATS = ("fp8_e4m3", "int8")
E4M3_MAX = 448.0


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode E4M3 bytes: (-1)^s * 2^(e - 7) * (1 + m/8) for e >= 1,
    (-1)^s * 2^-6 * m/8 for e = 0; e = 15, m = 7 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


def f32_to_e4m3(t: np.ndarray) -> np.ndarray:
    """Round fp32 values to E4M3 codes (nearest, ties to even, saturating)."""
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    out = np.zeros(t.shape, dtype=np.uint8)
    flat_t, flat_o = t.reshape(-1), out.reshape(-1)
    for i, x in enumerate(flat_t):
        if np.isnan(x):
            flat_o[i] = 0x7F
            continue
        sign = 0x80 if np.signbit(x) else 0
        a = min(abs(x), E4M3_MAX)
        if a == 0.0:
            flat_o[i] = sign
            continue
        E = max(int(np.floor(np.log2(a))), -6)      # binade; below 2^-6 the grid is 2^-9
        # the binade's grid spacing is 2^(E - 3); x / spacing is exact in fp64
        m = float(np.rint(a / 2.0 ** (E - 3)))        # ties to even
        v = m * 2.0 ** (E - 3)
        if v == 0.0:
            flat_o[i] = sign
            continue
        E2 = int(np.floor(np.log2(v)))
        if E2 < -6:
            flat_o[i] = sign | int(round(v / 2.0 ** -9))
        else:
            flat_o[i] = sign | ((E2 + 7) << 3) | (int(round(v / 2.0 ** (E2 - 3))) - 8)
    return out


def int8_quantize(rows: np.ndarray):
    """Per-row INT8 quantisation of fp32 rows [..., D] -> (int8 codes, fp32 scales)."""
    x = np.asarray(rows, dtype=np.float32)
    codes = np.zeros(x.shape, dtype=np.int8)
    scales = np.zeros(x.shape[:-1], dtype=np.float32)
    flat_x = x.reshape(-1, x.shape[-1])
    flat_c = codes.reshape(-1, x.shape[-1])
    flat_s = scales.reshape(-1)
    for r in range(flat_x.shape[0]):
        row = flat_x[r]
        if not np.all(np.isfinite(row)):
            flat_s[r] = np.float32(np.nan)
            continue
        amax = np.max(np.abs(row))
        if amax == 0:
            continue
        inv = np.float32(127.0) / amax                  # fp32 division
        t = (row * inv).astype(np.float32)              # fp32 products
        flat_c[r] = np.clip(np.rint(t), -127, 127).astype(np.int8)
        flat_s[r] = amax / np.float32(127.0)
    return codes, scales


def _quantize_rows(x32: np.ndarray, fmt: str, fp8_scale: float):
    if fmt == "fp8_e4m3":
        t = (x32 / np.float32(fp8_scale)).astype(np.float32)
        return f32_to_e4m3(t), None
    if fmt == "int8":
        codes, scales = int8_quantize(x32)
        return codes.view(np.uint8), scales
    raise ValueError(f"unknown KV cache format {fmt!r}")


def append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, in_dtype: str,
              slot_mapping, fmt: str, fp8_k_scale: float = 1.0, fp8_v_scale: float = 1.0) -> int:
    """Quantise each new token's K and V rows and store them at its slot.

    k_codes/v_codes: uint8 [nb, bs, Hkv, D]; k_scales/v_scales: fp32
    [nb, Hkv, bs] for INT8 (None for FP8).  k_new/v_new: raw [T, Hkv, D] in
    ``in_dtype``.  Slots as in ``append``.  Returns the out-of-range count.
    """
    nb, bs = k_codes.shape[0], k_codes.shape[1]
    bad = 0
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        if slot >= nb * bs:
            bad += 1
            continue
        blk, off = divmod(int(slot), bs)
        for codes, scales, new, s8 in ((k_codes, k_scales, k_new, fp8_k_scale),
                                       (v_codes, v_scales, v_new, fp8_v_scale)):
            x32 = to_f64(new[i], in_dtype).astype(np.float32)        # [Hkv, D]
            c, sc = _quantize_rows(x32, fmt, s8)
            codes[blk, off] = c
            if sc is not None:
                scales[blk, :, off] = sc
    return bad


def copy_blocks_q8(k_codes, v_codes, k_scales, v_scales, pairs) -> int:
    """``copy_blocks`` for an 8-bit pool: codes and (INT8) scales move together."""
    nb = k_codes.shape[0]
    bad = 0
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= src < nb and 0 <= dst < nb):
            bad += 1
            continue
        for a in (k_codes, v_codes, k_scales, v_scales):
            if a is not None:
                a[dst] = a[src].copy()
    return bad


def dequantize(codes: np.ndarray, scales, fmt: str, fp8_scale: float = 1.0) -> np.ndarray:
    """fp64 values of an 8-bit pool [nb, bs, Hkv, D] (scales [nb, Hkv, bs])."""
    if fmt == "fp8_e4m3":
        return e4m3_to_f64(codes) * float(fp8_scale)
    if fmt == "int8":
        c = np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)
        s = np.asarray(scales, dtype=np.float32).astype(np.float64).transpose(0, 2, 1)
        return c * s[..., None]
    raise ValueError(f"unknown KV cache format {fmt!r}")


def decode_q8(q, in_dtype: str, k_codes, v_codes, k_scales, v_scales, fmt: str,
              block_tables, seq_lens, scale: float, num_kv_heads: int,
              fp8_k_scale: float = 1.0, fp8_v_scale: float = 1.0) -> np.ndarray:
    """PagedAttention decode over an 8-bit pool: the pool's values are the
    dequantised codes (chapter 10, sec. 1: the reader turns them back into
    wider numbers), then the same definition as ``decode``."""
    B, Hq, D = q.shape
    if Hq % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = Hq // num_kv_heads
    qf = to_f64(q, in_dtype)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        ids = np.asarray(block_tables[b][: -(-L // k_codes.shape[1])], dtype=np.int64)
        if np.any((ids < 0) | (ids >= k_codes.shape[0])):
            raise ValueError("block table names a block outside the pool")
        Kb = dequantize(k_codes[ids], None if k_scales is None else k_scales[ids], fmt, fp8_k_scale)
        Vb = dequantize(v_codes[ids], None if v_scales is None else v_scales[ids], fmt, fp8_v_scale)
        K = Kb.reshape(-1, num_kv_heads, D)[:L]
        V = Vb.reshape(-1, num_kv_heads, D)[:L]
        for g in range(num_kv_heads):
            heads = slice(g * group, (g + 1) * group)
            s = scale * (qf[b, heads] @ K[:, g, :].T)
            s = s - s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w = w / w.sum(axis=1, keepdims=True)
            out[b, heads] = w @ V[:, g, :]
    return out



def prefill_q8(q, in_dtype: str, k_codes, v_codes, k_scales, v_scales, fmt: str, cu_seqlens,
               block_tables, seq_lens, scale: float, num_kv_heads: int, fp8_k_scale: float = 1.0,
               fp8_v_scale: float = 1.0) -> np.ndarray:
    """Chunked-prefill attention over an 8-bit pool: the pool's values are the
    dequantised codes ("Part 3: single node", ch. 10: the reader turns them
    back into wider numbers), then the definition of ``prefill`` ("Part 3",
    ch. 13 sec. 1-2): request b's C_b queries sit at positions L_b - C_b + i
    and attend causally to positions 0 .. L_b - C_b + i of its cache."""
    T, Hq, D = q.shape
    if Hq % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = Hq // num_kv_heads
    bs = k_codes.shape[1]
    qf = to_f64(q, in_dtype)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for b in range(len(cu) - 1):
        C = int(cu[b + 1] - cu[b])
        L = int(seq_lens[b])
        if C <= 0 or L <= 0:
            continue
        ids = np.asarray(block_tables[b][: -(-L // bs)], dtype=np.int64)
        if np.any((ids < 0) | (ids >= k_codes.shape[0])):
            raise ValueError("block table names a block outside the pool")
        K = dequantize(k_codes[ids], None if k_scales is None else k_scales[ids], fmt,
                       fp8_k_scale).reshape(-1, num_kv_heads, D)[:L]
        V = dequantize(v_codes[ids], None if v_scales is None else v_scales[ids], fmt,
                       fp8_v_scale).reshape(-1, num_kv_heads, D)[:L]
        for i in range(C):
            pos = L - C + i                                                 # query position
            if pos < 0:
                continue
            for g in range(num_kv_heads):
                heads = slice(g * group, (g + 1) * group)
                s = scale * (qf[cu[b] + i, heads] @ K[:pos + 1, g, :].T)   # [group, pos + 1]
                s = s - s.max(axis=1, keepdims=True)
                w = np.exp(s)
                w = w / w.sum(axis=1, keepdims=True)
                out[cu[b] + i, heads] = w @ V[:pos + 1, g, :]
    return out

# ------------------------------------------------------- swap to host ----
#
# "Lecture 3" (semidirectx.com, CS349D notes), sec. 5.2 and "Part 3: single
# node" (random-liu.github.io), ch. 14 sec. 3: a preempted request's KV blocks
# are copied to CPU memory (a CPU block allocator hands out the host blocks)
# and copied back to GPU blocks when it resumes.  The copy is whole blocks;
# the definition is the same as copy_blocks with the source and destination
# in different pools.

SWAP_OUT, SWAP_IN = 0, 1


def swap_blocks(gpu_arrays, host_arrays, pairs, direction: int) -> int:
    """For each (gpu_block, host_block) pair in order: host[h] <- gpu[g]
    (SWAP_OUT) or gpu[g] <- host[h] (SWAP_IN), for every array of the pool
    (K, V, and INT8 scales when present; leading axis = block).  Pairs naming a
    block outside either pool are skipped and counted."""
    ng, nh = gpu_arrays[0].shape[0], host_arrays[0].shape[0]
    bad = 0
    for g, h in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= g < ng and 0 <= h < nh):
            bad += 1
            continue
        for ga, ha in zip(gpu_arrays, host_arrays):
            if direction == SWAP_OUT:
                ha[h] = ga[g].copy()
            else:
                ga[g] = ha[h].copy()
    return bad


# ------------------------------------------------- paged (chunked) prefill --
#
# "Part 3: single node" (random-liu.github.io), ch. 13 sec. 1 and 2: the new
# tokens of every request in a batch are flattened into one stream whose
# request boundaries are cu_seqlens; a long prompt is cut into chunks of at
# most a token budget, processed one chunk per iteration, and a chunk's
# attention reads the earlier part of the prompt (and any cached prefix)
# through the block table, like decode.  Reading taken where the pages stop:
# request b's C_b = cu_seqlens[b+1] - cu_seqlens[b] queries are its last C_b
# positions, L_b - C_b .. L_b - 1 (L_b = seq_lens[b], the context after the
# chunk's own K/V were appended), and query i attends causally to positions
# 0 .. L_b - C_b + i.  C_b = 1 is decode.

def prefill(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, dtype: str,
            cu_seqlens: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
            scale: float, num_kv_heads: int) -> np.ndarray:
    """q [T, Hq, D] raw (T = cu_seqlens[-1]) -> fp64 out [T, Hq, D]."""
    T, Hq, D = q.shape
    group = Hq // num_kv_heads
    qf = to_f64(q, dtype)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for b in range(len(cu) - 1):
        C = int(cu[b + 1] - cu[b])
        L = int(seq_lens[b])
        if C <= 0 or L <= 0:
            continue
        K = to_f64(gather_kv(k_pool, block_tables[b], L), dtype)          # [L, Hkv, D]
        V = to_f64(gather_kv(v_pool, block_tables[b], L), dtype)
        for i in range(C):
            p = L - C + i                                                   # query position
            if p < 0:
                continue
            for g in range(num_kv_heads):
                heads = slice(g * group, (g + 1) * group)
                s = scale * (qf[cu[b] + i, heads] @ K[:p + 1, g, :].T)     # [group, p + 1]
                s = s - s.max(axis=1, keepdims=True)
                w = np.exp(s)
                w = w / w.sum(axis=1, keepdims=True)
                out[cu[b] + i, heads] = w @ V[:p + 1, g, :]
    return out
