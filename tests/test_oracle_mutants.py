"""Plant plausible mistakes in (a copy of) the numpy oracle and check that the
pins catch every one of them (no GPU).

Each mutant is the oracle's decode with one edit: a dropped term, a wrong
index or operand, an off-by-one.  The pin battery below is the same set of
facts the oracle pins use (closed forms, the torch SDPA reduction, the GQA
grouping, permutation invariance); the unmodified oracle passes all of them.
"""

import inspect
import math
import textwrap

import numpy as np
import pytest
import torch

from oracle import np_oracle
from paged_kv_cache_68_gb300 import workloads as wl

MUTATIONS = {
    "interleaved_gqa": ("heads = slice(g * group, (g + 1) * group)",
                        "heads = slice(g, None, num_kv_heads)"),
    "dropped_scale": ("s = scale * (qf[b, heads] @ K[:, g, :].T)", "s = (qf[b, heads] @ K[:, g, :].T)"),
    "no_normalisation": ("w = w / w.sum(axis=1, keepdims=True)", "w = w"),
    "k_for_v": ("out[b, heads] = w @ V[:, g, :]", "out[b, heads] = w @ K[:, g, :]"),
    "v_for_k": ("s = scale * (qf[b, heads] @ K[:, g, :].T)", "s = scale * (qf[b, heads] @ V[:, g, :].T)"),
    "length_off_by_one": ("L = int(seq_lens[b])", "L = int(seq_lens[b]) - 1"),
    "wrong_sign": ("w = np.exp(s)", "w = np.exp(-s)"),
    "kv_head_ignored": ("s = scale * (qf[b, heads] @ K[:, g, :].T)", "s = scale * (qf[b, heads] @ K[:, 0, :].T)"),
}

GATHER_MUTATIONS = {
    "table_ignored": ("ids = [int(table_row[j]) for j in range(nblk)]",
                      "ids = [j for j in range(nblk)]"),
    "no_truncation": ("return np.concatenate(blocks, axis=0)[:seq_len]",
                      "return np.concatenate(blocks, axis=0)"),
}


def _mutant(name):
    """Build a decode function with one planted edit."""
    ns = dict(vars(np_oracle))
    if name in MUTATIONS:
        old, new = MUTATIONS[name]
        src = textwrap.dedent(inspect.getsource(np_oracle.decode))
        assert old in src, name
        exec(src.replace(old, new), ns)
    else:
        old, new = GATHER_MUTATIONS[name]
        src = textwrap.dedent(inspect.getsource(np_oracle.gather_kv))
        assert old in src, name
        exec(src.replace(old, new), ns)
        exec(textwrap.dedent(inspect.getsource(np_oracle.decode)), ns)
    return ns["decode"]


def _appended(w):
    k, v = w.k_pool.copy(), w.v_pool.copy()
    np_oracle.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    return k, v


def pin_two_tokens(decode):
    pk, pv = wl.nan_fill((3, 4, 1, 4), "f32"), wl.nan_fill((3, 4, 1, 4), "f32")
    pk[2, 0, 0], pk[2, 1, 0] = [1, 0, 0, 0], [0, 1, 0, 0]
    pv[2, 0, 0], pv[2, 1, 0] = [4, 0, 0, 2], [0, 8, 0, 2]
    q = np.array([[[2, 0, 0, 0]]], dtype=np.float32)
    w0 = 1.0 / (1.0 + math.exp(-1.0))
    out = decode(q, pk, pv, "f32", np.array([[2]], np.int32), np.array([2], np.int32), 0.5, 1)
    return np.allclose(out[0, 0], [4 * w0, 8 * (1 - w0), 0, 2], rtol=0, atol=1e-12)


def pin_three_tokens_scattered(decode):
    pk, pv = wl.nan_fill((4, 2, 1, 2), "f32"), wl.nan_fill((4, 2, 1, 2), "f32")
    a, b = np.float32(math.log(2.0)), np.float32(math.log(5.0))
    pk[3, 0, 0], pk[3, 1, 0], pk[0, 0, 0] = [a, 0], [0, 0], [b, 0]
    pv[3, 0, 0], pv[3, 1, 0], pv[0, 0, 0] = [8, 0], [0, 8], [8, 8]
    out = decode(np.array([[[1, 0]]], np.float32), pk, pv, "f32", np.array([[3, 0]], np.int32),
                 np.array([3], np.int32), 1.0, 1)
    return np.allclose(out[0, 0], [7, 6], rtol=0, atol=1e-6)


def pin_gqa_grouping(decode):
    w = wl.build_step("g", 7, [5, 40], dtype="f32", num_q_heads=8, num_kv_heads=2,
                      head_dim=16, block_size=4)
    v = w.v_pool.copy()
    for g in range(2):
        v[:, :, g, :] = np.where(np.isnan(v[:, :, g, :]), np.nan, g + 1)
    vn = np.ones_like(w.v_new)
    vn[:, 1] = 2
    k = w.k_pool.copy()
    np_oracle.append(k, v, w.k_new, vn, w.slot_mapping)
    out = decode(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 2)
    return all(np.allclose(out[:, h], h // 4 + 1, rtol=0, atol=1e-12) for h in range(8))


def pin_sdpa_identity(decode):
    w = wl.build_step("id", 11, [1, 7, 33], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                      head_dim=32, block_size=8, placement="identity")
    k, v = _appended(w)
    out = decode(w.q, k, v, "bf16", w.block_tables, w.seq_lens, w.scale, 2)
    for b in range(w.batch):
        L, s0 = int(w.seq_lens[b]), int(w.block_tables[b, 0]) * 8
        kk = np_oracle.to_f64(k.reshape(-1, 2, 32)[s0:s0 + L], "bf16")
        vv = np_oracle.to_f64(v.reshape(-1, 2, 32)[s0:s0 + L], "bf16")
        qq = torch.from_numpy(np_oracle.to_f64(w.q[b], "bf16"))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, torch.from_numpy(kk).permute(1, 0, 2)[None], torch.from_numpy(vv).permute(1, 0, 2)[None],
            scale=w.scale, enable_gqa=True)[0, :, 0, :].numpy()
        if not np.allclose(out[b], ref, rtol=0, atol=1e-12):
            return False
    return True


def pin_permutation(decode):
    w = wl.build_step("p", 21, [3, 17, 70], dtype="f16", num_q_heads=4, num_kv_heads=2,
                      head_dim=16, block_size=8)
    k0, v0 = _appended(w)
    perm = np.random.default_rng(0).permutation(w.num_blocks)
    k1, v1 = np.empty_like(k0), np.empty_like(v0)
    k1[perm], v1[perm] = k0, v0
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    o0 = decode(w.q, k0, v0, "f16", w.block_tables, w.seq_lens, w.scale, 2)
    o1 = decode(w.q, k1, v1, "f16", bt, w.seq_lens, w.scale, 2)
    return np.array_equal(o0, o1) and np.isfinite(o0).all()


PINS = [pin_two_tokens, pin_three_tokens_scattered, pin_gqa_grouping, pin_sdpa_identity,
        pin_permutation]


def _failing(decode):
    bad = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                ok = pin(decode)
        except Exception:          # a crash counts as caught
            ok = False
        if not ok:
            bad.append(pin.__name__)
    return bad


def test_unmodified_oracle_passes_every_pin():
    assert _failing(np_oracle.decode) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS) + sorted(GATHER_MUTATIONS))
def test_planted_mistake_is_caught(name):
    assert _failing(_mutant(name)), f"no pin catches mutant {name}"
