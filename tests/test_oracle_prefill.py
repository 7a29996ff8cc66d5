"""Pins of the paged (chunked) prefill oracle against things other than itself
(no GPU): decode (one query per request), torch's causal SDPA on a contiguous
prompt, the consistency of one chunk with two, and the numpy / C twins; then
planted mistakes that some pin must catch."""

import inspect
import textwrap

import numpy as np
import pytest
import torch

from oracle import np_oracle as npo
from paged_kv_cache_68_gb300 import workloads as wl


def _appended(w):
    k, v = w.k_pool.copy(), w.v_pool.copy()
    npo.append(k, v, w.k_new, w.v_new, w.slot_mapping)
    return k, v


def test_one_query_per_request_is_decode(c_oracle):
    w = wl.chunked_prefill_step("p1", 1, [5, 0, 40, 17], [1, 1, 1, 1], dtype="f32", num_q_heads=8,
                                num_kv_heads=2, head_dim=16, block_size=4)
    k, v = _appended(w)
    ref = npo.decode(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 2)
    for f in (npo.prefill, c_oracle.prefill):
        out = f(w.q, k, v, "f32", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 2)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_whole_prompt_chunk_equals_torch_causal_sdpa(c_oracle, dtype):
    """No cached prefix, one chunk = the whole prompt: causal attention."""
    w = wl.chunked_prefill_step("p2", 2, [0, 0], [37, 20], dtype=dtype, num_q_heads=4,
                                num_kv_heads=4, head_dim=16, block_size=8)
    k, v = _appended(w)
    out = c_oracle.prefill(w.q, k, v, dtype, w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 4)
    for b in range(2):
        L = int(w.seq_lens[b])
        K = npo.to_f64(npo.gather_kv(k, w.block_tables[b], L), dtype)
        V = npo.to_f64(npo.gather_kv(v, w.block_tables[b], L), dtype)
        Q = npo.to_f64(w.q[w.cu_seqlens[b]:w.cu_seqlens[b + 1]], dtype)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(1, 0, 2)))
        ref = torch.nn.functional.scaled_dot_product_attention(t(Q), t(K), t(V), is_causal=True,
                                                               scale=w.scale)
        np.testing.assert_allclose(out[w.cu_seqlens[b]:w.cu_seqlens[b + 1]],
                                   ref.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_two_chunks_equal_one(c_oracle):
    """Chunked prefill splits a prompt over iterations: the rows of a second
    chunk (reading the first through the table) equal those rows of the
    prompt processed as one chunk."""
    w = wl.chunked_prefill_step("p3", 3, [0], [300], dtype="f32", num_q_heads=8, num_kv_heads=2,
                                head_dim=16, block_size=16)
    k, v = _appended(w)
    whole = c_oracle.prefill(w.q, k, v, "f32", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 2)
    first = c_oracle.prefill(w.q[:200], k, v, "f32", np.array([0, 200]), w.block_tables,
                             np.array([200]), w.scale, 2)
    second = c_oracle.prefill(np.ascontiguousarray(w.q[200:]), k, v, "f32", np.array([0, 100]),
                              w.block_tables, np.array([300]), w.scale, 2)
    np.testing.assert_allclose(first, whole[:200], rtol=0, atol=1e-13)
    np.testing.assert_allclose(second, whole[200:], rtol=0, atol=1e-13)


def test_numpy_and_c_agree_on_a_mixed_batch(c_oracle):
    w = wl.chunked_prefill_step("p4", 4, [33, 0, 100, 7, 64], [16, 9, 1, 40, 1], dtype="bf16",
                                num_q_heads=16, num_kv_heads=4, head_dim=32, block_size=16)
    k, v = _appended(w)
    a = npo.prefill(w.q, k, v, "bf16", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 4)
    b = c_oracle.prefill(w.q, k, v, "bf16", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 4,
                         num_threads=3)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_flop_count_of_the_workload():
    """Query i of a chunk sees L - C + i + 1 tokens."""
    w = wl.chunked_prefill_step("p5", 5, [10, 3], [4, 1], dtype="f32", num_q_heads=2,
                                num_kv_heads=1, head_dim=8, block_size=4)
    pairs = (11 + 12 + 13 + 14) + 4
    assert w.attention_flops() == pairs * 2 * 8 * 4


MUTATIONS = {
    "causal_off_by_one": ("s = scale * (qf[cu[b] + i, heads] @ K[:p + 1, g, :].T)",
                          "s = scale * (qf[cu[b] + i, heads] @ K[:p, g, :].T)"),
    "position_off_by_one": ("p = L - C + i                                                   # query position",
                            "p = min(L - 1, L - C + i + 1)"),
    "chunk_only": ("s = scale * (qf[cu[b] + i, heads] @ K[:p + 1, g, :].T)",
                   "s = scale * (qf[cu[b] + i, heads] @ K[L - C:p + 1, g, :].T)"),
    "no_causal_mask": ("s = scale * (qf[cu[b] + i, heads] @ K[:p + 1, g, :].T)",
                       "s = scale * (qf[cu[b] + i, heads] @ K[:, g, :].T)"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(npo.prefill))
    assert old in src, name
    if name == "chunk_only":
        src = src.replace(old, new).replace("out[cu[b] + i, heads] = w @ V[:p + 1, g, :]",
                                            "out[cu[b] + i, heads] = w @ V[L - C:p + 1, g, :]")
    elif name == "no_causal_mask":
        src = src.replace(old, new).replace("out[cu[b] + i, heads] = w @ V[:p + 1, g, :]",
                                            "out[cu[b] + i, heads] = w @ V[:, g, :]")
    else:
        src = src.replace(old, new)
        if name == "causal_off_by_one":
            src = src.replace("out[cu[b] + i, heads] = w @ V[:p + 1, g, :]",
                              "out[cu[b] + i, heads] = w @ V[:p, g, :] if p > 0 else 0.0")
    ns = dict(vars(npo))
    exec(src, ns)
    return ns["prefill"]


def _pins_pass(prefill, c_oracle):
    try:
        w = wl.chunked_prefill_step("m1", 1, [5, 0, 40, 17], [1, 1, 1, 1], dtype="f32",
                                    num_q_heads=8, num_kv_heads=2, head_dim=16, block_size=4)
        k, v = _appended(w)
        ref = npo.decode(w.q, k, v, "f32", w.block_tables, w.seq_lens, w.scale, 2)
        out = prefill(w.q, k, v, "f32", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 2)
        if not np.allclose(out, ref, rtol=0, atol=1e-12):
            return False
        w = wl.chunked_prefill_step("m2", 2, [0, 24], [37, 12], dtype="f32", num_q_heads=4,
                                    num_kv_heads=4, head_dim=16, block_size=8)
        k, v = _appended(w)
        ref = c_oracle.prefill(w.q, k, v, "f32", w.cu_seqlens, w.block_tables, w.seq_lens,
                               w.scale, 4)
        out = prefill(w.q, k, v, "f32", w.cu_seqlens, w.block_tables, w.seq_lens, w.scale, 4)
        return bool(np.allclose(out, ref, rtol=0, atol=1e-12))
    except Exception:
        return False


def test_prefill_pins_pass_on_the_oracle(c_oracle):
    assert _pins_pass(npo.prefill, c_oracle)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_prefill_pins_catch_planted_mistake(c_oracle, name):
    assert not _pins_pass(_mutant(name), c_oracle), f"mutant {name} passed"
