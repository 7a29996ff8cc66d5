"""GPU parity of the 8-bit KV cache (FP8 E4M3 with per-pool scales, INT8 with
per-token-head scales): the quantising append and the block copy byte for
byte against the C oracle, and decode against the oracle's fp64 attention over
the dequantised values (the 16-bit tolerance: the codes convert exactly, so
only fp32 arithmetic separates the two)."""

import ctypes

import numpy as np
import pytest
import torch

from parity import (TORCH_DTYPE, assert_q8_pools_equal, check_attention, gpu_step_q8,
                    oracle_step_q8)
from paged_kv_cache_68_gb300 import pagedkv
from paged_kv_cache_68_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CACHES = [("fp8_e4m3", 1.0, 1.0), ("fp8_e4m3", 0.25, 3.0), ("int8", 1.0, 1.0)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pagedkv.load()


def _check(w, cache, sk=1.0, sv=1.0, seed=7, what="", seqs=None):
    p = wl.q8_pools(w, cache, seed, sk, sv)
    gk, gv, gks, gvs, out, err = gpu_step_q8(w, p)
    rk, rv, rks, rvs, ref = oracle_step_q8(w, p, seqs)
    assert err == 0, f"{what}: device error bits {err:#x}"
    assert_q8_pools_equal((gk, gv, gks, gvs), (rk, rv, rks, rvs), what)
    sel = slice(None) if seqs is None else np.asarray(seqs)
    return check_attention(out[sel], ref, w.dtype, what)


@pytest.mark.parametrize("cache,sk,sv", CACHES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_q8_llama_small(cache, sk, sv, dtype):
    w = wl.build_step("q8", 1, [0, 1, 15, 16, 17, 33, 200, 1000, 555], dtype=dtype,
                      num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)
    _check(w, cache, sk, sv, what=f"{cache} {dtype}")


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("hq,hkv,bs", [(4, 4, 16), (8, 4, 32), (16, 4, 16), (16, 2, 16),
                                       (16, 2, 64), (40, 40, 16), (8, 1, 48)])
def test_q8_groups_and_block_sizes(cache, hq, hkv, bs):
    ctx = [0, 1, bs - 1, bs, 2 * bs + 3, 5 * bs, 301]
    w = wl.build_step("q8 shapes", 4, ctx, dtype="bf16", num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=128, block_size=bs)
    _check(w, cache, what=f"{cache} hq{hq} hkv{hkv} bs{bs}")


@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_copy_on_write_and_zero_length(cache):
    """Copy-on-write pairs move codes and scales; a zero-length sequence gives
    zeros; a padding slot writes nothing."""
    w = wl.shared_prefix(2, prompts=2, prompt_len=136, n=4, divergent=np.zeros(8, np.int64))
    assert w.pairs.shape[0] > 0
    w.seq_lens[3] = 0
    w.slot_mapping[3] = -1
    _check(w, cache, what=f"{cache} cow")


@pytest.mark.parametrize("cache,sk,sv", CACHES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_q8_append_special_rows(cache, sk, sv, dtype):
    """Rows of zeros, huge values (FP8 saturation), infinities and NaN, a
    padding slot and an out-of-range slot: the stored codes and scales equal
    the oracle's byte for byte."""
    w = wl.build_step("q8 special", 5, [3, 20, 40, 7, 64, 1], dtype=dtype, num_q_heads=8,
                      num_kv_heads=2, head_dim=128, block_size=16)
    h = wl.on_host(w)
    kn = wl.randn(np.random.default_rng(9), h.k_new.shape, dtype)
    kn[0] = wl.from_f32(np.zeros(h.k_new.shape[1:], np.float32), dtype)          # all zero
    big = np.full(h.k_new.shape[1:], 3000.0, np.float32)
    big[:, ::3] = -5000.0
    kn[1] = wl.from_f32(big, dtype)                                               # saturates
    tiny = np.full(h.k_new.shape[1:], 1e-4, np.float32)
    kn[2] = wl.from_f32(tiny, dtype)
    if cache == "int8":                       # FP8 NaN inputs keep an unspecified sign bit
        odd = np.ones(h.k_new.shape[1:], np.float32)
        odd[0, 5], odd[1, 7] = np.inf, np.nan
        kn[4] = wl.from_f32(odd, dtype)
    h.k_new = kn
    slots = h.slot_mapping.copy()
    slots[5] = -1
    h.slot_mapping = slots
    p = wl.q8_pools(h, cache, 3, sk, sv)
    gk, gv, gks, gvs, _, err = gpu_step_q8(h, p)
    rk, rv, rks, rvs, _ = oracle_step_q8(h, p, seqs=[])
    assert err == 0
    assert_q8_pools_equal((gk, gv, gks, gvs), (rk, rv, rks, rvs), f"{cache} special")
    # an out-of-range slot is skipped and flagged
    h.slot_mapping = slots.copy()
    h.slot_mapping[0] = h.num_blocks * h.block_size + 5
    h.k_new = wl.randn(np.random.default_rng(10), h.k_new.shape, dtype)
    gk, gv, gks, gvs, _, err = gpu_step_q8(h, p)
    assert err & pagedkv.KV_DEVERR_SLOT_RANGE
    rk, rv, rks, rvs, _ = oracle_step_q8(h, p, seqs=[])
    assert_q8_pools_equal((gk, gv, gks, gvs), (rk, rv, rks, rvs), f"{cache} out of range")


def test_q8_int8_v_scales_zero_then_jump():
    """INT8 V scales that are zero over each sequence's first two blocks and
    100x larger on one later block: the decode weighs P by each token's V
    scale over the largest one met so far in the piece, which starts at zero
    and then rises mid-sequence (with a rescale of the partial output)."""
    w = wl.build_step("q8 vscale", 6, [20, 40, 300, 700, 1500], dtype="bf16", num_q_heads=32,
                      num_kv_heads=8, head_dim=128, block_size=16)
    p = wl.q8_pools(w, "int8", 11)
    vs = np.array(p.v_scales, copy=True)                    # [N, Hkv, bs]
    bt = np.asarray(w.block_tables)
    for b, L in enumerate(np.asarray(w.seq_lens)):
        nb = (int(L) + 15) // 16
        for j in range(min(2, nb)):
            vs[bt[b, j]] = 0.0
        if nb > 4:
            vs[bt[b, (3 * nb) // 5]] *= 100.0
    p.v_scales = vs
    gk, gv, gks, gvs, out, err = gpu_step_q8(w, p)
    rk, rv, rks, rvs, ref = oracle_step_q8(w, p)
    assert err == 0
    assert_q8_pools_equal((gk, gv, gks, gvs), (rk, rv, rks, rvs), "int8 v scales")
    print(check_attention(out, ref, w.dtype, "int8 v scales"))


@pytest.mark.slow
@pytest.mark.parametrize("cache", ["fp8_e4m3", "int8"])
def test_q8_llama_full_sampled(cache):
    """The benchmark's Llama-3-8B-shaped step at full size; the oracle checks
    a sample of 24 sequences (every pool byte is compared)."""
    w = wl.llama3_8b_gqa(0, device="cuda")
    seqs = list(range(0, 256, 11))
    print(_check(w, cache, what=f"{cache} llama full", seqs=seqs))


def test_q8_host_argument_errors():
    lib = pagedkv.load()
    dev = torch.device("cuda")
    codes = torch.zeros((4, 16, 2, 128), dtype=torch.uint8, device=dev)
    sc = torch.zeros((4, 2, 16), dtype=torch.float32, device=dev)
    h = ctypes.c_void_p()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    create = lambda *a: lib.kv_pool_create_quantized(*a, ctypes.byref(h))
    bf16 = pagedkv.DTYPE_CODE[torch.bfloat16]
    # INT8 without scales, FP8 with scales, FP8 with a non-positive scale
    assert create(4, 16, 2, 128, pagedkv.KV_INT8, bf16, P(codes), P(codes), None, None, 1.0, 1.0) \
        == pagedkv.KV_EINVAL
    assert create(4, 16, 2, 128, pagedkv.KV_FP8_E4M3, bf16, P(codes), P(codes), P(sc), P(sc), 1.0,
                  1.0) == pagedkv.KV_EINVAL
    assert create(4, 16, 2, 128, pagedkv.KV_FP8_E4M3, bf16, P(codes), P(codes), None, None, 0.0,
                  1.0) == pagedkv.KV_EINVAL
    # head_dim 64, block size 8, fp32 queries, a 16-bit cache type: not built
    assert create(4, 16, 4, 64, pagedkv.KV_INT8, bf16, P(codes), P(codes), P(sc), P(sc), 1.0,
                  1.0) == pagedkv.KV_EUNSUPPORTED
    assert create(8, 8, 2, 128, pagedkv.KV_INT8, bf16, P(codes), P(codes), P(sc), P(sc), 1.0,
                  1.0) == pagedkv.KV_EUNSUPPORTED
    assert create(4, 16, 2, 128, pagedkv.KV_INT8, 0, P(codes), P(codes), P(sc), P(sc), 1.0,
                  1.0) == pagedkv.KV_EUNSUPPORTED
    assert create(4, 16, 2, 128, bf16, bf16, P(codes), P(codes), None, None, 1.0,
                  1.0) == pagedkv.KV_EUNSUPPORTED
    assert create(4, 16, 2, 128, pagedkv.KV_INT8, bf16, P(codes), P(codes), P(sc), P(sc), 1.0,
                  1.0) == pagedkv.KV_OK
    pagedkv.kv_pool_destroy(h)


def test_q8_cascade_call_decodes_plainly():
    """The cascade entry point on an 8-bit pool of a shape without a prefix
    pass (block size 64) gives the plain decode's bits."""
    w = wl.shared_prefix(3, prompts=2, prompt_len=300, n=4, max_divergent=30, block_size=64)
    assert (np.asarray(w.groups)[:, 2] > 0).all()
    p = wl.q8_pools(w, "int8", 1)
    dev = torch.device("cuda")
    tv = lambda a: wl.value_to_torch(a, w.dtype, dev)
    pool = pagedkv.KVPool(torch.from_numpy(p.k_codes).to(dev), torch.from_numpy(p.v_codes).to(dev),
                          cache="int8", dtype=TORCH_DTYPE[w.dtype],
                          k_scales=torch.from_numpy(p.k_scales).to(dev),
                          v_scales=torch.from_numpy(p.v_scales).to(dev))
    try:
        pool.append(tv(w.k_new), tv(w.v_new), torch.from_numpy(w.slot_mapping).to(dev))
        q = tv(w.q)
        tables = torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(dev)
        lens = torch.from_numpy(w.seq_lens).to(dev)
        a = pool.decode(q, tables, lens, w.scale)
        b = pool.decode_cascade(q, tables, lens, w.scale,
                                torch.from_numpy(np.ascontiguousarray(w.groups)).to(dev))
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert pool.get_error() == 0
    finally:
        pool.close()
