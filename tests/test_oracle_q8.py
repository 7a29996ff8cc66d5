"""Pins of the 8-bit KV cache oracle (FP8 E4M3 and INT8) against things
other than itself (no GPU): a library's FP8 format, closed forms, the
quantisation error bound, and the already-pinned 16-bit attention oracle run
on the dequantised values.  Both oracles (numpy and plain C) go through each
pin; a second block plants plausible mistakes and checks that a pin fails.
"""

import inspect
import math
import textwrap

import numpy as np
import pytest
import torch

from oracle import np_oracle as npo
from paged_kv_cache_68_gb300 import workloads as wl


# --- E4M3: the format ---------------------------------------------------------

def test_e4m3_decode_all_codes_matches_torch(c_oracle):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(npo.e4m3_to_f64(codes), ref, equal_nan=True)
    c = np.array([c_oracle.e4m3_decode(int(x)) for x in codes])
    assert np.array_equal(c, ref, equal_nan=True)


def _sweep():
    rng = np.random.default_rng(5)
    vals = npo.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))          # 0 .. 448
    mids = (vals[1:] + vals[:-1]) / 2                                   # every tie
    x = [rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)]
    x += [mids, -mids, vals, -vals, np.nextafter(mids, 0), np.nextafter(mids, 1e9)]
    x = np.concatenate(x).astype(np.float32)
    return x[np.abs(x) < 464]


def test_e4m3_encode_matches_torch_in_range(c_oracle):
    """Round to nearest, ties to even, over every midpoint of the format."""
    x = _sweep()
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(npo.f32_to_e4m3(x), ref)
    sub = x[::7]
    c = np.array([c_oracle.e4m3_encode(float(v)) for v in sub], dtype=np.uint8)
    assert np.array_equal(c, ref[::7])


@pytest.mark.parametrize("x, code", [(1.0, 0x38), (448.0, 0x7E), (-448.0, 0xFE), (2.0 ** -9, 0x01),
                                     (2.0 ** -6, 0x08), (0.5 * 2.0 ** -9, 0x00),
                                     (1.5 * 2.0 ** -9, 0x02), (1.0625, 0x38), (1.1875, 0x3A),
                                     (-0.0, 0x80), (1e6, 0x7E), (math.inf, 0x7E),
                                     (-math.inf, 0xFE), (465.0, 0x7E), (math.nan, 0x7F)])
def test_e4m3_encode_closed_forms(c_oracle, x, code):
    """Exact values, ties to even, signed zero, saturation beyond 448 (the
    reading for values past the largest finite), NaN -> 0x7F."""
    assert int(npo.f32_to_e4m3(np.array([x], np.float32))[0]) == code
    assert c_oracle.e4m3_encode(x) == code


# --- INT8: per-row scale ---------------------------------------------------------

def test_int8_closed_form_row(c_oracle):
    """amax 127 gives scale 1: codes are x rounded half to even."""
    x = np.array([127.0, -63.5, 0.5, 1.5, -2.5, 2.5, -127.0, 3.49], np.float32)
    want = np.array([127, -64, 0, 2, -2, 2, -127, 3], np.int8)
    for codes, scale in (npo.int8_quantize(x[None])[0][0], npo.int8_quantize(x[None])[1][0]), \
            c_oracle.int8_quantize_row(x):
        assert np.array_equal(codes, want)
        assert scale == np.float32(1.0)


def test_int8_zero_and_nonfinite_rows(c_oracle):
    for row, want_scale in ((np.zeros(16, np.float32), 0.0),
                            (np.array([1.0, np.nan] + [0.0] * 14, np.float32), np.nan),
                            (np.array([1.0, -np.inf] + [0.0] * 14, np.float32), np.nan)):
        c, s = npo.int8_quantize(row[None])
        c2, s2 = c_oracle.int8_quantize_row(row)
        assert not c.any() and not c2.any()
        assert (math.isnan(s[0]) and math.isnan(s2)) if math.isnan(want_scale) else s[0] == s2 == 0


def test_int8_error_bound_and_full_range(c_oracle):
    """|x - code * scale| <= scale / 2 (plus fp32 slack) and the largest |x|
    maps to +-127, for rows of very different magnitudes."""
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((300, 64)) * np.exp(rng.uniform(-12, 12, (300, 1)))).astype(np.float32)
    codes, scales = npo.int8_quantize(rows)
    deq = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    err = np.abs(rows.astype(np.float64) - deq)
    assert np.all(err <= scales.astype(np.float64)[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(codes).max(axis=1) == 127)
    for i in range(0, 300, 37):
        c2, s2 = c_oracle.int8_quantize_row(rows[i])
        assert np.array_equal(c2, codes[i]) and s2 == scales[i]


# --- append / copy / decode over an 8-bit pool -----------------------------------

def _q8_setup(fmt, in_dtype, seed, lens, hq=8, hkv=2, d=32, bs=4, spare=3):
    """A small pool: every context token written through the quantising append."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    nblk = [-(-L // bs) for L in lens]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    tables = np.full((B, max(nblk) + 1), -1, np.int32)
    pos, slots = 0, []
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[pos:pos + n]
        pos += n
        slots += [tables[b, t // bs] * bs + t % bs for t in range(lens[b])]
    T = len(slots)
    kx = wl.from_f32((rng.standard_normal((T, hkv, d)) * 1.5).astype(np.float32), in_dtype)
    vx = wl.from_f32(rng.standard_normal((T, hkv, d)).astype(np.float32), in_dtype)
    kc = np.full((nb, bs, hkv, d), 0x7F, np.uint8)          # E4M3 NaN / INT8 127: never read
    vc = np.full((nb, bs, hkv, d), 0x7F, np.uint8)
    ks = np.full((nb, hkv, bs), np.nan, np.float32) if fmt == "int8" else None
    vs = np.full((nb, hkv, bs), np.nan, np.float32) if fmt == "int8" else None
    q = wl.from_f32(rng.standard_normal((B, hq, d)).astype(np.float32), in_dtype)
    return dict(q=q, kc=kc, vc=vc, ks=ks, vs=vs, kx=kx, vx=vx, slots=np.array(slots, np.int64),
                tables=tables, lens=np.array(lens, np.int32), hkv=hkv, bs=bs, d=d)


FMTS = [("fp8_e4m3", 1.0, 1.0), ("fp8_e4m3", 0.25, 3.0), ("int8", 1.0, 1.0)]


@pytest.mark.parametrize("fmt, sk, sv", FMTS)
@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_append_q8_numpy_and_c_agree(c_oracle, fmt, sk, sv, in_dtype):
    s = _q8_setup(fmt, in_dtype, 1, [5, 9, 1])
    pools = []
    for impl in (npo, c_oracle):
        kc, vc = s["kc"].copy(), s["vc"].copy()
        ks = None if s["ks"] is None else s["ks"].copy()
        vs = None if s["vs"] is None else s["vs"].copy()
        slots = np.concatenate([s["slots"], [-1, kc.shape[0] * kc.shape[1] + 3]])
        kx = np.concatenate([s["kx"], s["kx"][:2]])
        vx = np.concatenate([s["vx"], s["vx"][:2]])
        bad = impl.append_q8(kc, vc, ks, vs, kx, vx, in_dtype, slots, fmt, sk, sv)
        assert bad == 1
        pools.append((kc, vc, ks, vs))
    for a, b in zip(pools[0], pools[1]):
        if a is not None:
            assert np.array_equal(a, b, equal_nan=True)


@pytest.mark.parametrize("fmt, sk, sv", FMTS)
def test_append_q8_codes_at_slots(c_oracle, fmt, sk, sv):
    """The row of token i lands at block slot // bs, row slot % bs, and holds
    the row's own quantisation (the format pins above)."""
    s = _q8_setup(fmt, "bf16", 2, [6, 3])
    kc, vc, ks, vs = s["kc"], s["vc"], s["ks"], s["vs"]
    c_oracle.append_q8(kc, vc, ks, vs, s["kx"], s["vx"], "bf16", s["slots"], fmt, sk, sv)
    bs = s["bs"]
    for i, slot in enumerate(s["slots"]):
        blk, off = divmod(int(slot), bs)
        x = npo.to_f64(s["kx"][i], "bf16").astype(np.float32)
        if fmt == "int8":
            c, sc = npo.int8_quantize(x)
            assert np.array_equal(kc[blk, off].view(np.int8), c)
            assert np.array_equal(ks[blk, :, off], sc)
        else:
            assert np.array_equal(kc[blk, off], npo.f32_to_e4m3((x / np.float32(sk)).astype(np.float32)))


def test_copy_blocks_q8_moves_codes_and_scales(c_oracle):
    s = _q8_setup("int8", "bf16", 3, [8, 4])
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "bf16", s["slots"], "int8")
    src, dst = int(s["tables"][0, 1]), int(s["tables"][1, 0])
    pools = [tuple(a.copy() for a in (s["kc"], s["vc"], s["ks"], s["vs"])) for _ in range(2)]
    npo.copy_blocks_q8(*pools[0], [[src, dst]])
    c_oracle.copy_blocks_q8(*pools[1], [[src, dst], [0, 999]])
    for a, b, orig in zip(pools[0], pools[1], (s["kc"], s["vc"], s["ks"], s["vs"])):
        assert np.array_equal(a, b, equal_nan=True)
        assert np.array_equal(a[dst], orig[src], equal_nan=True)


def _decoders(c_oracle):
    return [("numpy", npo.decode_q8), ("c", c_oracle.decode_q8),
            ("c3", lambda *a, **k: c_oracle.decode_q8(*a, num_threads=3, **k))]


@pytest.mark.parametrize("fmt, sk, sv", FMTS)
def test_decode_q8_equals_16bit_oracle_on_dequantised_pool(c_oracle, fmt, sk, sv):
    """Reduction to the pinned attention oracle: an fp32 pool that holds the
    dequantised values gives the same output."""
    s = _q8_setup(fmt, "f16", 4, [7, 1, 12, 0, 4])
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "f16", s["slots"], fmt, sk, sv)
    deqk = npo.dequantize(s["kc"], s["ks"], fmt, sk)
    deqv = npo.dequantize(s["vc"], s["vs"], fmt, sv)
    assert np.array_equal(deqk, deqk.astype(np.float32), equal_nan=True) or fmt == "int8"
    q32 = npo.to_f64(s["q"], "f16").astype(np.float32)
    ref = npo.decode(q32, deqk.astype(np.float32), deqv.astype(np.float32), "f32", s["tables"],
                     s["lens"], 0.3, s["hkv"]) if fmt != "int8" else None
    for name, dec in _decoders(c_oracle):
        out = dec(s["q"], "f16", s["kc"], s["vc"], s["ks"], s["vs"], fmt, s["tables"], s["lens"],
                  0.3, s["hkv"], fp8_k_scale=sk, fp8_v_scale=sv)
        if ref is not None:
            np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12, err_msg=name)
        # INT8 values (code * fp32 scale) need more than fp32: compare in fp64
        B, Hq, D = s["q"].shape
        g = Hq // s["hkv"]
        for b in range(B):
            L = int(s["lens"][b])
            for h in range(Hq):
                if L == 0:
                    assert not out[b, h].any()
                    continue
                tb = s["tables"][b]
                K = np.stack([deqk[tb[t // s["bs"]], t % s["bs"], h // g] for t in range(L)])
                V = np.stack([deqv[tb[t // s["bs"]], t % s["bs"], h // g] for t in range(L)])
                sc = 0.3 * (K @ npo.to_f64(s["q"][b, h], "f16"))
                w = np.exp(sc - sc.max())
                np.testing.assert_allclose(out[b, h], (w / w.sum()) @ V, rtol=0, atol=1e-12,
                                           err_msg=name)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "int8"])
def test_decode_q8_one_token_is_dequantised_v0(c_oracle, fmt):
    s = _q8_setup(fmt, "bf16", 5, [1, 1])
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "bf16", s["slots"], fmt)
    deqv = npo.dequantize(s["vc"], s["vs"], fmt)
    for name, dec in _decoders(c_oracle):
        out = dec(s["q"], "bf16", s["kc"], s["vc"], s["ks"], s["vs"], fmt, s["tables"], s["lens"],
                  0.7, s["hkv"])
        for b in range(2):
            blk = s["tables"][b, 0]
            for h in range(8):
                assert np.array_equal(out[b, h], deqv[blk, 0, h // 4]), name


def test_decode_q8_identity_table_equals_torch_sdpa(c_oracle):
    """Contiguous placement: torch's SDPA in float64 on the dequantised K/V."""
    s = _q8_setup("int8", "bf16", 6, [9, 16, 3], hq=4, hkv=4, d=16, bs=4)
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "bf16", s["slots"], "int8")
    deqk = npo.dequantize(s["kc"], s["ks"], "int8")
    deqv = npo.dequantize(s["vc"], s["vs"], "int8")
    out = c_oracle.decode_q8(s["q"], "bf16", s["kc"], s["vc"], s["ks"], s["vs"], "int8",
                             s["tables"], s["lens"], 0.25, 4)
    for b, L in enumerate(s["lens"]):
        tb = s["tables"][b]
        K = torch.from_numpy(np.stack([deqk[tb[t // 4], t % 4] for t in range(L)])).permute(1, 0, 2)
        V = torch.from_numpy(np.stack([deqv[tb[t // 4], t % 4] for t in range(L)])).permute(1, 0, 2)
        Q = torch.from_numpy(npo.to_f64(s["q"][b], "bf16"))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=0.25)[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)


# --- planted mistakes ---------------------------------------------------------------

Q8_MUTATIONS = {
    "int8_divisor_128": (npo.int8_quantize, "inv = np.float32(127.0) / amax", "inv = np.float32(128.0) / amax"),
    "int8_truncation": (npo.int8_quantize, "np.clip(np.rint(t), -127, 127)", "np.clip(np.trunc(t), -127, 127)"),
    "int8_scale_inverted": (npo.int8_quantize, "flat_s[r] = amax / np.float32(127.0)",
                            "flat_s[r] = np.float32(127.0) / amax"),
    "e4m3_ties_away": (npo.f32_to_e4m3, "m = float(np.rint(a / 2.0 ** (E - 3)))",
                       "m = float(np.floor(a / 2.0 ** (E - 3) + 0.5))"),
    "e4m3_bias_8": (npo.f32_to_e4m3, "flat_o[i] = sign | ((E2 + 7) << 3)", "flat_o[i] = sign | ((E2 + 8) << 3)"),
    "e4m3_no_saturation": (npo.f32_to_e4m3, "a = min(abs(x), E4M3_MAX)", "a = abs(x)"),
    "dequant_scale_layout": (npo.dequantize, ".transpose(0, 2, 1)", ""),
    "dequant_fp8_scale_dropped": (npo.dequantize, "return e4m3_to_f64(codes) * float(fp8_scale)",
                                  "return e4m3_to_f64(codes)"),
}


def _q8_mutant(name):
    fn, old, new = Q8_MUTATIONS[name]
    ns = dict(vars(npo))
    src = textwrap.dedent(inspect.getsource(fn))
    assert old in src, name
    exec(src.replace(old, new), ns)
    return ns


def _pins_pass(ns):
    """The numpy-side pins above, run against a (possibly mutated) namespace."""
    try:
        x = _sweep()
        ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        if not np.array_equal(ns["f32_to_e4m3"](x), ref):
            return False
        if int(ns["f32_to_e4m3"](np.array([1e6], np.float32))[0]) != 0x7E:
            return False
        row = np.array([[127.0, -63.5, 0.5, 1.5, -2.5, 2.5, -127.0, 3.49]], np.float32)
        c, sc = ns["int8_quantize"](row)
        if not (np.array_equal(c[0], [127, -64, 0, 2, -2, 2, -127, 3]) and sc[0] == 1.0):
            return False
        rng = np.random.default_rng(6)
        rows = (rng.standard_normal((50, 32)) * 7.0).astype(np.float32)
        c, sc = ns["int8_quantize"](rows)
        err = np.abs(rows - c.astype(np.float64) * sc.astype(np.float64)[:, None])
        if not np.all(err <= sc.astype(np.float64)[:, None] * (0.5 + 1e-5)):
            return False
        # dequantisation: scales differ per token and head, fp8 pool scale != 1
        codes = rng.integers(-127, 128, (2, 3, 2, 4)).astype(np.int8).view(np.uint8)
        scales = rng.uniform(0.5, 2.0, (2, 2, 3)).astype(np.float32)
        d = ns["dequantize"](codes, scales, "int8")
        want = codes.view(np.int8).astype(np.float64) * np.transpose(scales, (0, 2, 1))[..., None]
        if not np.array_equal(d, want):
            return False
        f8 = ns["dequantize"](np.array([0x38], np.uint8), None, "fp8_e4m3", 3.0)
        return float(f8[0]) == 3.0
    except Exception:
        return False


def test_q8_pins_pass_on_the_oracle():
    assert _pins_pass(dict(vars(npo)))


@pytest.mark.parametrize("name", sorted(Q8_MUTATIONS))
def test_q8_pins_catch_planted_mistake(name):
    assert not _pins_pass(_q8_mutant(name)), f"mutant {name} passed every pin"


# -- chunked prefill over an 8-bit pool -----------------------------------------

@pytest.mark.parametrize("fmt, sk, sv", FMTS)
def test_prefill_q8_equals_16bit_prefill_on_dequantised_pool(c_oracle, fmt, sk, sv):
    """Reduction to the pinned prefill oracle: with power-of-two FP8 scales the
    dequantised values are exact in fp32, so an fp32 pool holding them gives
    the same output; INT8 (code * fp32 scale needs more than fp32) is checked
    against the causal definition written out in fp64."""
    lens = [7, 1, 12, 5]
    s = _q8_setup(fmt, "f16", 6, lens)
    sk2, sv2 = (0.5, 2.0) if fmt == "fp8_e4m3" else (sk, sv)
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "f16", s["slots"],
                       fmt, sk2, sv2)
    rng = np.random.default_rng(7)
    C = [3, 1, 12, 2]                                    # queries: the last C_b positions
    cu = np.concatenate([[0], np.cumsum(C)]).astype(np.int32)
    q = wl.from_f32(rng.standard_normal((int(cu[-1]), 8, s["d"])).astype(np.float32), "f16")
    out = npo.prefill_q8(q, "f16", s["kc"], s["vc"], s["ks"], s["vs"], fmt, cu, s["tables"],
                         s["lens"], 0.3, s["hkv"], fp8_k_scale=sk2, fp8_v_scale=sv2)
    deqk = npo.dequantize(s["kc"], s["ks"], fmt, sk2)
    deqv = npo.dequantize(s["vc"], s["vs"], fmt, sv2)
    if fmt == "fp8_e4m3":
        assert np.array_equal(deqk, deqk.astype(np.float32), equal_nan=True)
        q32 = npo.to_f64(q, "f16").astype(np.float32)
        ref = npo.prefill(q32, deqk.astype(np.float32), deqv.astype(np.float32), "f32", cu,
                          s["tables"], s["lens"], 0.3, s["hkv"])
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    g = 8 // s["hkv"]
    for b, (L, c) in enumerate(zip(lens, C)):
        tb = s["tables"][b]
        for i in range(c):
            pos = L - c + i
            for h in range(8):
                K = np.stack([deqk[tb[t // s["bs"]], t % s["bs"], h // g] for t in range(pos + 1)])
                V = np.stack([deqv[tb[t // s["bs"]], t % s["bs"], h // g] for t in range(pos + 1)])
                sc = 0.3 * (K @ npo.to_f64(q[cu[b] + i, h], "f16"))
                w = np.exp(sc - sc.max())
                np.testing.assert_allclose(out[cu[b] + i, h], (w / w.sum()) @ V, rtol=0, atol=1e-12)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "int8"])
def test_prefill_q8_one_query_per_request_is_decode_q8(c_oracle, fmt):
    """C_b = 1 is a decode step: the query sits at the last position and sees
    the whole context."""
    s = _q8_setup(fmt, "bf16", 8, [9, 3, 16, 1])
    c_oracle.append_q8(s["kc"], s["vc"], s["ks"], s["vs"], s["kx"], s["vx"], "bf16", s["slots"], fmt)
    cu = np.arange(5, dtype=np.int32)
    a = npo.prefill_q8(s["q"], "bf16", s["kc"], s["vc"], s["ks"], s["vs"], fmt, cu, s["tables"],
                       s["lens"], 0.4, s["hkv"])
    d = c_oracle.decode_q8(s["q"], "bf16", s["kc"], s["vc"], s["ks"], s["vs"], fmt, s["tables"],
                           s["lens"], 0.4, s["hkv"])
    np.testing.assert_allclose(a, d, rtol=0, atol=1e-12)
