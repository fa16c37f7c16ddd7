"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks the oracle against something other than itself: IEEE 754
worked cases, numpy's independent binary16 conversion, closed forms of the
softmax, hand-worked RoPE/RMSNorm examples, and invariants the definition
implies (one key returns its value row, key-shift invariance, relative
positions of RoPE, step == row of the causal prefill, GQA == MHA with the KV
heads repeated).  The cases are chosen so that a dropped term, a swapped
operand, a wrong head offset or an off-by-one length fails at least one.
"""
import math
import os

import numpy as np
import pytest

from kv_cache_decode_asr_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(x):
    """float values -> binary16 bits via numpy (independent of the oracle)."""
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def dec(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


# ------------------------------------------------------------ binary16 ----

def test_f16_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle_mod.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signs of zeros survive
    assert math.copysign(1.0, mine[0x8000]) == -1.0


def test_f16_encode_golden_cases(oracle_mod):
    rows = []
    with open(os.path.join(GOLDEN, "f16_rne_cases.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            x = float(parts[0]) if "inf" in parts[0] else float.fromhex(parts[0])
            rows.append((x, int(parts[1], 16)))
    assert len(rows) >= 17
    xs = np.array([r[0] for r in rows], np.float32)
    assert np.array_equal(xs.astype(np.float64), np.array([r[0] for r in rows]))  # exact f32
    got = oracle_mod.f32_to_f16(xs)
    for (x, want), g in zip(rows, got):
        assert int(g) == want, f"{x!r}: got {int(g):#06x} want {want:#06x}"
    got64 = oracle_mod.f64_to_f16(xs.astype(np.float64))
    assert np.array_equal(got64, got)


def test_f16_encode_matches_numpy_random(oracle_mod):
    r = syn.rng(7)
    # a million values over the whole binary16 range and beyond: normals,
    # subnormals, overflow, random signs; plus exact ties.
    e = r.uniform(-27.0, 17.0, size=1_000_000)
    x = (np.sign(r.standard_normal(e.size)) * np.exp2(e)).astype(np.float32)
    ties = (dec(r.integers(0, 0x7bff, 20000).astype(np.uint16)) +
            dec(r.integers(0, 0x7bff, 20000).astype(np.uint16))) / 2.0
    x = np.concatenate([x, ties.astype(np.float32), np.float32([0.0, -0.0, np.inf, -np.inf])])
    mine = oracle_mod.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(mine, ref)
    # double inputs take one rounding straight to binary16 (numpy does too)
    xd = r.standard_normal(200_000) * np.exp2(r.uniform(-26, 16, 200_000))
    with np.errstate(over="ignore"):
        ref64 = xd.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle_mod.f64_to_f16(xd), ref64)


# ------------------------------------------------------------ attention ---

def _cache(B, cap, heads, hd, k, v):
    """Assemble rows K(all heads) || V(all heads) from k/v float [B, cap, heads, hd]."""
    c = np.zeros((B, cap, 2 * heads * hd), np.uint16)
    c[:, :, : heads * hd] = f16(k).reshape(B, cap, heads * hd)
    c[:, :, heads * hd:] = f16(v).reshape(B, cap, heads * hd)
    return c


def test_one_key_returns_its_value_row(oracle_mod):
    r = syn.rng(1)
    hd = 64
    k = r.standard_normal((1, 4, 2, hd))
    v = r.standard_normal((1, 4, 2, hd))
    cache = _cache(1, 4, 2, hd, k, v)
    q = r.standard_normal((1, 2 * hd)).astype(np.float32) * 10
    out, bad = oracle_mod.self_attn_step(q, cache, [1], 2, hd, hd ** -0.5)
    assert bad == 0
    want = dec(cache[0, 0, 2 * hd:])
    assert np.array_equal(out[0], want)


def test_worked_example_two_keys(oracle_mod):
    """hd=64, scale 1/8: q = (8 ln 3, 0...), k0 = e0, k1 = 0 gives scores
    (ln 3, 0), weights (3/4, 1/4); with v0 = 1, v1 = -1 the output is 0.5."""
    hd = 64
    k = np.zeros((1, 3, 1, hd))
    v = np.zeros((1, 3, 1, hd))
    k[0, 0, 0, 0] = 1.0
    v[0, 0, 0, :] = 1.0
    v[0, 1, 0, :] = -1.0
    k[0, 2, 0, 0] = 100.0   # row 2 is beyond the length: must be ignored
    v[0, 2, 0, :] = 7.0
    cache = _cache(1, 3, 1, hd, k, v)
    q = np.zeros((1, hd), np.float32)
    q[0, 0] = 8.0 * math.log(3.0)
    out, _ = oracle_mod.self_attn_step(q, cache, [2], 1, hd, 0.125)
    assert np.allclose(out[0], 0.5, atol=1e-6)
    # L = 3 includes row 2, whose score 8 ln3 * 100 / 8 dominates
    out3, _ = oracle_mod.self_attn_step(q, cache, [3], 1, hd, 0.125)
    assert np.allclose(out3[0], 7.0, atol=1e-9)


def test_two_key_sigmoid_closed_form(oracle_mod):
    r = syn.rng(2)
    hd = 64
    for trial in range(20):
        z = r.uniform(-6, 6, size=2)
        # q = 8 e0 * scale^-1 ... pick k_j = z_j e0 exactly representable
        zq = np.round(z * 64) / 64           # dyadic, exact in f16
        k = np.zeros((1, 2, 1, hd))
        k[0, :, 0, 0] = zq
        v = r.standard_normal((1, 2, 1, hd))
        cache = _cache(1, 2, 1, hd, k, v)
        q = np.zeros((1, hd), np.float32)
        q[0, 0] = 8.0                        # scores = zq
        out, _ = oracle_mod.self_attn_step(q, cache, [2], 1, hd, 0.125)
        sig = 1.0 / (1.0 + math.exp(-(zq[0] - zq[1])))
        vv = dec(cache[0, :, hd:])
        assert np.allclose(out[0], sig * vv[0] + (1 - sig) * vv[1], atol=1e-12)


def test_equal_scores_give_mean_of_values(oracle_mod):
    r = syn.rng(3)
    hd, L = 64, 1500
    kk = np.tile(r.standard_normal((1, 1, 1, hd)), (1, L, 1, 1))   # all keys equal
    v = r.standard_normal((1, L, 1, hd))
    cache = _cache(1, L, 1, hd, kk, v)
    q = r.standard_normal((1, hd)).astype(np.float32)
    out, _ = oracle_mod.cross_attn_step(q, cache, [0], 1, hd, hd ** -0.5)
    assert np.allclose(out[0], dec(cache[0, :, hd:]).mean(axis=0), atol=1e-12)
    # q = 0 gives equal scores for any keys
    k2 = r.standard_normal((1, L, 1, hd))
    cache2 = _cache(1, L, 1, hd, k2, v)
    out0, _ = oracle_mod.cross_attn_step(np.zeros((1, hd), np.float32), cache2, [0], 1, hd, 0.125)
    assert np.allclose(out0[0], dec(cache2[0, :, hd:]).mean(axis=0), atol=1e-12)


def test_heads_read_their_own_segments(oracle_mod):
    """Head h's query selects row h+1 by a huge score; the V segments of the
    heads are different constants, so a wrong K or V offset shows."""
    H, hd, L = 3, 64, 5
    k = np.zeros((1, L, H, hd))
    v = np.zeros((1, L, H, hd))
    for h in range(H):
        k[0, h + 1, h, h] = 50.0
        for j in range(L):
            v[0, j, h, :] = 10 * h + j
    cache = _cache(1, L, H, hd, k, v)
    q = np.zeros((1, H * hd), np.float32)
    for h in range(H):
        q[0, h * hd + h] = 8.0
    out, _ = oracle_mod.self_attn_step(q, cache, [L], H, hd, 0.125)
    for h in range(H):
        assert np.allclose(out[0, h * hd:(h + 1) * hd], 10 * h + h + 1, atol=1e-9)


def test_key_shift_invariance(oracle_mod):
    """Adding one vector c to every key adds q.c to every score, which the
    softmax ignores (keys and c are small dyadics, so k + c is exact in f16)."""
    r = syn.rng(4)
    H, hd, L = 2, 64, 37
    k = r.integers(-8, 9, size=(1, L, H, hd)) / 4.0
    c = r.integers(-4, 5, size=(1, 1, H, hd)) / 4.0
    v = r.standard_normal((1, L, H, hd))
    q = r.standard_normal((1, H * hd)).astype(np.float32)
    a, _ = oracle_mod.self_attn_step(q, _cache(1, L, H, hd, k, v), [L], H, hd, hd ** -0.5)
    b, _ = oracle_mod.self_attn_step(q, _cache(1, L, H, hd, k + c, v), [L], H, hd, hd ** -0.5)
    assert np.allclose(a, b, atol=1e-12)


def test_cross_group_mapping(oracle_mod):
    G, H, hd, F = 3, 2, 64, 11
    r = syn.rng(5)
    k = r.standard_normal((G, F, H, hd))
    v = np.zeros((G, F, H, hd))
    for g in range(G):
        v[g] = g + 1
    cross = _cache(G, F, H, hd, k, v)
    group = np.array([2, 0, 1, 2, 2], np.int32)
    q = r.standard_normal((5, H * hd)).astype(np.float32)
    out, bad = oracle_mod.cross_attn_step(q, cross, group, H, hd, hd ** -0.5)
    assert bad == 0
    for b in range(5):
        assert np.allclose(out[b], group[b] + 1, atol=1e-12)
    out, bad = oracle_mod.cross_attn_step(q, cross, [0, 3, -1, 1, 2], H, hd, 0.125)
    assert bad == 2 and np.all(out[1] == 0) and np.all(out[2] == 0)


def test_self_lengths_out_of_range_are_skipped(oracle_mod):
    r = syn.rng(6)
    cache = _cache(3, 4, 1, 64, r.standard_normal((3, 4, 1, 64)), r.standard_normal((3, 4, 1, 64)))
    q = r.standard_normal((3, 64)).astype(np.float32)
    out, bad = oracle_mod.self_attn_step(q, cache, [0, 4, 5], 1, 64, 0.125)
    assert bad == 2 and np.all(out[0] == 0) and np.all(out[2] == 0) and np.any(out[1] != 0)


# ------------------------------------------------------------- append ----

def test_append_matches_numpy_rounding(oracle_mod):
    r = syn.rng(8)
    B, H, hd, cap = 3, 2, 64, 6
    qkv = (r.standard_normal((B, 3 * H * hd)) * 100).astype(np.float32)
    cache = np.full((B, cap, 2 * H * hd), 0xAAAA, np.uint16)
    slot = np.array([0, 5, 6], np.int32)
    before = cache.copy()
    # k and v are views into the [q|k|v] rows (row stride 3*H*hd floats)
    kv = np.ascontiguousarray(qkv)
    k_view = kv[:, H * hd:]
    v_view = kv[:, 2 * H * hd:]
    skipped = oracle_mod._lib().orc_kv_append(
        k_view.ctypes.data_as(oracle_mod._f32p), v_view.ctypes.data_as(oracle_mod._f32p),
        3 * H * hd, cache.ctypes.data_as(oracle_mod._u16p), cap * 2 * H * hd,
        slot.ctypes.data_as(oracle_mod._i32p), B, H, hd, cap)
    assert skipped == 1
    for b in range(2):
        want = np.concatenate([f16(qkv[b, H * hd:2 * H * hd]), f16(qkv[b, 2 * H * hd:])])
        assert np.array_equal(cache[b, slot[b]], want)
        others = [s for s in range(cap) if s != slot[b]]
        assert np.array_equal(cache[b, others], before[b, others])
    assert np.array_equal(cache[2], before[2])


# ------------------------------------------------------------ rearrange --

def test_rearrange_is_a_row_gather(oracle_mod):
    r = syn.rng(9)
    B, nl, cap, row = 7, 3, 10, 16
    src = r.integers(0, 65536, size=(B, nl, cap, row)).astype(np.uint16)
    lens = r.integers(1, cap + 1, size=B).astype(np.int32)
    idx = syn.beam_permutation(B, 3, 1)
    idx[1] = idx[0]                       # repeats are allowed (take semantics)
    dst = np.full_like(src, 0x1234)
    lens_dst, bad = oracle_mod.kv_rearrange(src, dst, idx, lens, cap)
    assert bad == 0
    taken = np.take(src, idx, axis=0)
    for b in range(B):
        n = lens[idx[b]] - 1
        assert np.array_equal(dst[b, :, :n], taken[b, :, :n])
        assert np.all(dst[b, :, n:] == 0x1234)          # rows past the history untouched
    assert np.array_equal(lens_dst, lens[idx])
    # identity
    dst2 = np.zeros_like(src)
    oracle_mod.kv_rearrange(src, dst2, np.arange(B, dtype=np.int32), lens, cap)
    for b in range(B):
        assert np.array_equal(dst2[b, :, :lens[b] - 1], src[b, :, :lens[b] - 1])
    # bad index / bad length are skipped with lens_dst = 0
    lens_bad = lens.copy()
    lens_bad[2] = cap + 1
    dst3 = np.zeros_like(src)
    ld, bad = oracle_mod.kv_rearrange(src, dst3, np.array([B, 2, 0, 1, 3, 4, -1], np.int32),
                                      lens_bad, cap)
    assert bad == 3 and ld[0] == 0 and ld[1] == 0 and ld[6] == 0 and ld[2] == lens[0]


# --------------------------------------------------------- RMSNorm, RoPE --

def test_rmsnorm_worked_example(oracle_mod):
    y = oracle_mod.rmsnorm([3.0, 4.0], [1.0, 1.0], 0.0)
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5), atol=1e-15)
    y = oracle_mod.rmsnorm([3.0, 4.0], [2.0, -1.0], 1e-6)
    assert np.allclose(y, np.array([6.0, -4.0]) / math.sqrt(12.5 + 1e-6), atol=1e-15)
    r = syn.rng(10)
    x = r.standard_normal(128)
    y = oracle_mod.rmsnorm(x, np.ones(128), 0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-12
    assert np.allclose(oracle_mod.rmsnorm(7.5 * x, np.ones(128), 0.0), y, atol=1e-12)


def test_rope_worked_example_hd4():
    """hd=4, base 1e6, position 1: theta = (1, 1e-3); pairs (0,2) and (1,3)."""
    import oracle
    x = np.array([1.0, 2.0, 3.0, 4.0])
    y = oracle.rope_neox(x, 1, 1e6)
    c1, s1 = math.cos(1.0), math.sin(1.0)
    c2, s2 = math.cos(1e-3), math.sin(1e-3)
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    assert np.allclose(y, want, atol=1e-15)


def test_rope_properties(oracle_mod):
    r = syn.rng(11)
    hd = 128
    x = r.standard_normal(hd)
    k = r.standard_normal(hd)
    assert np.array_equal(oracle_mod.rope_neox(x, 0, 1e6), x)
    y = oracle_mod.rope_neox(x, 4093, 1e6)
    # norm of every (i, i + hd/2) pair is preserved (NeoX pairing)
    assert np.allclose(y[:64] ** 2 + y[64:] ** 2, x[:64] ** 2 + x[64:] ** 2, atol=1e-12)
    # the score depends on the position difference only
    d1 = oracle_mod.rope_neox(x, 3000, 1e6) @ oracle_mod.rope_neox(k, 1000, 1e6)
    d2 = oracle_mod.rope_neox(x, 2100, 1e6) @ oracle_mod.rope_neox(k, 100, 1e6)
    d3 = oracle_mod.rope_neox(x, 2000, 1e6) @ k
    assert abs(d1 - d2) < 1e-9 and abs(d1 - d3) < 1e-9
    # rotations compose
    assert np.allclose(oracle_mod.rope_neox(oracle_mod.rope_neox(x, 17, 1e6), 25, 1e6),
                       oracle_mod.rope_neox(x, 42, 1e6), atol=1e-12)


# ---------------------------------------------------- GQA step, prefill --

def _gqa_inputs(B, Hq, Hkv, hd, cap, seed):
    r = syn.rng(seed)
    q = r.standard_normal((B, Hq * hd)).astype(np.float32)
    kn = r.standard_normal((B, Hkv * hd)).astype(np.float32)
    vn = r.standard_normal((B, Hkv * hd)).astype(np.float32)
    wq = (1 + 0.1 * r.standard_normal(hd)).astype(np.float32)
    wk = (1 + 0.1 * r.standard_normal(hd)).astype(np.float32)
    cache = syn.host_normal_f16bits((B, cap, 2 * Hkv * hd), seed + 1)
    return q, kn, vn, wq, wk, cache


def test_gqa_step_equals_mha_with_repeated_kv_heads(oracle_mod):
    B, Hq, Hkv, hd, cap = 3, 4, 2, 128, 40
    q, kn, vn, wq, wk, cache = _gqa_inputs(B, Hq, Hkv, hd, cap, 12)
    n_past = np.array([0, 17, 39], np.int32)
    out, bad = oracle_mod.gqa_step(q, kn, vn, wq, wk, 1e-6, 1e6, n_past, cache, Hq, Hkv, hd,
                                   hd ** -0.5)
    assert bad == 0
    # the appended row: f16 of the normed + roped key, f16 of v
    for b in range(B):
        p = n_past[b]
        for h in range(Hkv):
            kh = oracle_mod.rope_neox(
                oracle_mod.rmsnorm(kn[b, h * hd:(h + 1) * hd].astype(np.float64), wk, 1e-6), p, 1e6)
            assert np.array_equal(cache[b, p, h * hd:(h + 1) * hd], kh.astype(np.float16).view(np.uint16))
        assert np.array_equal(cache[b, p, Hkv * hd:], f16(vn[b]))
    # MHA over the same cache with each KV head repeated for its query group
    rep = Hq // Hkv
    kpart = cache[:, :, :Hkv * hd].reshape(B, cap, Hkv, hd)
    vpart = cache[:, :, Hkv * hd:].reshape(B, cap, Hkv, hd)
    mha = np.concatenate([np.repeat(kpart, rep, axis=2).reshape(B, cap, Hq * hd),
                          np.repeat(vpart, rep, axis=2).reshape(B, cap, Hq * hd)], axis=2)
    qhat = np.zeros((B, Hq * hd), np.float64)
    for b in range(B):
        for h in range(Hq):
            qhat[b, h * hd:(h + 1) * hd] = oracle_mod.rope_neox(
                oracle_mod.rmsnorm(q[b, h * hd:(h + 1) * hd].astype(np.float64), wq, 1e-6),
                n_past[b], 1e6)
    ref, _ = oracle_mod.self_attn_step(qhat.astype(np.float32), np.ascontiguousarray(mha),
                                       n_past + 1, Hq, hd, hd ** -0.5)
    assert np.allclose(out, ref, atol=2e-6)   # q^ rounded to float32 on the MHA side
    # n_past == 0: the only key is the new one, so the output is f16(v)
    for h in range(Hq):
        assert np.array_equal(out[0, h * hd:(h + 1) * hd],
                              dec(f16(vn[0, (h // rep) * hd:(h // rep + 1) * hd])))


def test_gqa_step_bad_position_skipped(oracle_mod):
    B, Hq, Hkv, hd, cap = 2, 2, 1, 64, 8
    q, kn, vn, wq, wk, cache = _gqa_inputs(B, Hq, Hkv, hd, cap, 13)
    before = cache.copy()
    out, bad = oracle_mod.gqa_step(q, kn, vn, wq, wk, 1e-6, 1e6, [8, -1], cache, Hq, Hkv, hd, 0.125)
    assert bad == 2 and np.all(out == 0) and np.array_equal(cache, before)


def test_prefill_rows_equal_steps(oracle_mod):
    """Row t of the causal prefill equals a one-token step at position t over
    rows [0, t] of the cache the prefill wrote (GQA via repeated KV heads)."""
    B, T, Hq, Hkv, hd, cap = 2, 9, 4, 2, 64, 12
    q = syn.host_normal_f16bits((B, T, Hq * hd), 20)
    k = syn.host_normal_f16bits((B, T, Hkv * hd), 21)
    v = syn.host_normal_f16bits((B, T, Hkv * hd), 22)
    wq = syn.host_normal_f32(hd, 23, 1.0, 0.1)
    wk = syn.host_normal_f32(hd, 24, 1.0, 0.1)
    cache = np.zeros((B, cap, 2 * Hkv * hd), np.uint16)
    out, qhat = oracle_mod.prefill_attn(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, hd, hd ** -0.5, cache)
    assert np.array_equal(cache[:, :T, Hkv * hd:], v)          # V copied bitwise
    assert np.all(cache[:, T:] == 0)                          # nothing past T
    rep = Hq // Hkv
    kpart = cache[:, :, :Hkv * hd].reshape(B, cap, Hkv, hd)
    vpart = cache[:, :, Hkv * hd:].reshape(B, cap, Hkv, hd)
    mha = np.ascontiguousarray(np.concatenate(
        [np.repeat(kpart, rep, axis=2).reshape(B, cap, Hq * hd),
         np.repeat(vpart, rep, axis=2).reshape(B, cap, Hq * hd)], axis=2))
    for t in range(T):
        qt = dec(qhat[:, t]).astype(np.float32)
        ref, _ = oracle_mod.self_attn_step(qt, mha, np.full(B, t + 1, np.int32), Hq, hd, hd ** -0.5)
        assert np.allclose(out[:, t], ref, atol=1e-12)
    # the first position has one key: its output is that V row
    for h in range(Hq):
        assert np.array_equal(out[:, 0, h * hd:(h + 1) * hd], dec(v[:, 0, (h // rep) * hd:(h // rep + 1) * hd]))
    # causality: changing later keys does not move earlier rows
    k2 = k.copy()
    k2[:, 5:] = syn.host_normal_f16bits(k2[:, 5:].shape, 25)
    out2, _ = oracle_mod.prefill_attn(q, k2, v, wq, wk, 1e-6, 1e6, Hq, Hkv, hd, hd ** -0.5,
                                      np.zeros_like(cache))
    assert np.array_equal(out2[:, :5], out[:, :5])
    assert not np.allclose(out2[:, 5:], out[:, 5:])
    # the preparation alone writes the same cache and queries
    cache_p = np.zeros_like(cache)
    qhat_p = oracle_mod.prefill_prep(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, hd, cache_p)
    assert np.array_equal(cache_p, cache) and np.array_equal(qhat_p, qhat)
    # sampled rows through the per-row entry point agree
    ts = np.array([0, 3, 8], np.int32)
    rows = oracle_mod.prefill_attn_rows(qhat[1, ts, 3 * hd:4 * hd], ts, cache[1], Hq, Hkv, hd, 3,
                                        hd ** -0.5)
    assert np.array_equal(rows, out[1, ts, 3 * hd:4 * hd])


def test_step_key_equals_prefill_key(oracle_mod):
    """A key appended by the step at n_past = p is bit-identical to the key the
    prefill writes at row p from the same input values."""
    B, T, Hq, Hkv, hd, cap = 1, 6, 2, 2, 128, 8
    q = syn.host_normal_f16bits((B, T, Hq * hd), 30)
    k = syn.host_normal_f16bits((B, T, Hkv * hd), 31)
    v = syn.host_normal_f16bits((B, T, Hkv * hd), 32)
    wq = syn.host_normal_f32(hd, 33, 1.0, 0.1)
    wk = syn.host_normal_f32(hd, 34, 1.0, 0.1)
    pre = np.zeros((B, cap, 2 * Hkv * hd), np.uint16)
    outp, _ = oracle_mod.prefill_attn(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, hd, hd ** -0.5, pre)
    step = pre.copy()
    step[:, T - 1] = 0
    outs, _ = oracle_mod.gqa_step(dec(q[:, T - 1]).astype(np.float32),
                                  dec(k[:, T - 1]).astype(np.float32),
                                  dec(v[:, T - 1]).astype(np.float32), wq, wk, 1e-6, 1e6,
                                  [T - 1], step, Hq, Hkv, hd, hd ** -0.5)
    assert np.array_equal(step, pre)
    # outputs differ only by the f16 rounding of the prefill's query
    assert np.allclose(outs[0], outp[0, T - 1], atol=2e-2)


# ------------------------------------------- MHA prompt prefill, encoder ----

def _np_attention(q, k, v, heads, hd, scale, causal, L):
    """Textbook softmax(scale q k^T) v in float64 with numpy, over the first L
    positions of one sequence (q, k, v: f16 bits [T, heads*hd])."""
    qd, kd, vd = dec(q), dec(k), dec(v)
    out = np.full(qd.shape, np.nan)
    for h in range(heads):
        sl = slice(h * hd, (h + 1) * hd)
        s = scale * qd[:L, sl] @ kd[:L, sl].T
        if causal:
            s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:L, sl] = (p / p.sum(axis=1, keepdims=True)) @ vd[:L, sl]
    return out


def test_mha_attn_matches_numpy_brute_force(oracle_mod):
    """Tiny causal and unmasked cases with per-sequence lengths against a
    numpy restatement (independent f16 decode, matrix form)."""
    B, T, H, hd = 3, 6, 2, 4
    q = syn.host_normal_f16bits((B, T, H * hd), 40)
    k = syn.host_normal_f16bits((B, T, H * hd), 41)
    v = syn.host_normal_f16bits((B, T, H * hd), 42)
    lens = np.array([6, 3, 1], np.int32)
    for causal in (True, False):
        out, bad = oracle_mod.mha_attn(q, k, v, H, hd, 0.7, causal, lens=lens)
        assert bad == 0
        for b in range(B):
            ref = _np_attention(q[b], k[b], v[b], H, hd, 0.7, causal, lens[b])
            assert np.allclose(out[b, :lens[b]], ref[:lens[b]], rtol=1e-12, atol=1e-12)
            assert np.all(np.isnan(out[b, lens[b]:]))        # rows past the length untouched
    # one real position: its output is its own V row, exactly
    out, _ = oracle_mod.mha_attn(q, k, v, H, hd, 0.7, False, lens=np.array([1, 1, 1], np.int32))
    assert np.array_equal(out[:, 0], dec(v[:, 0]))


def test_mha_prefill_rows_equal_steps_and_cache(oracle_mod):
    """Causal row t equals the one-token self-attention step over the cache
    rows [0, t] the prefill wrote; the cache rows are k || v bitwise and
    nothing is written past a sequence's length."""
    B, T, H, hd, cap = 2, 7, 3, 64, 9
    q = syn.host_normal_f16bits((B, T, H * hd), 43)
    k = syn.host_normal_f16bits((B, T, H * hd), 44)
    v = syn.host_normal_f16bits((B, T, H * hd), 45)
    lens = np.array([7, 4], np.int32)
    cache = np.zeros((B, cap, 2 * H * hd), np.uint16)
    out, bad = oracle_mod.mha_attn(q, k, v, H, hd, hd ** -0.5, True, lens=lens, cache=cache)
    assert bad == 0
    for b in range(B):
        L = lens[b]
        assert np.array_equal(cache[b, :L, :H * hd], k[b, :L])
        assert np.array_equal(cache[b, :L, H * hd:], v[b, :L])
        assert np.all(cache[b, L:] == 0)
    for t in range(T):
        live = np.nonzero(lens > t)[0]
        qt = dec(q[live, t]).astype(np.float32)
        ref, _ = oracle_mod.self_attn_step(qt, np.ascontiguousarray(cache[live]),
                                           np.full(live.size, t + 1, np.int32), H, hd, hd ** -0.5)
        assert np.allclose(out[live, t], ref, atol=1e-12)


def test_encoder_attn_rows_equal_cross_step(oracle_mod):
    """Unmasked: every row equals the one-query cross-attention over all the
    sequence's frames, and a shorter length equals the truncated sequence."""
    B, T, H, hd = 2, 10, 2, 64
    q = syn.host_normal_f16bits((B, T, H * hd), 46)
    k = syn.host_normal_f16bits((B, T, H * hd), 47)
    v = syn.host_normal_f16bits((B, T, H * hd), 48)
    out, _ = oracle_mod.mha_attn(q, k, v, H, hd, hd ** -0.5, False)
    cross = np.ascontiguousarray(np.concatenate([k, v], axis=2))  # [B][T][K | V]
    for t in (0, 4, 9):
        ref, _ = oracle_mod.cross_attn_step(dec(q[:, t]).astype(np.float32), cross,
                                            np.arange(B, dtype=np.int32), H, hd, hd ** -0.5)
        assert np.allclose(out[:, t], ref, atol=1e-12)
    L = 6
    out_l, _ = oracle_mod.mha_attn(q, k, v, H, hd, hd ** -0.5, False,
                                   lens=np.array([L, L], np.int32))
    out_t, _ = oracle_mod.mha_attn(np.ascontiguousarray(q[:, :L]), np.ascontiguousarray(k[:, :L]),
                                   np.ascontiguousarray(v[:, :L]), H, hd, hd ** -0.5, False)
    assert np.array_equal(out_l[:, :L], out_t)
    # the encoder attends to every frame: changing the last key moves row 0
    k2 = k.copy()
    k2[:, T - 1] = syn.host_normal_f16bits(k2[:, T - 1].shape, 49)
    out2, _ = oracle_mod.mha_attn(q, k2, v, H, hd, hd ** -0.5, False)
    assert not np.allclose(out2[:, 0], out[:, 0])
    # a length outside [0, T] is counted and skipped
    _, bad = oracle_mod.mha_attn(q, k, v, H, hd, hd ** -0.5, False, lens=np.array([T + 1, 3], np.int32))
    assert bad == 1


# ----------------------------------------------------------- cross K/V fill ----

def test_cross_kv_fill_matches_numpy_and_closed_forms(oracle_mod):
    """The fill against numpy's float64 matmul of the decoded f16 operands
    (then numpy's own f16 rounding); identity weights return the encoder
    rows (K) and the rows plus the bias (V); a zero input gives K = 0 and
    V = f16(bias); rows past the frames are untouched."""
    G, frames, d, cap = 2, 5, 16, 7
    enc = syn.host_normal_f16bits((G, frames, d), 50)
    w = f16(syn.host_normal_f32((2 * d, d), 51) * d ** -0.5)
    bias = syn.host_normal_f32(d, 52)
    cross0 = syn.host_normal_f16bits((G, cap, 2 * d), 53)
    cross = cross0.copy()
    oracle_mod.cross_kv_fill(enc, w, bias, cross)
    ref = dec(enc) @ dec(w).T
    ref[..., d:] += bias.astype(np.float64)
    # numpy rounds the float64 result straight to binary16 (nearest even)
    assert np.array_equal(cross[:, :frames], ref.astype(np.float16).view(np.uint16))
    assert np.array_equal(cross[:, frames:], cross0[:, frames:])
    # identity weights: K = enc exactly, V = f16(enc + bias)
    eye = np.zeros((2 * d, d), np.float32)
    eye[np.arange(d), np.arange(d)] = 1
    eye[d + np.arange(d), np.arange(d)] = 1
    c2 = np.zeros_like(cross0)
    oracle_mod.cross_kv_fill(enc, f16(eye), bias, c2)
    assert np.array_equal(c2[:, :frames, :d], enc)
    want_v = (dec(enc) + bias.astype(np.float64)).astype(np.float16).view(np.uint16)
    assert np.array_equal(c2[:, :frames, d:], want_v)
    # zero input
    c3 = np.zeros_like(cross0)
    oracle_mod.cross_kv_fill(np.zeros_like(enc), w, bias, c3)
    assert np.all(c3[:, :frames, :d] == 0)
    assert np.array_equal(c3[:, :frames, d:], np.broadcast_to(f16(bias), (G, frames, d)))


# ------------------------------------------- dense steps of a decoder layer --

def test_layer_norm_worked_examples(oracle_mod):
    """torch.nn.LayerNorm's definition: biased variance, eps inside the root.
    [1, 2, 3, 4] has mean 2.5 and variance 1.25 (the unbiased 5/3 would fail);
    an alternating row +-a normalises to +-a/sqrt(a^2 + eps); a constant row
    gives the bias exactly; the weight scales and the bias shifts."""
    one = np.ones(4, np.float32)
    zero = np.zeros(4, np.float32)
    y = oracle_mod.layer_norm(np.array([[1, 2, 3, 4]], np.float32), one, zero, eps=0.0)
    want = np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25)
    np.testing.assert_allclose(y[0], want, rtol=0, atol=1e-15)
    a, eps = 2.0, 1e-5
    row = np.array([[a, -a, a, -a, a, -a]], np.float32)
    y = oracle_mod.layer_norm(row, np.ones(6, np.float32), np.zeros(6, np.float32), eps=eps)
    s = a / math.sqrt(a * a + eps)
    np.testing.assert_allclose(y[0], [s, -s, s, -s, s, -s], rtol=0, atol=1e-15)
    b = np.array([0.25, -1.0, 3.0, 0.5], np.float32)
    y = oracle_mod.layer_norm(np.full((1, 4), 7.5, np.float32), one, b, eps=eps)
    assert np.array_equal(y[0], b.astype(np.float64))
    g = np.array([2.0, -1.0, 0.5, 3.0], np.float32)
    x = np.array([[0.3, -1.2, 2.5, 0.1]], np.float32)
    y0 = oracle_mod.layer_norm(x, one, zero, eps=eps)
    y1 = oracle_mod.layer_norm(x, g, b, eps=eps)
    np.testing.assert_allclose(y1, y0 * g + b, rtol=0, atol=1e-14)
    # random rows: zero mean, mean square var / (var + eps)
    xr = syn.host_normal_f32((5, 64), 60, mean=0.7, std=2.0)
    yr = oracle_mod.layer_norm(xr, np.ones(64, np.float32), np.zeros(64, np.float32), eps=eps)
    var = xr.astype(np.float64).var(axis=1)
    np.testing.assert_allclose(yr.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose((yr ** 2).mean(axis=1), var / (var + eps), rtol=1e-12)


def test_gelu_erf_table_values(oracle_mod):
    """gelu(v) = v * Phi(v), Phi the standard normal CDF: Phi(1) =
    0.8413447460685429, Phi(2) = 0.9772498680518208 (normal tables); gelu(v)
    - gelu(-v) = v; the tanh approximation (0.8411919906 at 1) is not it."""
    g = oracle_mod.gelu_erf(np.array([0.0, 1.0, -1.0, 2.0, -2.0]))
    np.testing.assert_allclose(g, [0.0, 0.8413447460685429, -0.15865525393145707,
                                   1.9544997361036416, -0.04550026389635842], rtol=0,
                               atol=1e-15)
    v = syn.host_normal_f32(50, 61, std=3.0).astype(np.float64)
    np.testing.assert_allclose(oracle_mod.gelu_erf(v) - oracle_mod.gelu_erf(-v), v, atol=1e-14)
    assert abs(oracle_mod.gelu_erf(1.0) - 0.8411919906082768) > 1e-4


def test_linear_matches_numpy_and_closed_forms(oracle_mod):
    """The dense step against numpy's float64 matmul of the decoded f16
    weights, in each mode; identity weights return x (+ bias); zero weights
    leave the residual untouched; LayerNorm of an alternating row is its
    closed form before the product."""
    M, K, N = 3, 64, 40
    x = syn.host_normal_f32((M, K), 62)
    w = f16(syn.host_normal_f32((N, K), 63) * K ** -0.5)
    bias = syn.host_normal_f32(N, 64)
    y0 = syn.host_normal_f32((M, N), 65)
    ref = x.astype(np.float64) @ dec(w).T + bias
    np.testing.assert_allclose(oracle_mod.linear(x, w, bias), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle_mod.linear(x, w, bias, mode="residual", y=y0),
                               y0 + ref, rtol=0, atol=1e-12)
    gref = 0.5 * ref * (1 + np.vectorize(math.erf)(ref / math.sqrt(2)))
    np.testing.assert_allclose(oracle_mod.linear(x, w, bias, mode="gelu"), gref, rtol=0,
                               atol=1e-12)
    np.testing.assert_allclose(oracle_mod.linear(x, w, None), ref - bias, rtol=0, atol=1e-12)
    eye = f16(np.eye(K, dtype=np.float32))
    bk = syn.host_normal_f32(K, 66)
    np.testing.assert_allclose(oracle_mod.linear(x, eye, bk), x.astype(np.float64) + bk,
                               rtol=0, atol=0)
    zw = np.zeros((N, K), np.uint16)
    assert np.array_equal(oracle_mod.linear(x, zw, None, mode="residual", y=y0),
                          y0.astype(np.float64))
    # LayerNorm first: rows +-a normalise to +-a/sqrt(a^2+eps), then g, b
    a, eps = 1.5, 1e-5
    alt = np.tile(np.array([a, -a], np.float32), (M, K // 2))
    g = syn.host_normal_f32(K, 67, mean=1.0, std=0.1)
    b = syn.host_normal_f32(K, 68, std=0.1)
    s = a / math.sqrt(a * a + eps)
    an = np.tile(np.array([s, -s]), (M, K // 2)) * g + b
    np.testing.assert_allclose(oracle_mod.linear(alt, w, bias, ln=(g, b), eps=eps),
                               an @ dec(w).T + bias, rtol=0, atol=1e-12)


def _layer_params(d, inner, seed, zero_out=False):
    p = {}
    for i, (name, n_out, n_in) in enumerate((("qkv", 3 * d, d), ("o", d, d), ("cq", d, d),
                                              ("co", d, d), ("fc1", inner, d),
                                              ("fc2", d, inner))):
        w = syn.host_normal_f32((n_out, n_in), seed + 2 * i) * n_in ** -0.5
        if zero_out and name in ("o", "co", "fc2"):
            w[:] = 0
        p["w_" + name] = f16(w)
        p["b_" + name] = syn.host_normal_f32(n_out, seed + 2 * i + 1, std=0.1)
    p["b_qkv"][d:2 * d] = 0  # the key projection has no bias
    for j in (1, 2, 3):
        p[f"ln{j}_g"] = syn.host_normal_f32(d, seed + 20 + j, mean=1.0, std=0.1)
        p[f"ln{j}_b"] = syn.host_normal_f32(d, seed + 30 + j, std=0.1)
    return p


def test_decoder_layer_step_residuals_and_cache(oracle_mod):
    """With the three output projections zero, the layer adds exactly its
    three output biases to x (each sum rounded to f32, as the buffers are
    f32); the new token's k, v land in cache row lens-1 as f16 of the
    LayerNorm-ed projection and no other row changes.  With identity output
    projections the two attentions' outputs are added onto the stream."""
    B, H, hd, cap, F = 3, 2, 8, 6, 5
    d, inner = H * hd, 4 * H * hd
    x = syn.host_normal_f32((B, d), 70)
    lens = np.array([1, 4, 6], np.int32)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * d), 71)
    cross = syn.host_normal_f16bits((2, F, 2 * d), 72)
    group = np.array([0, 0, 1], np.int32)
    p = _layer_params(d, inner, 80, zero_out=True)
    cache = cache0.copy()
    xo, mid = oracle_mod.whisper_decoder_layer_step(x, p, cache, lens, cross, group, H, hd)
    x1 = (x.astype(np.float64) + p["b_o"]).astype(np.float32)
    x2 = (x1.astype(np.float64) + p["b_co"]).astype(np.float32)
    x3 = (x2.astype(np.float64) + p["b_fc2"]).astype(np.float32)
    assert np.array_equal(xo, x3)
    ln1 = oracle_mod.layer_norm(x, p["ln1_g"], p["ln1_b"])
    kv = ln1 @ dec(p["w_qkv"][d:]).T + p["b_qkv"][d:]
    for bi in range(B):
        assert np.array_equal(cache[bi, lens[bi] - 1], f16(kv[bi].astype(np.float32)))
        keep = np.arange(cap) != lens[bi] - 1
        assert np.array_equal(cache[bi, keep], cache0[bi, keep])
    # identity output projections: x1 = x + self-attention, x2 = x1 + cross
    p = _layer_params(d, inner, 90, zero_out=True)
    p["w_o"] = f16(np.eye(d, dtype=np.float32))
    p["w_co"] = f16(np.eye(d, dtype=np.float32))
    for k in ("b_o", "b_co", "b_fc2"):
        p[k][:] = 0
    cache = cache0.copy()
    xo, mid = oracle_mod.whisper_decoder_layer_step(x, p, cache, lens, cross, group, H, hd)
    scale = hd ** -0.5
    att, _ = oracle_mod.self_attn_step(mid["qkv"], cache, lens, H, hd, scale, q_stride=3 * d)
    assert np.array_equal(mid["x1"], (x.astype(np.float64) + att.astype(np.float32)).astype(
        np.float32))
    attc, _ = oracle_mod.cross_attn_step(mid["qx"], cross, group, H, hd, scale)
    assert np.array_equal(xo, (mid["x1"].astype(np.float64) + attc.astype(np.float32)).astype(
        np.float32))


def test_silu_values(oracle_mod):
    """silu(v) = v * sigmoid(v): silu(0) = 0, silu(1) = 1/(1 + 1/e) =
    0.7310585786300049, silu(v) - silu(-v) = v, and silu(30) = 30 - 2.807e-12
    (30 e^-30 below 30)."""
    np.testing.assert_allclose(oracle_mod.silu([0.0, 1.0, -1.0, 30.0]),
                               [0.0, 0.7310585786300049, -0.2689414213699951, 29.999999999997193],
                               rtol=0, atol=1e-14)
    v = syn.host_normal_f32(40, 90, std=4.0).astype(np.float64)
    np.testing.assert_allclose(oracle_mod.silu(v) - oracle_mod.silu(-v), v, atol=1e-13)


def test_linear_rms_and_swiglu(oracle_mod):
    """RMSNorm before the product equals the (pinned) per-vector RMSNorm of
    each row, then numpy's matmul; a row of equal values c normalises to
    c/sqrt(c^2 + eps) * w; the SwiGLU input is silu(gate) * up of the two
    halves of each row (numpy brute force with the closed-form sigmoid)."""
    M, K, N = 3, 64, 24
    x = syn.host_normal_f32((M, K), 91, mean=0.2, std=1.3)
    w = f16(syn.host_normal_f32((N, K), 92) * K ** -0.5)
    g = syn.host_normal_f32(K, 93, mean=1.0, std=0.1)
    eps = 1e-6
    a = np.stack([oracle_mod.rmsnorm(x[m].astype(np.float64), g.astype(np.float64), eps)
                  for m in range(M)])
    np.testing.assert_allclose(oracle_mod.linear(x, w, None, rms=g, eps=eps), a @ dec(w).T,
                               rtol=0, atol=1e-12)
    c = np.float32(1.75)
    flat = np.full((1, K), c, np.float32)
    want = (float(c) / math.sqrt(float(c) ** 2 + eps) * g.astype(np.float64)) @ dec(w).T
    np.testing.assert_allclose(oracle_mod.linear(flat, w, None, rms=g, eps=eps)[0], want,
                               rtol=0, atol=1e-12)
    xg = syn.host_normal_f32((M, 2 * K), 94, std=2.0)
    gate, up = xg[:, :K].astype(np.float64), xg[:, K:].astype(np.float64)
    act = gate / (1.0 + np.exp(-gate)) * up
    y0 = syn.host_normal_f32((M, N), 95)
    np.testing.assert_allclose(oracle_mod.linear(xg, w, None, mode="residual", y=y0, swiglu=True),
                               y0 + act @ dec(w).T, rtol=0, atol=1e-12)


def test_qwen3_decoder_layer_step_residuals_and_cache(oracle_mod):
    """With the output and down projections zero the layer leaves x
    unchanged; the new k, v land in cache row n_past as the GQA step writes
    them; otherwise the attention output goes through w_o onto the stream and
    the MLP adds silu(gate) * up through w_down (numpy brute force)."""
    B, Hq, Hkv, hd, cap, d, inner = 2, 4, 2, 64, 8, 128, 192
    x = syn.host_normal_f32((B, d), 96)
    n_past = np.array([0, 5], np.int32)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * Hkv * hd), 97)
    nq, nk = Hq * hd, Hkv * hd

    def params(seed, zero_out):
        p = {"w_qkv": f16(syn.host_normal_f32((nq + 2 * nk, d), seed) * d ** -0.5),
             "w_o": f16(np.zeros((d, nq), np.float32) if zero_out else
                        syn.host_normal_f32((d, nq), seed + 1) * nq ** -0.5),
             "w_gu": f16(syn.host_normal_f32((2 * inner, d), seed + 2) * d ** -0.5),
             "w_down": f16(np.zeros((d, inner), np.float32) if zero_out else
                           syn.host_normal_f32((d, inner), seed + 3) * inner ** -0.5),
             "rms1": syn.host_normal_f32(d, seed + 4, mean=1.0, std=0.1),
             "rms2": syn.host_normal_f32(d, seed + 5, mean=1.0, std=0.1),
             "q_norm": syn.host_normal_f32(hd, seed + 6, mean=1.0, std=0.1),
             "k_norm": syn.host_normal_f32(hd, seed + 7, mean=1.0, std=0.1)}
        return p

    p = params(100, True)
    cache = cache0.copy()
    xo, mid = oracle_mod.qwen3_decoder_layer_step(x, p, cache, n_past, Hq, Hkv, hd)
    assert np.array_equal(xo, x)
    ref = cache0.copy()
    qkv = mid["qkv"]
    oracle_mod.gqa_step(np.ascontiguousarray(qkv[:, :nq]), np.ascontiguousarray(qkv[:, nq:nq + nk]),
                        np.ascontiguousarray(qkv[:, nq + nk:]), p["q_norm"], p["k_norm"], 1e-6,
                        1e6, n_past, ref, Hq, Hkv, hd, hd ** -0.5)
    assert np.array_equal(cache, ref)
    # non-zero output and down projections: each adds its product onto the stream
    p = params(200, False)
    cache = cache0.copy()
    xo, mid = oracle_mod.qwen3_decoder_layer_step(x, p, cache, n_past, Hq, Hkv, hd)
    x1 = (x.astype(np.float64) + mid["att"].astype(np.float64) @ dec(p["w_o"]).T).astype(
        np.float32)
    np.testing.assert_allclose(mid["x1"], x1, rtol=0, atol=1e-6)
    gate, up = mid["gu"][:, :inner].astype(np.float64), mid["gu"][:, inner:].astype(np.float64)
    x2 = (x1.astype(np.float64) + (gate / (1 + np.exp(-gate)) * up) @ dec(p["w_down"]).T).astype(
        np.float32)
    np.testing.assert_allclose(xo, x2, rtol=0, atol=1e-6)
