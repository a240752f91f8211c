"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against a closed form, an invariant, a library
routine (numpy / scipy), a hand-derived fixture under tests/golden/, or a
brute-force re-computation, so that a dropped term, a wrong sign or index or
a transposed operand in oracle/ fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import numerics as L
from kv_cache_decode_flash_gb300 import synth
from golden_io import q4_0_blocks, q8_0_blocks, hexfile

# ---------------------------------------------------------------- fp16 ----


def test_f16_roundtrip_exhaustive():
    h = np.arange(65536, dtype=np.uint16)
    e = (h >> 10) & 31
    m = h & 1023
    finite_or_inf = ~((e == 31) & (m != 0))
    h = h[finite_or_inf]
    x = oracle.f16_to_f64(h)
    back = np.array([L.lib.orc_f64_to_f16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(back, h)


def test_f16_decode_known_values():
    known = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0**-24, 0x0400: 2.0**-14, 0x7BFF: 65504.0,
             0x3555: 0.333251953125, 0x7C00: math.inf, 0xFC00: -math.inf, 0x8000: -0.0}
    for bits, val in known.items():
        assert oracle.f16_to_f64(np.array([bits]))[0] == val


def test_f16_encode_matches_numpy():
    # numpy's float32 -> float16 cast is an IEEE round-to-nearest-even library routine
    rng_bits = synth.raw_u64(0, synth.stream_id("misc", extra=1), 200000)
    f = (rng_bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    f = f[np.isfinite(f)]
    # concentrate on the fp16 range, subnormals and the overflow edge
    scaled = np.concatenate([f, f * np.float32(1e-30), np.float32([65504, 65519.996, 65520, 6e-8,
                                                                   2.0**-25, 3 * 2.0**-25])])
    scaled = scaled[np.isfinite(scaled)].astype(np.float32)
    ref = scaled.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(scaled)
    assert np.array_equal(got, ref)


def test_f16_ties_to_even():
    cases = [(1 + 2.0**-11, 0x3C00), (1 + 3 * 2.0**-11, 0x3C02), (2.0**-25, 0x0000),
             (3 * 2.0**-25, 0x0002), (65520.0, 0x7C00), (-65520.0, 0xFC00), (65519.0, 0x7BFF)]
    for x, bits in cases:
        assert L.lib.orc_f64_to_f16(x) == bits, x


# ---------------------------------------------------------------- q8_0 ----


@pytest.mark.parametrize("blk", q8_0_blocks(), ids=lambda b: b[0])
def test_q8_0_golden_blocks(blk):
    name, x, q, sc = blk
    codes, scales = oracle.q8_0_quantize(x)
    assert np.array_equal(codes, q)
    assert int(scales[0]) == sc


@pytest.mark.parametrize("c", [1.0, -1.0, 0.0, 3.25, -1e-3, 7e-5, 1234.5, -65.0])
def test_q8_0_all_equal_block(c):
    x = np.full(32, c, np.float32)
    codes, scales = oracle.q8_0_quantize(x)
    want = 0 if c == 0 else int(math.copysign(127, c))
    assert (codes == want).all()
    d32 = np.float32(abs(np.float32(c))) / np.float32(127)
    assert scales[0] == np.float16(d32).view(np.uint16)


def _blocks(n, seed=0, sigma=1.0):
    return synth.normal(seed, synth.stream_id("misc", extra=2), 32 * n, sigma).reshape(n, 32)


def test_q8_0_max_element_is_127():
    x = _blocks(2000)
    codes, _ = oracle.q8_0_quantize(x)
    i = np.abs(x).argmax(1)
    top = codes[np.arange(len(x)), i].astype(int)
    assert np.array_equal(np.abs(top), np.full(len(x), 127))
    assert np.array_equal(np.sign(top), np.sign(x[np.arange(len(x)), i]).astype(int))
    assert np.abs(codes.astype(int)).max() <= 127


def test_q8_0_exact_multiples():
    k = synth.randint(3, synth.stream_id("misc", extra=3), 32 * 500, -127, 127).reshape(500, 32)
    k[:, 0] = 127  # fixes amax = 127 * d
    d = np.float32(0.0371)
    x = (k.astype(np.float32) * d).astype(np.float32)
    codes, _ = oracle.q8_0_quantize(x)
    assert np.array_equal(codes.astype(int), k)


def test_q8_0_error_bound():
    x = _blocks(4000, sigma=0.5)
    codes, scales = oracle.q8_0_quantize(x)
    xh = oracle.q8_0_dequantize(codes, scales)
    amax = np.abs(x).max(1).astype(np.float64)
    d = amax / 127.0
    dh = oracle.f16_to_f64(scales[:, 0])
    bound = d / 2 + 127 * np.abs(d - dh) + 1e-6 * amax
    assert (np.abs(xh - x).max(1) <= bound).all()


def test_q8_0_dequant_exact_in_fp32():
    # float(fp16 scale) * code has at most 11 + 8 significant bits: exact in fp32
    scales = oracle.f32_to_f16(np.float32([1e-4, 0.0078, 0.5, 1.0, 3.7, 250.0, 6e-6]))
    for s in scales:
        codes = np.arange(-128, 128, dtype=np.int8)
        v64 = oracle.q8_0_dequantize(codes.reshape(8, 32), np.full((8, 1), s, np.uint16)).ravel()
        v32 = np.float32(np.array([s], np.uint16).view(np.float16)[0]) * codes.astype(np.float32)
        assert np.array_equal(v64, v32.astype(np.float64))


# ---------------------------------------------------------------- q4_0 ----


def _nibble_decode(packed, scale_bits):
    """Values of one packed q4_0 block read directly off the stated layout:
    element i sits in byte i % 16, low four bits for i < 16, high for i >= 16."""
    d = oracle.f16_to_f64(np.array([scale_bits], np.uint16))[0]
    return np.array([(((int(packed[i % 16]) >> (4 * (i // 16))) & 15) - 8) * d for i in range(32)])


@pytest.mark.parametrize("blk", q4_0_blocks(), ids=lambda b: b[0])
def test_q4_0_golden_blocks(blk):
    name, x, codes, packed, scale = blk
    got_p, got_s = oracle.q4_0_quantize(x.reshape(1, 32))
    assert got_p[0].tobytes() == packed.tobytes(), name
    assert int(got_s[0, 0]) == scale, name
    # the codes of the fixture, packed by hand, are the fixture's bytes
    assert bytes(int(codes[j]) | (int(codes[j + 16]) << 4) for j in range(16)) == packed.tobytes()
    np.testing.assert_array_equal(oracle.q4_0_dequantize(got_p, got_s)[0], _nibble_decode(packed, scale))


def test_q4_0_largest_element_decodes_to_itself_and_codes_stay_in_range():
    x = synth.normal(21, synth.stream_id("misc", extra=21), 4096 * 32).astype(np.float32).reshape(-1, 32)
    p, sc = oracle.q4_0_quantize(x)
    v = oracle.q4_0_dequantize(p, sc)
    d16 = oracle.f16_to_f64(sc)[:, 0]
    idx = np.argmax(np.abs(x), axis=1)  # numpy's argmax takes the first maximum, as the reading does
    m = x[np.arange(len(x)), idx].astype(np.float64)
    # code 0 decodes to -8 * fp16(m / -8)
    np.testing.assert_array_equal(v[np.arange(len(x)), idx], -8.0 * d16)
    # and -8 * fp16(m / -8) is m up to the scale's fp16 rounding
    assert (np.abs(-8.0 * d16 - m) <= 8 * 2.0**-11 * np.abs(m) + 2.0**-21).all()
    # every decoded value lies on the grid (c - 8) * fp16(d), c in 0..15
    c = np.rint(v / np.where(d16 == 0, 1, d16)[:, None]) + 8
    assert ((c >= 0) & (c <= 15)).all()


def test_q4_0_error_bound():
    # |x - x^| <= |d| / 2 + 8 |d - fp16(d)| away from the clamped top code, and at most
    # |d| + 8 |d - fp16(d)| where x * id rounds past 15 (the asymmetric clamp of the format)
    x = synth.normal(22, synth.stream_id("misc", extra=22), 2048 * 32).astype(np.float32).reshape(-1, 32)
    p, sc = oracle.q4_0_quantize(x)
    v = oracle.q4_0_dequantize(p, sc)
    d16 = oracle.f16_to_f64(sc)[:, 0][:, None]
    m = x[np.arange(len(x)), np.argmax(np.abs(x), axis=1)].astype(np.float64)[:, None]
    d = m / -8.0
    slack = 8 * np.abs(d - d16) + 1e-6 * np.abs(d)
    t = x / d
    err = np.abs(x - v)
    inner = t < 7.5 - 1e-5  # below the clamped top code
    assert (err <= np.abs(d) / 2 + slack + np.where(inner, 0.0, np.abs(d) / 2)).all()
    assert (np.abs(x - v)[~inner] <= np.abs(d)[np.nonzero(~inner)[0]][:, 0] + 1e-6).all()


def test_q4_0_attention_closed_forms():
    # identical V rows: any softmax gives that row back; K q8_0 as in the asymmetric cache
    H, Hk, D, n = 8, 2, 64, 40
    (kc, ks), _ = _cache(n, Hk, D, 23)
    vrow = synth.normal(23, synth.stream_id("v"), Hk * D).astype(np.float32).reshape(1, Hk, D)
    vp, vs = oracle.q4_0_quantize(np.repeat(vrow, n, axis=0))
    q = synth.normal(23, synth.stream_id("q"), H * D).reshape(H, D)
    out = oracle.attn(q, L.Q8_0, kc, ks, L.Q4_0, vp, vs, 0.125)
    V = oracle.q4_0_dequantize(vp, vs)
    for h in range(H):
        np.testing.assert_allclose(out[h], V[0, h // 4], rtol=0, atol=1e-14)
    # random V: the two-pass oracle against the per-token long-double formulation and
    # against numpy / scipy over the decoded values
    v = synth.normal(24, synth.stream_id("v"), n * Hk * D).reshape(n, Hk, D)
    vp, vs = oracle.q4_0_quantize(v)
    a = oracle.attn(q, L.Q8_0, kc, ks, L.Q4_0, vp, vs, 0.125)
    b = oracle.attn_bruteforce(q, L.Q8_0, kc, ks, L.Q4_0, vp, vs, 0.125)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    K, V = oracle.q8_0_dequantize(kc, ks), oracle.q4_0_dequantize(vp, vs)
    for h in range(H):
        p_ = scipy.special.softmax(0.125 * (K[:, h // 4, :] @ q[h].astype(np.float64)))
        np.testing.assert_allclose(a[h], p_ @ V[:, h // 4, :], rtol=1e-12, atol=1e-13)


def test_q4_0_state_layout_and_roundtrip():
    c = oracle.OracleCache(2, 4, 2, 64, L.Q8_0, L.Q4_0, 10000.0, 0)
    for l in range(2):
        k = synth.normal(25, synth.stream_id("k", l), 30 * 2 * 64).reshape(30, 2, 64)
        v = synth.normal(25, synth.stream_id("v", l), 30 * 2 * 64).reshape(30, 2, 64)
        c.append(l, 0, 0, k, v)
    blob = c.state_get(0, 5, 25)
    n = 20
    pad = lambda x: (x + 15) // 16 * 16
    ksec = pad(2 * n * 64) + pad(2 * n * 2 * 2)
    vsec = pad(2 * n * 32) + pad(2 * n * 2 * 2)
    assert len(blob) == 64 + pad(4 * n) + 2 * (ksec + vsec) == oracle.state_size(2, 2, 64, L.Q8_0, L.Q4_0, n)
    # layer 1's V codes, head-major, equal the quantiser applied to the same rows
    v1 = synth.normal(25, synth.stream_id("v", 1), 30 * 2 * 64).reshape(30, 2, 64)[5:25]
    vp, vs = oracle.q4_0_quantize(v1)
    off = 64 + pad(4 * n) + (ksec + vsec) + ksec
    got = np.frombuffer(blob, np.uint8, 2 * n * 32, off).reshape(2, n, 32).transpose(1, 0, 2)
    assert np.array_equal(got, vp)
    c.state_set(3, blob)
    assert c.state_get(3, -1, -1) == blob
    c.seq_add(3, -1, -1, 7)  # rotates K only: the V bytes stay
    after = c.state_get(3, -1, -1)
    assert after[off:off + 2 * n * 32] == blob[off:off + 2 * n * 32]


# ----------------------------------------------------------- attention ----


def _cache(n, Hk, D, seed, type_=L.Q8_0, sigma=1.0):
    k = synth.normal(seed, synth.stream_id("k"), n * Hk * D, sigma).reshape(n, Hk, D)
    v = synth.normal(seed, synth.stream_id("v"), n * Hk * D, sigma).reshape(n, Hk, D)
    if type_ == L.Q8_0:
        kc, ks = oracle.q8_0_quantize(k)
        vc, vs = oracle.q8_0_quantize(v)
        return (kc, ks), (vc, vs)
    return (oracle.f32_to_f16(k), None), (oracle.f32_to_f16(v), None)


def _deq(t, type_):
    a, s = t
    return oracle.q8_0_dequantize(a, s) if type_ == L.Q8_0 else oracle.f16_to_f64(a)


@pytest.mark.parametrize("type_", [L.Q8_0, L.F16])
def test_attn_matches_numpy_scipy(type_):
    H, Hk, D, n = 8, 2, 64, 97
    (kc, ks), (vc, vs) = _cache(n, Hk, D, 1, type_)
    q = synth.normal(1, synth.stream_id("q"), H * D).reshape(H, D)
    out = oracle.attn(q, type_, kc, ks, type_, vc, vs, 0.125)
    K, V = _deq((kc, ks), type_), _deq((vc, vs), type_)
    r = H // Hk
    for h in range(H):
        s = 0.125 * (K[:, h // r, :] @ q[h].astype(np.float64))
        p = scipy.special.softmax(s)
        np.testing.assert_allclose(out[h], p @ V[:, h // r, :], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("type_", [L.Q8_0, L.F16])
def test_attn_vs_bruteforce(type_):
    H, Hk, D, n = 4, 2, 32, 40
    (kc, ks), (vc, vs) = _cache(n, Hk, D, 2, type_)
    q = synth.normal(2, synth.stream_id("q"), H * D).reshape(H, D)
    a = oracle.attn(q, type_, kc, ks, type_, vc, vs, 0.17)
    b = oracle.attn_bruteforce(q, type_, kc, ks, type_, vc, vs, 0.17)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_attn_identical_keys_gives_mean_v():
    H, Hk, D, n = 8, 2, 64, 50
    (kc, ks), (vc, vs) = _cache(n, Hk, D, 3)
    kc[:] = kc[0]
    ks[:] = ks[0]
    q = synth.normal(3, synth.stream_id("q"), H * D).reshape(H, D)
    out = oracle.attn(q, L.Q8_0, kc, ks, L.Q8_0, vc, vs, 0.125)
    V = _deq((vc, vs), L.Q8_0)
    for h in range(H):
        np.testing.assert_allclose(out[h], V[:, h // 4].mean(0), rtol=0, atol=1e-14)


def test_attn_zero_query_gives_mean_v():
    H, Hk, D, n = 8, 2, 64, 33
    (kc, ks), (vc, vs) = _cache(n, Hk, D, 4)
    out = oracle.attn(np.zeros((H, D), np.float32), L.Q8_0, kc, ks, L.Q8_0, vc, vs, 0.125)
    V = _deq((vc, vs), L.Q8_0)
    for h in range(H):
        np.testing.assert_allclose(out[h], V[:, h // 4].mean(0), rtol=0, atol=1e-14)


def test_attn_single_row_and_empty():
    H, Hk, D = 8, 2, 64
    (kc, ks), (vc, vs) = _cache(1, Hk, D, 5)
    q = synth.normal(5, synth.stream_id("q"), H * D).reshape(H, D)
    out = oracle.attn(q, L.Q8_0, kc, ks, L.Q8_0, vc, vs, 0.125)
    V = _deq((vc, vs), L.Q8_0)
    for h in range(H):
        assert np.array_equal(out[h], V[0, h // 4])
    empty = oracle.attn(q, L.Q8_0, kc[:0], ks[:0], L.Q8_0, vc[:0], vs[:0], 0.125)
    assert (empty == 0).all()


def test_attn_gqa_contiguous_groups():
    # every row of kv head g carries V = g + 1 exactly, so out[h] = h // r + 1
    H, Hk, D, n = 12, 3, 32, 20
    (kc, ks), _ = _cache(n, Hk, D, 6)
    vc = np.full((n, Hk, D), 127, np.int8)
    vs = np.zeros((n, Hk, 1), np.uint16)
    for g in range(Hk):
        vs[:, g, 0] = oracle.f32_to_f16(np.float32([(g + 1) / 127.0]))[0]
    q = synth.normal(6, synth.stream_id("q"), H * D).reshape(H, D)
    out = oracle.attn(q, L.Q8_0, kc, ks, L.Q8_0, vc, vs, 0.2)
    for h in range(H):
        g = h // (H // Hk)
        want = 127 * oracle.f16_to_f64(vs[0, g])[0]
        np.testing.assert_allclose(out[h], want, rtol=1e-14)


def test_attn_row_permutation_invariance():
    H, Hk, D, n = 8, 2, 64, 64
    (kc, ks), (vc, vs) = _cache(n, Hk, D, 7)
    q = synth.normal(7, synth.stream_id("q"), H * D).reshape(H, D)
    perm = np.argsort(synth.uniform01(7, 99, n))
    a = oracle.attn(q, L.Q8_0, kc, ks, L.Q8_0, vc, vs, 0.125)
    b = oracle.attn(q, L.Q8_0, kc[perm], ks[perm], L.Q8_0, vc[perm], vs[perm], 0.125)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- RoPE ----


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_closed_form_unit_vector(mode):
    D = 64
    x = np.zeros(D)
    x[0] = 1.0
    y = oracle.rope_rotate(x, mode, 10000.0, 1)  # pair 0 has theta = 1
    partner = D // 2 if mode == 0 else 1
    assert abs(y[0] - math.cos(1.0)) < 1e-15 and abs(y[partner] - math.sin(1.0)) < 1e-15
    # pair i = D/4 has theta = 10000^(-1/2) = 0.01; delta 100 -> angle 1 rad
    i = D // 4
    a, b = (i, i + D // 2) if mode == 0 else (2 * i, 2 * i + 1)
    x = np.zeros(D)
    x[b] = 1.0
    y = oracle.rope_rotate(x, mode, 10000.0, 100)
    assert abs(y[a] + math.sin(1.0)) < 1e-12 and abs(y[b] - math.cos(1.0)) < 1e-12


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_group_properties(mode):
    D = 128
    x = synth.normal(8, synth.stream_id("misc", extra=8), 4 * D).astype(np.float64).reshape(4, D)
    base = 1e6
    y = oracle.rope_rotate(oracle.rope_rotate(x, mode, base, 12345), mode, base, -12345)
    np.testing.assert_allclose(y, x, atol=1e-12)
    ab = oracle.rope_rotate(oracle.rope_rotate(x, mode, base, 700), mode, base, -8192)
    np.testing.assert_allclose(ab, oracle.rope_rotate(x, mode, base, 700 - 8192), atol=1e-11)
    assert np.array_equal(oracle.rope_rotate(x, mode, base, 0), x)
    z = oracle.rope_rotate(x, mode, base, 131072)
    ia = np.arange(D // 2) if mode == 0 else 2 * np.arange(D // 2)
    ib = ia + D // 2 if mode == 0 else ia + 1
    np.testing.assert_allclose(z[:, ia] ** 2 + z[:, ib] ** 2, x[:, ia] ** 2 + x[:, ib] ** 2, rtol=1e-12)
    # same shift on q and k leaves q.k unchanged (RoPE depends on relative position)
    q, k = x[0:1], x[1:2]
    dot = (oracle.rope_rotate(q, mode, base, 5000) * oracle.rope_rotate(k, mode, base, 5000)).sum()
    assert abs(dot - (q * k).sum()) < 1e-10


def test_rope_shift_zero_is_identity_on_stored_rows():
    x = synth.normal(9, synth.stream_id("misc", extra=9), 64 * 128).reshape(64, 128)
    c, s = oracle.q8_0_quantize(x)
    c2, s2 = oracle.rope_shift_q8_0(c, s, 0, 1e6, 0)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    h = oracle.f32_to_f16(x)
    assert np.array_equal(oracle.rope_shift_f16(h, 0, 1e6, 0), h)


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_shift_q8_0_within_quantisation_error(mode):
    x = synth.normal(10, synth.stream_id("misc", extra=10), 32 * 128, 0.5).reshape(32, 128)
    c, s = oracle.q8_0_quantize(x)
    c2, s2 = oracle.rope_shift_q8_0(c, s, mode, 1e6, -8192)
    exact = oracle.rope_rotate(oracle.q8_0_dequantize(c, s), mode, 1e6, -8192)
    got = oracle.q8_0_dequantize(c2, s2)
    # requantisation error of a block: d/2 + 127 |d - fp16(d)|, d = max|x|/127
    amax = np.abs(exact.astype(np.float32)).reshape(32, 4, 32).max(2).astype(np.float64)
    d = amax / 127.0
    dh = oracle.f16_to_f64(s2)
    bound = np.repeat(d / 2 + 127 * np.abs(d - dh) + 1e-6 * amax, 32, axis=1)
    assert (np.abs(got - exact) <= bound).all()


def test_rope_shift_f16_within_half_ulp():
    x = synth.normal(11, synth.stream_id("misc", extra=11), 16 * 64).reshape(16, 64)
    h = oracle.f32_to_f16(x)
    got = oracle.f16_to_f64(oracle.rope_shift_f16(h, 0, 1e4, 77))
    exact = oracle.rope_rotate(oracle.f16_to_f64(h), 0, 1e4, 77)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 2.0**-14))) - 10)
    assert (np.abs(got - exact) <= 0.5 * ulp * (1 + 1e-9)).all()


# ---------------------------------------------------- seq ops and state ----


def _tiny_from_fixture():
    blocks = {b[0]: b for b in q8_0_blocks()}
    c = oracle.OracleCache(1, 1, 1, 32, L.Q8_0, L.Q8_0, 10000.0, 0)
    c.append(0, 0, 7, blocks["A"][1].reshape(1, 1, 32), blocks["B"][1].reshape(1, 1, 32))
    return c


def test_state_bytes_match_hand_layout():
    c = _tiny_from_fixture()
    want = hexfile("state_tiny.hex")
    assert len(want) == 176 == oracle.state_size(1, 1, 32, L.Q8_0, L.Q8_0, 1)
    assert c.state_get(0, -1, -1) == want


def _filled(type_=L.Q8_0, n=300, n_layer=2, Hk=2, D=64, seed=12):
    c = oracle.OracleCache(n_layer, 4, Hk, D, type_, type_, 10000.0, 0)
    for l in range(n_layer):
        k = synth.normal(seed, synth.stream_id("k", l), n * Hk * D).reshape(n, Hk, D)
        v = synth.normal(seed, synth.stream_id("v", l), n * Hk * D).reshape(n, Hk, D)
        c.append(l, 0, 0, k, v)
    return c


@pytest.mark.parametrize("type_", [L.Q8_0, L.F16])
def test_state_roundtrip_and_copy(type_):
    c = _filled(type_)
    blob = c.state_get(0, 40, 200)
    c.state_set(5, blob)
    assert c.state_get(5, -1, -1) == blob
    c.seq_cp(0, 6, 40, 200)
    assert c.state_get(6, -1, -1) == blob
    assert np.array_equal(c.positions(6), np.arange(40, 200))


def test_state_rejects_bad_blobs():
    c = _filled()
    blob = bytearray(c.state_get(0, 0, 10))
    for mutate in (lambda b: b.__setitem__(0, 0), lambda b: b.__setitem__(4, 2),
                   lambda b: b.__setitem__(16, 65)):
        b = bytearray(blob)
        mutate(b)
        with pytest.raises(ValueError):
            c.parse_state(bytes(b))
    with pytest.raises(ValueError):
        c.parse_state(bytes(blob[:-1]))


def test_seq_rm_ranges():
    c = _filled()
    before = c.state_get(0, -1, -1)
    c.seq_rm(0, 500, 600)  # empty range
    assert c.state_get(0, -1, -1) == before
    c.seq_rm(0, 10, 20)
    assert np.array_equal(c.positions(0), np.concatenate([np.arange(10), np.arange(20, 300)]))
    c.seq_rm(0, -1, -1)
    assert c.n_tokens(0) == 0


def test_context_shift_reading_of_tiny_config():
    # remove [0, 128) then slide [128, 512) down by 128: 384 rows at 0..383
    c = oracle.OracleCache(1, 8, 2, 64, L.Q8_0, L.Q8_0, 10000.0, 0)
    k = synth.normal(0, synth.stream_id("k"), 512 * 2 * 64).reshape(512, 2, 64)
    c.append(0, 0, 0, k, k)
    kept_v = c.seqs[0].V[0].a[128:].copy()
    c.seq_rm(0, 0, 128)
    c.seq_add(0, 128, 512, -128)
    assert np.array_equal(c.positions(0), np.arange(384))
    assert np.array_equal(c.seqs[0].V[0].a, kept_v)  # V untouched by the shift
    with pytest.raises(ValueError):
        c.seq_add(0, 0, 10, -1)  # would go negative


def test_seq_add_rotates_k_only_for_selected_rows():
    c = _filled(L.F16, n=64)
    k0 = c.seqs[0].K[1].a.copy()
    c.seq_add(0, 32, 64, 1000)
    assert np.array_equal(c.seqs[0].K[1].a[:32], k0[:32])
    assert np.array_equal(c.seqs[0].K[1].a[32:], oracle.rope_shift_f16(k0[32:], 0, 1e4, 1000))
    assert np.array_equal(c.positions(0), np.concatenate([np.arange(32), np.arange(1032, 1064)]))


# ---------------------------------------------------------------- KeyDiff --
# Pins of the KeyDiff score ("F5 - Advanced KV Cache Techniques", M1:
# distinctiveness = mean over KV heads of 1 - cos(key, the head's mean key))
# and of the minimum-sum window search.

def _f16_keys(x):
    return oracle.f32_to_f16(np.asarray(x, np.float32))


def test_keydiff_closed_forms():
    # two orthogonal unit keys: mean (1/2, 1/2), cos = 1/sqrt(2) for both
    sc = oracle.keydiff_scores(oracle.F16, _f16_keys([[[1, 0]], [[0, 1]]]), None)
    assert np.allclose(sc, 1 - 1 / math.sqrt(2), atol=1e-15, rtol=0)
    # identical keys: every cosine is 1, every score 0
    sc = oracle.keydiff_scores(oracle.F16, _f16_keys([[[3, -1, 2]]] * 5), None)
    assert np.allclose(sc, 0, atol=1e-15)
    # antipodal keys have a zero mean: the degenerate cosine is read as 0
    sc = oracle.keydiff_scores(oracle.F16, _f16_keys([[[2, 0]], [[-2, 0]]]), None)
    assert np.array_equal(sc, [1.0, 1.0])
    # the score averages over heads: head 0 identical keys (0), head 1 orthogonal
    sc = oracle.keydiff_scores(oracle.F16, _f16_keys([[[1, 1], [1, 0]], [[1, 1], [0, 1]]]), None)
    assert np.allclose(sc, (1 - 1 / math.sqrt(2)) / 2, atol=1e-15)
    # three unit axes in 3-d: mean (1,1,1)/3, cos = 1/sqrt(3)
    sc = oracle.keydiff_scores(oracle.F16, _f16_keys([[[1, 0, 0]], [[0, 1, 0]], [[0, 0, 1]]]), None)
    assert np.allclose(sc, 1 - 1 / math.sqrt(3), atol=1e-15)


def test_keydiff_invariances():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (40, 3, 64)).astype(np.float32)
    base = oracle.keydiff_scores(oracle.F16, _f16_keys(x), None)
    # a positive power-of-two scale of every key (exact in fp16) leaves cosines alone
    assert np.allclose(oracle.keydiff_scores(oracle.F16, _f16_keys(x * 4), None), base, atol=1e-12)
    # permuting the rows permutes the scores (the mean is order-free)
    perm = rng.permutation(40)
    assert np.allclose(oracle.keydiff_scores(oracle.F16, _f16_keys(x[perm]), None), base[perm], atol=1e-12)
    # permuting the dimensions of every key together changes nothing
    dp = rng.permutation(64)
    assert np.allclose(oracle.keydiff_scores(oracle.F16, _f16_keys(x[:, :, dp]), None), base, atol=1e-12)
    # scores lie in [0, 2]
    assert base.min() >= 0 and base.max() <= 2
    # a row equal to its head's mean direction in every head scores 0
    y = np.concatenate([x, x.mean(axis=0, keepdims=True)], axis=0)
    sy = oracle.keydiff_scores(oracle.F16, _f16_keys(y), None)
    assert abs(sy[-1]) < 1e-3  # fp16 rounding of the appended mean row


def test_keydiff_q8_0_equals_f16_on_exact_values():
    # integer keys with max |x| = 127 per block quantise to scale 1.0 and
    # codes equal to the values: both storage types describe the same keys
    rng = np.random.default_rng(6)
    x = rng.integers(-126, 127, (30, 2, 64)).astype(np.float32)
    x[:, :, ::32] = 127.0
    codes, scales = oracle.q8_0_quantize(x)
    assert np.all(oracle.f16_to_f64(scales) == 1.0) and np.array_equal(codes.astype(np.float32), x)
    a = oracle.keydiff_scores(oracle.Q8_0, codes, scales)
    b = oracle.keydiff_scores(oracle.F16, _f16_keys(x), None)
    assert np.array_equal(a, b)


def test_min_window_against_brute_force():
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        sc = rng.random(n)
        lo, hi, w = int(rng.integers(0, n)), int(rng.integers(0, n + 1)), int(rng.integers(1, 8))
        got = oracle.min_window(sc, lo, hi, w)
        starts = [s for s in range(lo, hi - w + 1)]
        if not starts:
            assert got == -1
            continue
        sums = [sum(sc[s:s + w]) for s in starts]
        assert got == starts[int(np.argmin(sums))]
    # ties go to the first window
    assert oracle.min_window(np.ones(10), 2, 9, 3) == 2
    # the window never leaves [lo, hi)
    assert oracle.min_window(np.array([5, 5, 0, 0, 5, 5.0]), 0, 3, 2) == 1


def test_evict_window_removes_the_least_distinctive_rows():
    # 24 rows; rows 10..13 repeat the mean direction of every head (score ~0):
    # the width-4 window inside [4, 20) must be exactly those rows
    rng = np.random.default_rng(8)
    H, Hk, D, n = 4, 2, 64, 24
    k = rng.normal(0, 1, (n, Hk, D)).astype(np.float32)
    k[10:14] = k.mean(axis=0)
    v = rng.normal(0, 1, (n, Hk, D)).astype(np.float32)
    c = oracle.OracleCache(1, H, Hk, D, oracle.F16, oracle.F16, 1e4, 0)
    c.append(0, 0, 0, k, v)
    sc = c.key_scores(0, 0)
    assert sc[10:14].max() < sc[np.r_[0:10, 14:24]].min()
    v_before = c.seqs[0].V[0].a.copy()
    p0 = c.evict_window(0, 0, n_keep=4, n_discard=4, n_recent=4)
    assert p0 == 10
    assert np.array_equal(c.positions(0), np.arange(n - 4))  # slid down over the gap
    keep = np.r_[0:10, 14:24]
    assert np.array_equal(c.seqs[0].V[0].a, v_before[keep])   # V untouched, window gone
    # no window fits: nothing changes
    assert c.evict_window(0, 0, n_keep=10, n_discard=8, n_recent=4) == -1
    assert c.n_tokens(0) == n - 4


# Pins of the host-RAM cold store policy (Plan: lossless long context, #3
# Host-RAM KV cold store + retrieval, llama - KV-byte offload): bounded in
# tokens, blocks dropped most evictable class first and least recently
# stored first within a class, never a less evictable block for a more
# evictable one; admit in append mode; evict -> admit is lossless.

def _cold_cache(n, n_seq=2, seed=9):
    rng = np.random.default_rng(seed)
    c = oracle.OracleCache(2, 4, 2, 64, oracle.Q8_0, oracle.Q8_0, 1e4, 0)
    for l in range(2):
        c.append(l, 0, 0, rng.normal(0, 1, (n, 2, 64)).astype(np.float32),
                 rng.normal(0, 1, (n, 2, 64)).astype(np.float32))
    return c


def test_cold_store_victim_order_closed_case():
    c = _cold_cache(100)
    s = oracle.ColdStore(10)
    # evicting from the tail keeps the arithmetic simple: no slide
    assert s.evict(c, 0, 1, 96, 100, key=1, cls=0) == (1, 4)    # A: 4 tokens, class 0
    assert s.evict(c, 0, 1, 93, 96, key=2, cls=1) == (1, 3)     # B: 3, class 1
    assert s.evict(c, 0, 1, 90, 93, key=3, cls=1) == (1, 3)     # C: 3, class 1 -> store full (10)
    assert s.evict(c, 0, 1, 87, 90, key=4, cls=1) == (1, 3)     # D: drops B (class 1, oldest)
    assert [b["key"] for b in s.blocks] == [1, 3, 4] and s.stats["dropped"] == 1
    assert s.evict(c, 0, 1, 82, 87, key=5, cls=0) == (1, 5)     # E (5, class 0): drops C then D, keeps A
    assert [b["key"] for b in s.blocks] == [1, 5] and s.tokens == 9 and s.stats["dropped"] == 3
    assert s.evict(c, 0, 1, 80, 82, key=6, cls=2) == (0, 2)     # class 2 may drop nothing here: not kept
    assert s.evict(c, 0, 1, 69, 80, key=7, cls=9) == (0, 11)    # larger than the budget: not kept
    assert s.stats["rejected"] == 2 and s.tokens == 9
    assert c.n_tokens(0) == 69 and c.n_tokens(1) == 0           # evicted rows left the cache either way
    assert s.admit(c, 0, 1, key=3) == (0, 0) and s.stats["misses"] == 1


def test_cold_store_tail_round_trip_is_lossless():
    c = _cold_cache(64)
    before = c.state_get(0, -1, -1)
    s = oracle.ColdStore(1000)
    assert s.evict(c, 0, 1, 40, 64, key=7, cls=0) == (1, 24)
    assert c.n_tokens(0) == 40
    assert s.admit(c, 0, 1, key=7) == (1, 24)                   # back at position 40: no shift
    assert c.state_get(0, -1, -1) == before and s.blocks == [] and c.n_tokens(1) == 0


def test_cold_store_admit_after_slide_equals_manual_ops():
    # evict the head, which slides the rest down; admit returns it at the tail, shifted
    a, b = _cold_cache(80), _cold_cache(80)
    s = oracle.ColdStore(100)
    assert s.evict(a, 0, 1, 0, 16, key=3, cls=0) == (1, 16)
    assert np.array_equal(a.positions(0), np.arange(64))
    assert s.admit(a, 0, 1, key=3) == (1, 16)
    assert np.array_equal(a.positions(0), np.arange(80))
    # the same steps by hand
    b.seq_cp(0, 1, 0, 16)
    blob = b.state_get(1, -1, -1)
    b.seq_rm(1, -1, -1)
    b.seq_rm(0, 0, 16)
    b.seq_add(0, 16, -1, -16)
    b.state_set(1, blob)
    b.seq_add(1, -1, -1, 64)
    b.seq_cp(1, 0, -1, -1)
    b.seq_rm(1, -1, -1)
    assert a.state_get(0, -1, -1) == b.state_get(0, -1, -1)


def test_cold_store_invariants_random():
    rng = np.random.default_rng(11)
    for trial in range(20):
        c = _cold_cache(400, seed=trial)
        s = oracle.ColdStore(int(rng.integers(20, 120)))
        key = 0
        for _ in range(12):
            n = c.n_tokens(0)
            if n < 2:
                break
            w = int(rng.integers(1, min(40, n) + 1))
            p0 = int(rng.integers(0, n - w + 1))
            cls = int(rng.integers(0, 3))
            before = [(b["key"], b["cls"], b["stamp"], b["n"]) for b in s.blocks]
            key += 1
            stored, got = s.evict(c, 0, 1, p0, p0 + w, key=key, cls=cls)
            assert got == w and s.tokens <= s.budget
            after = {b["key"] for b in s.blocks}
            gone = [x for x in before if x[0] not in after]
            # every dropped block was at least as evictable as the new one, and a kept block of a
            # class above a dropped one's, or older in the same class, was not passed over
            assert all(g[1] >= cls for g in gone)
            for g in gone:
                for x in before:
                    if x[0] in after and x[1] >= cls:
                        assert (x[1], -x[2]) <= (g[1], -g[2])
            assert stored == (key in after)
            if not stored:
                assert gone == []


def test_cold_store_restore_model_fit_and_decision():
    # the fitted line against numpy's least-squares polynomial fit
    cs = oracle.ColdStore(100)
    rows = [512, 2048, 8192, 1024, 4096]
    us = [900.0 + 0.85 * n + (13.0 if i % 2 else -9.0) for i, n in enumerate(rows)]
    fixed, per = cs.fit_restore_model(list(zip(rows, us)))
    slope, icpt = np.polyfit(np.array(rows, float), np.array(us, float), 1)
    assert abs(per - slope) <= 1e-12 * abs(slope) + 1e-12 and abs(fixed - icpt) <= 1e-9 * abs(icpt) + 1e-9
    # one block size only: a line through 0; no samples: no model
    assert cs.fit_restore_model([(2048, 1000.0), (2048, 1200.0)]) == (0.0, 2200.0 / 4096.0)
    assert cs.fit_restore_model([]) is None
    # the decision: restore while fixed + per * n < recompute_fixed + recompute_per * n
    cs.blocks.append({"key": 7, "cls": 0, "n": 1000, "first": 0, "stamp": 0, "blob": b""})
    assert cs.plan_admit(7, 0.0, 1.0) == (1, -1.0, 1000)          # no model: the stored bytes first
    assert cs.plan_admit(8, 0.0, 1.0) == (0, 0.0, 0)              # absent: recompute
    m = (1500.0, 0.9)                                             # restore 2400 us for 1000 rows
    assert cs.plan_admit(7, 0.0, 2.5, model=m) == (1, 2400.0, 1000)   # recompute 2500 us
    assert cs.plan_admit(7, 0.0, 2.3, model=m)[0] == 0                # recompute 2300 us
    assert cs.plan_admit(7, 2400.0 - 2300.0, 2.3, model=m)[0] == 0    # equal cost: recompute
    # the crossover: restore wins above n* = fixed / (recompute_per - per)
    for n, want in ((1000, 1), (900, 0)):
        cs.blocks[0]["n"] = n
        assert cs.plan_admit(7, 0.0, 2.5, model=m)[0] == want
