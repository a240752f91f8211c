"""Exact-arithmetic identities the CUDA kernels rely on, checked exhaustively
or densely on the CPU (numpy float32 arithmetic rounds to nearest even, as the
GPU's does).  No GPU and no code of the library: each identity is restated
here from its mathematics.

- The RoPE shift re-quantises with round half away from zero (the q8_0
  quantiser: code = round(x / d)), computed as the truncation of
  q + copysign(0.49999997, q) in fp32.
- It dequantises a stored q8_0 code as one fused multiply-add: the code byte u
  placed at bits 8..15 of 2^23 is the float 2^23 + 256 u, and
  (2^23 + 256 u) * (s / 256) - (2^23 + 2^15) * (s / 256) = s (u - 128) with one
  rounding, exact for every fp16 scale s.
- The attention turns stored int8 codes and q4_0 nibbles into exact fp16
  operands through the mantissa of 1024.
"""
import numpy as np

PRED_HALF = np.frombuffer(np.uint32(0x3EFFFFFF).tobytes(), np.float32)[0]  # largest float below 1/2


def _round_half_away(q):
    """Round half away from zero, in float64 (exact for float32 inputs)."""
    qd = q.astype(np.float64)
    return np.sign(qd) * np.floor(np.abs(qd) + 0.5)


def _biased_trunc(q):
    bias = np.where(np.signbit(q), -PRED_HALF, PRED_HALF).astype(np.float32)
    return np.trunc((q + bias).astype(np.float32)).astype(np.float64)


def test_pred_half_is_the_float_below_one_half():
    assert PRED_HALF < np.float32(0.5) and np.nextafter(PRED_HALF, np.float32(1)) == np.float32(0.5)


def test_biased_truncation_rounds_half_away_from_zero():
    rng = np.random.default_rng(3)
    parts = [rng.uniform(-128, 128, 2_000_000).astype(np.float32)]
    # every half-integer and integer in (-130, 130) with 64 neighbours on each side
    for k in range(-130, 131):
        for c in (k + 0.5, float(k)):
            bits = np.array([c], np.float32).view(np.int32)[0]
            nb = np.arange(bits - 64, bits + 65, dtype=np.int64).astype(np.int32).view(np.float32)
            parts.append(nb)
            parts.append(-nb)
    # a dense sweep of [0, 2) (subnormals included), and both signs
    small = np.arange(0, 0x40000000, 1021, dtype=np.uint32).view(np.float32)
    parts += [small, -small]
    q = np.concatenate(parts)
    q = q[np.isfinite(q) & (np.abs(q) < 2**22)]
    got, want = _biased_trunc(q), _round_half_away(q)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, q[bad[:5]]


def test_plain_half_bias_would_round_the_predecessor_of_one_half_up():
    # the reason for the predecessor: 0.49999997 + 0.5 rounds to 1.0 in fp32
    q = np.array([PRED_HALF, -PRED_HALF], np.float32)
    plain = np.trunc((q + np.where(np.signbit(q), -0.5, 0.5).astype(np.float32)).astype(np.float32))
    assert list(plain) == [1.0, -1.0] and list(_biased_trunc(q)) == [0.0, 0.0]


def test_dequantisation_by_one_fma_is_exact_for_every_scale_and_code():
    s = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)  # finite, >= 0
    u = np.arange(256, dtype=np.float64)
    s8 = (s * np.float32(1 / 256)).astype(np.float32)
    off = (np.float32(-8421376.0) * s8).astype(np.float32)  # -(2^23 + 2^15) s / 256
    assert np.array_equal(off.astype(np.float64), -8421376.0 * s8.astype(np.float64))  # no rounding
    f = 2.0**23 + 256.0 * u  # the byte at bits 8..15 of 2^23
    fma = (f[None, :] * s8.astype(np.float64)[:, None] + off.astype(np.float64)[:, None]).astype(np.float32)
    exact = s.astype(np.float64)[:, None] * (u[None, :] - 128.0)
    assert np.array_equal(fma.astype(np.float64), exact)


def _half(bits):
    return np.array(bits, np.uint16).view(np.float16)


def test_int8_codes_to_fp16_by_the_mantissa_of_1024():
    # the attention kernel's QK and PV operands: an offset-binary byte u = c + 128 placed in the
    # low byte of 0x64uu is the half 1024 + u; subtracting half(1152) leaves c exactly
    u = np.arange(256)
    h = _half(0x6400 | u)
    assert np.array_equal(h.astype(np.float64), 1024.0 + u)
    c = (h - np.float16(1152)).astype(np.float64)  # float16 arithmetic, one rounding
    assert np.array_equal(c, u - 128.0)


def test_q4_0_nibbles_to_fp16_exactly():
    # low nibble n in the mantissa of 1024: (1024 + n) - 1032 = n - 8; high nibble as 16 n:
    # (1024 + 16 n) * (1/16) - 72 = n - 8, each with one rounding of an exact value
    n = np.arange(16)
    lo = (_half(0x6400 | n) - np.float16(1032)).astype(np.float64)
    assert np.array_equal(lo, n - 8.0)
    hi_in = _half(0x6400 | (n << 4))
    hi = (hi_in.astype(np.float32) * np.float32(1 / 16) + np.float32(-72)).astype(np.float16).astype(np.float64)
    assert np.array_equal(hi, n - 8.0)
    assert np.float16(1 / 16) == _half(0x2C00) and np.float16(-72) == _half(0xD480)
    assert np.float16(1032) == _half(0x6408) and np.float16(1152) == _half(0x6480)
