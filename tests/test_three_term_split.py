"""The three-term bf16 split that carries -L/scale and -D into the d = 96/128
backward's S^T and dP^T products (host only, no GPU).

A value v (fp32) is written as hi = bf16(v), mid = bf16(v - hi) and
lo = bf16(v - hi - mid), each rounded to nearest even; the extra k-step
multiplies each by 1.0 and the tensor core adds them into the fp32
accumulator.  The sum must reproduce v exactly, so that
S^T - L/scale and dP^T - D come out of the products as the threads would
have formed them.  bf16 rounding is emulated on the fp32 bit patterns.
"""

import numpy as np


def _bf16(x):
    """Round fp32 values to bf16 (nearest, ties to even), returned as fp32."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    out = rounded.astype(np.uint32).view(np.float32)
    return np.where(np.isfinite(x), out, x)


def _split(v):
    v = np.asarray(v, dtype=np.float32)
    hi = _bf16(v)
    r1 = (v - hi).astype(np.float32)
    mid = _bf16(r1)
    lo = _bf16((r1 - mid).astype(np.float32))
    return hi, mid, lo


def test_bf16_rounding_emulation_matches_known_values():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even gives 1.
    assert _bf16(np.float32(1 + 2.0 ** -8)) == 1.0
    assert _bf16(np.float32(1 + 3 * 2.0 ** -8)) == np.float32(1 + 2 * 2.0 ** -7)
    assert _bf16(np.float32(3.0)) == 3.0
    assert np.isneginf(_bf16(np.float32(-np.inf)))


def test_three_terms_reproduce_the_fp32_value():
    rng = np.random.default_rng(0)
    # -L/scale: L up to ~60 in natural-log units, scale down to 1/16; -D: O(1)
    # of either sign; plus values spread over many binades.
    v = np.concatenate([
        -rng.uniform(0, 60, 20000) / rng.choice([1 / 8, 1 / 11.3137, 1 / 16], 20000),
        rng.normal(0, 3, 20000),
        rng.choice([-1, 1], 20000) * 2.0 ** rng.uniform(-30, 20, 20000),
    ]).astype(np.float32)
    hi, mid, lo = _split(v)
    # An fp32 significand has 24 bits and each bf16 term takes 8 of what is
    # left, so the three terms carry v exactly (summed in fp64 here); the
    # only rounding is the accumulator's own fp32 addition in the product.
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(total, v.astype(np.float64))
    # Every term is a bf16 value (its low 16 bits are zero).
    for t in (hi, mid, lo):
        assert np.all((t.view(np.uint32) & 0xFFFF) == 0)


def test_dead_rows_carry_minus_infinity_alone():
    """Rows past N carry -inf in the first term and zeros after it, so that
    the product gives -inf (P = 0) and no inf - inf arises."""
    v = np.float32(-np.inf)
    hi = _bf16(v)
    assert np.isneginf(hi)
    # the kernel writes mid = lo = 0 for non-finite values
    assert np.isneginf(np.float64(hi) + 0.0 + 0.0)
