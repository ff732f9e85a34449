"""The E4M3 quantiser decides, value by value, whether the product x * (1/s)
already has the code of the IEEE quotient x / s, or whether it must divide.
The CUDA source states that test twice: as unsigned ranges on the fp32 bits,
and as float compares.  Both must mean the same thing.

The property proved in the source: y is used when its low 20 fraction bits
are more than 4 from 0x80000 (the rounding midpoints of a normal E4M3
binade) and 2^-6 <= |y| <= 512.  These tests restate both spellings in
numpy.  They compare them on every sign and exponent, crossed with the
fractions around the midpoint, the range limits, and random fractions.  The
GPU tests check the kernels' codes bit for bit against the oracle.
"""
import numpy as np


def needs_division_bits(b: np.ndarray) -> np.ndarray:
    """Unsigned-range form (e4m3_needs_division)."""
    b = b.astype(np.uint32)
    return ((b & np.uint32(0xFFFFF)) - np.uint32(0x7FFFC) <= np.uint32(8)) | \
        ((b & np.uint32(0x7FFFFFFF)) - np.uint32(0x3C800000) > np.uint32(0x07800000))


def product_usable_compares(b: np.ndarray) -> np.ndarray:
    """Float-compare form (e4m3_product_usable)."""
    y = b.astype(np.uint32).view(np.float32)
    frac = b.astype(np.uint32) & np.uint32(0xFFFFF)
    dist = np.where(frac > 0x80000, frac - np.uint32(0x80000), np.uint32(0x80000) - frac)
    with np.errstate(invalid="ignore"):
        ay = np.abs(y)
        return (dist > 4) & (ay >= np.float32(2.0 ** -6)) & (ay <= np.float32(512.0))


def bit_patterns(seed: int = 3) -> np.ndarray:
    hi = np.arange(512, dtype=np.uint32) << np.uint32(23)          # every sign and exponent
    edges = np.concatenate([np.arange(0x7FFF0, 0x80011), np.arange(0, 9), np.arange(0x7FFFF8, 0x800000),
                            np.arange(0xFFFF0, 0x100010)]).astype(np.uint32) & np.uint32(0x7FFFFF)
    rnd = np.random.default_rng(seed).integers(0, 1 << 23, size=4096, dtype=np.uint32)
    frac = np.unique(np.concatenate([edges, rnd]))
    return (hi[:, None] | frac[None, :]).ravel()


def test_both_spellings_agree():
    b = bit_patterns()
    assert b.size > 2_000_000
    assert np.array_equal(needs_division_bits(b), ~product_usable_compares(b))


def test_the_test_means_what_the_proof_needs():
    f = np.float32
    def usable(v):
        return bool(product_usable_compares(np.array([v], np.float32).view(np.uint32))[0])
    assert usable(f(1.0)) and usable(f(448.0)) and usable(f(512.0)) and usable(f(2.0 ** -6))
    assert not usable(f(0.0)) and not usable(f(-0.0)) and not usable(f(np.nan))
    assert not usable(np.nextafter(f(2.0 ** -6), f(0.0)))              # below E4M3's normal range
    assert not usable(np.nextafter(f(512.0), f(1024.0)))               # 1/s overflowed
    mid = np.uint32(0x3F880000)                                         # 1.0625: a midpoint of [1, 2)
    for d in range(-4, 5):
        assert not usable((mid + np.uint32(d) if d >= 0 else mid - np.uint32(-d)).view(np.float32))
    assert usable((mid + np.uint32(5)).view(np.float32)) and usable((mid - np.uint32(5)).view(np.float32))
