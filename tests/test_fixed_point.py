"""The single-launch decode kernel adds its partial sums in 64-bit fixed point
(2^-32 units) and forms round(v * 2^32) without a float-to-integer
conversion: A = |v| 2^32 is exact; below 2^23 the float sum A + 2^23 has a
unit ulp, so its bits minus those of 2^23 are round-to-nearest-even(A); from
2^23 up A is an integer, its significand (hidden bit included) shifted left by
(biased exponent - 150); the sign is applied last (round-to-nearest-even is
odd-symmetric).  This replays those steps in fp32 / uint32 arithmetic (numpy,
IEEE round-to-nearest) and checks them against the exact value computed in
fp64, on random floats of every magnitude below 2^23 and on the tie cases."""
import numpy as np

TWO23 = np.float32(2.0 ** 23)


def to_fix_f32(v: np.ndarray) -> np.ndarray:
    v = v.astype(np.float32)
    A = (np.abs(v) * np.float32(4294967296.0)).astype(np.float32)
    b = A.view(np.uint32).astype(np.uint64)
    small = A < TWO23
    rs = ((A + TWO23).astype(np.float32).view(np.uint32).astype(np.uint64) - 0x4B000000)
    mant = (b & 0x7FFFFF) | 0x800000
    sh = np.where(small, 0, b >> np.uint64(23)).astype(np.int64) - 150
    sh = np.where(small, 0, sh).astype(np.uint64)
    big = mant << sh                                  # < 2^55: no wrap in 64 bits
    m = np.where(small, rs, big)
    assert np.all(np.where(small, rs <= 2 ** 23, (sh <= 31)))
    return np.where(v < 0, -m.astype(np.int64), m.astype(np.int64))


def exact(v: np.ndarray) -> np.ndarray:
    return np.rint(v.astype(np.float64) * 4294967296.0).astype(np.int64)  # v * 2^32 is exact in fp64


def test_fixed_point_identity_random_bits():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 2.0 ** 23)]
    assert v.size > 500_000
    assert np.array_equal(to_fix_f32(v), exact(v))


def test_fixed_point_identity_ties_and_edges():
    u = np.float32(2.0 ** -32)
    v = np.array([0.5 * u, 1.5 * u, 2.5 * u, -2.5 * u, 3.5 * u, -0.5 * u, 1e-30, -1e-30, 0.0, -0.0,
                  1e-45, -1e-45,                       # denormals
                  0.3, -0.3, 1.0, -1.0, 12345.678, -12345.678, 8388607.5, -8388607.5,
                  np.nextafter(np.float32(2.0 ** -9), np.float32(0.0)), 2.0 ** -9, -2.0 ** -9,
                  (2.0 ** 23 - 0.5) * 2.0 ** -32, (2.0 ** 23 - 1.5) * 2.0 ** -32,
                  np.nextafter(np.float32(1.0), np.float32(0.0))], dtype=np.float32)
    assert np.array_equal(to_fix_f32(v), exact(v))


def test_fixed_point_every_small_magnitude_band():
    """Every binade of |v| 2^32 below 2^23 (the rounding path) and from 2^23 to
    2^55 (the shift path), with the tie values of each binade."""
    vals = []
    for e in range(-40, 23):
        base = np.float32(2.0 ** e)
        ulp = np.float32(2.0 ** (e - 23))
        for k in range(0, 64):
            vals.append(base + np.float32(k) * ulp)
        vals.append(np.nextafter(base, np.float32(0.0)))
        if e - 32 < 0:  # A's binade below 2^23: ties of A at half-integers
            half = np.float32(2.0 ** -33)
            for k in range(1, 9, 2):
                vals.append(np.float32(k) * half)
    v = np.array(vals, dtype=np.float32)
    v = np.concatenate([v, -v])
    assert np.array_equal(to_fix_f32(v), exact(v))
