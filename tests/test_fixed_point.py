"""The single-launch decode kernel adds its partial sums in 64-bit fixed point
(2^-32 units) and forms round(v * 2^32) from 32-bit operations only: for
a = |v|, h = floor(a) and f = a - h are exact, h * 2^32 is even, so
round(a * 2^32) = h * 2^32 + round(f * 2^32), and round-to-nearest-even is
odd-symmetric.  This checks that identity in fp32 arithmetic (numpy, IEEE
round-to-nearest) against the exact value computed in fp64, on random floats
of every magnitude below 2^31 and on the tie cases."""
import numpy as np


def to_fix_f32(v: np.ndarray) -> np.ndarray:
    v = v.astype(np.float32)
    a = np.abs(v)
    h = np.floor(a)                                   # exact
    f = (a - h).astype(np.float32)                    # exact for a >= 0
    lo = np.rint((f * np.float32(4294967296.0)).astype(np.float32)).astype(np.uint64)
    assert np.all(lo < 2 ** 32)
    m = (h.astype(np.uint64) << np.uint64(32)) | lo
    return np.where(v < 0, -m.astype(np.int64), m.astype(np.int64))


def exact(v: np.ndarray) -> np.ndarray:
    return np.rint(v.astype(np.float64) * 4294967296.0).astype(np.int64)  # v * 2^32 is exact in fp64


def test_fixed_point_identity_random_bits():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 2.0 ** 31)]
    assert np.array_equal(to_fix_f32(v), exact(v))


def test_fixed_point_identity_ties_and_edges():
    u = np.float32(2.0 ** -32)
    v = np.array([0.5 * u, 1.5 * u, 2.5 * u, -2.5 * u, 3.5 * u, -0.5 * u, 1e-30, -1e-30, 0.0, -0.0,
                  0.3, -0.3, 1.0, -1.0, 12345.678, -12345.678, 2147483520.0, -2147483520.0,
                  np.nextafter(np.float32(1.0), np.float32(0.0))], dtype=np.float32)
    assert np.array_equal(to_fix_f32(v), exact(v))
