"""The flush kernel takes each 2-bit code without a division: with
y = (x - z) / s and f = fl(y) (IEEE fp32, round to nearest even), the code
clamp(rint(f), 0, 3) (zijie-tian.site sec. 2.1: asymmetric 2-bit
quantization with scale s and zero z) equals

    [f > 0.5] + [f >= 1.5] + [f > 2.5]

and, because fp32 rounding is monotone with ties to even, each bracket is a
comparison of a = fl(x - z) with one fp32 threshold of s:

    f > 0.5  <=>  a > RD(s (1/2 + 2^-25))
    f >= 1.5 <=>  a >= RU(s (3/2 - 2^-24))
    f > 2.5  <=>  a > RD(s (5/2 + 2^-23))

(RD/RU: fp32 rounding down/up of the exact product; 0.5, 1.5 and 2.5 have
even significands, so a tie at each midpoint rounds onto them). This test
pins the rule on the CPU against numpy's IEEE fp32 division and rint, on
random pairs and on every a within a few ulps of each threshold, for scales
that are fp16 values (as the library's scales are), subnormals included.
"""
import numpy as np

F32 = np.float32


def _rd(x: float) -> np.float32:
    f = F32(x)
    return np.nextafter(f, F32(-np.inf)) if float(f) > x else f


def _ru(x: float) -> np.float32:
    f = F32(x)
    return np.nextafter(f, F32(np.inf)) if float(f) < x else f


def _thresholds(s: np.float32):
    s64 = float(s)   # s has 11 significant bits: each product is exact in fp64
    return (_rd(s64 * (0.5 + 2.0 ** -25)), _ru(s64 * (1.5 - 2.0 ** -24)), _rd(s64 * (2.5 + 2.0 ** -23)))


def _code_div(a: np.ndarray, s: np.float32) -> np.ndarray:
    with np.errstate(over="ignore"):
        return np.clip(np.rint(a / s), 0, 3).astype(np.int64)


def _code_thr(a: np.ndarray, s: np.float32) -> np.ndarray:
    t1, t2, t3 = _thresholds(s)
    return (a > t1).astype(np.int64) + (a >= t2) + (a > t3)


def _fp16_scales(rng, n):
    bits = rng.integers(1, 0x7BFF, size=n, dtype=np.int64).astype(np.uint16)   # positive finite fp16
    extra = np.array([1, 2, 3, 0x3FF, 0x400, 0x3C00, 0x3555, 0x7BFF], np.uint16)  # subnormals, 1, 1/3, max
    return np.concatenate([bits, extra]).view(np.float16).astype(F32)


def test_random_pairs():
    rng = np.random.default_rng(1)
    for s in _fp16_scales(rng, 300):
        a = (rng.random(4000) * 3.6 * float(s)).astype(F32)
        assert np.array_equal(_code_div(a, s), _code_thr(a, s)), s


def test_every_value_near_each_threshold():
    rng = np.random.default_rng(2)
    for s in _fp16_scales(rng, 400):
        for c in (0.5, 1.5, 2.5):
            m = F32(float(s) * c)
            a = [m]
            lo = hi = m
            for _ in range(6):
                lo = np.nextafter(lo, F32(-np.inf))
                hi = np.nextafter(hi, F32(np.inf))
                a += [lo, hi]
            a = np.array(a, F32)
            a = a[a >= 0]
            assert np.array_equal(_code_div(a, s), _code_thr(a, s)), (s, c)


def test_a_dropped_tie_rule_is_caught():
    """Sanity of the pin itself: with ties rounding away from the even
    neighbour (> instead of >= at 1.5), some a near 1.5 s disagrees."""
    rng = np.random.default_rng(3)
    bad = 0
    for s in _fp16_scales(rng, 200):
        m = F32(float(s) * 1.5)
        a = np.array([np.nextafter(m, F32(-np.inf)), m, np.nextafter(m, F32(np.inf))], F32)
        t1, t2, t3 = _thresholds(s)
        wrong = (a > t1).astype(np.int64) + (a > t2) + (a > t3)
        bad += int((wrong != _code_div(a, s)).sum())
    assert bad > 0
