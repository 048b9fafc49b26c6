"""The ranking pass's bucket map, restated in IEEE float32 arithmetic on the
CPU: it must never put a larger score into a lower bucket, and must stay
inside the bucket range, for every distribution (ties, both signs,
subnormals, values near the float32 limits).  The ranking pass is correct for
any monotone in-range map (members of one bucket are compared exactly), so
these are the two properties its correctness rests on.  The GPU tests
(`test_gpu_sort_by_score.py`) check the kernel itself end to end.

Map (per row): c = (max - min) / 64 (rounded), coordinate
f(v) = sign(v) * (bits(c + |v|) - bits(c)) in two's complement, x = f(v) - f(min)
as uint32, bucket = x when range < NB, else floor(x * mul / 2^32) with
mul = floor(float(NB * 2^32 * (1 - 2^-20)) / float_ru(range + 1)).
"""
import numpy as np
import pytest

# bucket counts of the kernel's row sizes (one bucket per rankable unit slot:
# 256, 2048 and 4096 units), and twice the largest
NBS = (256, 2048, 4096, 8192)


def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)


def _coord(v, c):
    v = np.asarray(v, np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        h = (_bits(np.float32(c) + np.abs(v)) - _bits(c)) & 0xFFFFFFFF
    return np.where(v >= 0, h, (0 - h) & 0xFFFFFFFF).astype(np.uint64)


def _round_up(x):
    """x rounded up to float32 (the kernel's _ru conversions and additions)."""
    f = np.float32(x)
    return np.nextafter(f, np.float32(np.inf)) if float(f) < x else f


def _buckets(v, NB):
    v = np.asarray(v, np.float32)
    vmin, vmax = v.min(), v.max()
    with np.errstate(over="ignore", invalid="ignore"):
        c = np.float32(np.float32(vmax - vmin) * np.float32(1.0 / 64.0))
    lo = int(_coord(np.array([vmin], np.float32), c)[0])
    rng = (int(_coord(np.array([vmax], np.float32), c)[0]) - lo) & 0xFFFFFFFF
    x = (_coord(v, c) + np.uint64((1 << 32) - lo)) & np.uint64(0xFFFFFFFF)
    if rng < NB:
        return x.astype(np.int64)
    num = np.float32(NB * 4294967296.0 * (1.0 - 2.0 ** -20))   # exact: NB * (2^32 - 2^12)
    den = _round_up(float(_round_up(rng)) + 1.0)
    mul = int(np.floor(np.float64(np.float32(np.float64(num) / np.float64(den)))))
    assert 0 < mul < 2 ** 32
    return ((x * np.uint64(mul)) >> np.uint64(32)).astype(np.int64)


def _dists(rng, n):
    yield rng.standard_normal(n)
    yield rng.lognormal(0, 3, n) * rng.choice([-1, 1], n)
    yield rng.integers(-5, 5, n).astype(np.float64)              # heavy ties, both signs
    yield rng.standard_normal(n) * 1e-40                        # subnormals
    yield rng.standard_normal(n) * 3e38                         # near the float32 limit
    yield np.concatenate([rng.standard_normal(max(n - 3, 1)), [0.0, -0.0, 1e30]])
    yield np.where(rng.random(n) < 0.01, 2.0 ** 20, 1.0) * np.abs(rng.standard_normal(n))


@pytest.mark.parametrize("NB", NBS)
@pytest.mark.parametrize("seed", range(6))
def test_bucket_map_is_monotone_and_in_range(seed, NB):
    rng = np.random.default_rng(seed)
    for n in (2, 37, 2048):
        for v in _dists(rng, n):
            with np.errstate(over="ignore"):
                v = np.asarray(v, np.float32)
            v = v[np.isfinite(v)]
            if v.size < 2 or v.min() == v.max():
                continue
            b = _buckets(v, NB)
            assert b.min() >= 0 and b.max() < NB
            order = np.argsort(v, kind="stable")
            assert np.all(np.diff(b[order]) >= 0), "a larger score landed in a lower bucket"
            if (v == 0).any():   # -0 and +0 share a bucket
                assert np.all(b[v == 0] == b[v == 0][0])
