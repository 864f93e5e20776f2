"""The quantizer kernel's shortcut for q = clamp(roundf((w - b) / s), 0, 15),
checked as arithmetic on the CPU (no GPU, no library code).

The kernel forms q' = (w - b) * r with r an approximate reciprocal of s
(within a few units in the last place), and keeps roundf(q') wherever q' lies
farther than 1e-5 * max(1, |q'|) from the nearest half-integer; elsewhere it
divides.  That is exact when roundf(q') equals roundf of the correctly rounded
quotient in every kept case.  Here the reciprocal is the correctly rounded
1/s moved by up to four units in the last place either way (a looser error
than the hardware's), and the claim is checked on random and on adversarial
quotients next to half-integers.
"""
import numpy as np


def _round_half_away(v):
    return np.where(v >= 0, np.floor(v + 0.5), -np.floor(-v + 0.5))


def _kept(qf):
    fl = np.floor(qf)
    return np.abs((qf - fl) - np.float32(0.5)) > np.float32(1e-5) * np.maximum(np.float32(1.0), np.abs(qf))


def _check(d, s, ulps):
    d = d.astype(np.float32)
    s = s.astype(np.float32)
    exact = (d / s).astype(np.float32)                      # IEEE float32 division, round to nearest
    r = (np.float32(1.0) / s).astype(np.float32)
    for k in range(-ulps, ulps + 1):
        rk = r.copy()
        step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
        for _ in range(abs(k)):
            rk = np.nextafter(rk, step, dtype=np.float32)
        qf = (d * rk).astype(np.float32)
        keep = _kept(qf)
        # roundf is only ever applied to values whose halves are exact in float32
        a = _round_half_away(qf.astype(np.float64))
        b = _round_half_away(exact.astype(np.float64))
        bad = keep & (a != b)
        assert not bad.any(), (d[bad][:4], s[bad][:4], qf[bad][:4], exact[bad][:4])


def test_random_quotients_in_and_around_the_code_range():
    rng = np.random.default_rng(7)
    s = np.float16(rng.uniform(1e-4, 1.0, 400_000)).astype(np.float32)
    s = s[s > 0]
    q = rng.uniform(-2.0, 17.0, s.size)
    d = (q * s.astype(np.float64)).astype(np.float32)
    _check(d, s, ulps=4)


def test_quotients_next_to_half_integers():
    rng = np.random.default_rng(8)
    s = np.float16(rng.uniform(1e-3, 0.5, 200_000)).astype(np.float32)
    k = rng.integers(-1, 16, s.size).astype(np.float64) + 0.5
    d0 = (k * s.astype(np.float64)).astype(np.float32)
    for off in range(-3, 4):                                 # a few float32 steps from the boundary
        d = d0.copy()
        step = np.float32(np.inf) if off > 0 else np.float32(-np.inf)
        for _ in range(abs(off)):
            d = np.nextafter(d, step, dtype=np.float32)
        _check(d, s, ulps=4)
    # and just outside the margin, where the shortcut decides
    for rel in (1.2e-5, -1.2e-5, 3e-5, -3e-5):
        d = ((k + rel * np.maximum(1.0, np.abs(k))) * s.astype(np.float64)).astype(np.float32)
        _check(d, s, ulps=4)


def test_large_and_tiny_quotients():
    rng = np.random.default_rng(9)
    s = np.float16(rng.uniform(6e-5, 2.0, 100_000)).astype(np.float32)
    q = np.concatenate([rng.uniform(-1e6, 1e6, s.size // 2), rng.uniform(-1e-6, 1e-6, s.size - s.size // 2)])
    d = (q * s.astype(np.float64)).astype(np.float32)
    _check(d, s, ulps=4)
