"""Pins of the oracle's router-noise generator (the StandardNormal() draws of
the noisy router, "MoE notes", KeepTopK), when the draws are made rather than
passed in: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, SC 2011) and the
Box-Muller transform.

- the generator against the known-answer vectors its authors publish with it
  (counter, key -> output), three of them;
- the draws against the standard normal: mean, variance, and the
  Kolmogorov-Smirnov distance to the normal CDF over a million draws, plus
  the symmetry of the distribution and the tail mass beyond 3 sigma;
- independence: other seeds and counters give uncorrelated draws, and the
  same (seed, counter) gives the same draws."""
import numpy as np
import pytest
from scipy import stats

import oracle

KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_philox_known_answers(ctr, key, want):
    assert [int(v) for v in oracle.philox4x32_10(ctr, key)] == list(want)


def test_draws_are_standard_normal():
    eps = oracle.draw_noise(2048, 512, seed=0x5EED, counter=7).ravel()
    n = eps.size
    assert abs(eps.mean()) < 5 / np.sqrt(n)
    assert abs(eps.var() - 1.0) < 5 * np.sqrt(2.0 / n)
    assert stats.kstest(eps, "norm").statistic < 2.0 / np.sqrt(n)
    assert abs((eps > 0).mean() - 0.5) < 5 * 0.5 / np.sqrt(n)
    tail = (np.abs(eps) > 3).mean()
    assert abs(tail - 2 * stats.norm.sf(3)) < 5 * np.sqrt(2 * stats.norm.sf(3) / n)


def test_streams_are_independent_and_repeatable():
    a = oracle.draw_noise(256, 64, seed=1, counter=0)
    assert np.array_equal(a, oracle.draw_noise(256, 64, seed=1, counter=0))
    for b in (oracle.draw_noise(256, 64, seed=2, counter=0),
              oracle.draw_noise(256, 64, seed=1, counter=1),
              oracle.draw_noise(256, 64, seed=1 + (1 << 32), counter=0),
              oracle.draw_noise(256, 64, seed=1, counter=1 << 32)):
        assert abs(np.corrcoef(a.ravel(), b.ravel())[0, 1]) < 5 / np.sqrt(a.size)
    # element (t, e) depends on (t, e) only: a smaller table is a corner of a larger one
    assert np.array_equal(oracle.draw_noise(16, 8, seed=1, counter=0), a[:16, :8])
