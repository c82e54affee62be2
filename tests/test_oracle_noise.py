"""Pins for oracle.noise, the coupled Gumbel noise generated from
Philox4x32-10 (CPU only).  SPOT review, "How it is used": one noise value
per (absolute output position, token), shared by drafter and target; over
the noise, argmax(l/T + G) is distributed as softmax(l/T) (Proposition 2).

* Philox4x32-10 against the published known-answer vectors
  (tests/golden/philox4x32_10_kat.txt).
* The counter layout: tokens 0..3 of position 0 under seed 0 are the four
  words of the first known-answer vector.
* The fp32 logarithm against the library logarithm (math.log): within 2
  units in the last place over a dense grid (the operation sequence keeps
  the series remainder at 4e-9 relative and has no cancellation).
* The uniforms: exact values at the extremes, inside the open interval.
* The Gumbel law (Kolmogorov-Smirnov against exp(-exp(-g)), a library
  routine) and Proposition 2 at T = 0.7, 1, 1.5 (chi-square at V = 4).
"""
import math

import numpy as np
import pytest

from oracle import noise as N
from oracle import accept as A
from golden_io import GOLDEN


def _kat():
    rows = []
    with open(f"{GOLDEN}/philox4x32_10_kat.txt") as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line and line[0] == "kat":
                rows.append([int(x, 16) for x in line[1:]])
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for r in rows:
        out = N.philox4x32_10(r[0], r[1], r[2], r[3], r[4], r[5])
        assert [int(x) for x in out] == r[6:10]


def test_counter_layout_against_first_vector():
    kat = _kat()[0]           # counter (0, 0, 0, 0), key (0, 0)
    bits = N.noise_bits(0, [0], 8)[0]
    assert [int(x) for x in bits[:4]] == kat[6:10]
    # tokens 4..7 come from counter word c0 = 1
    out = N.philox4x32_10(1, 0, 0, 0, 0, 0)
    assert [int(x) for x in bits[4:8]] == [int(x) for x in out]
    # position and seed enter as c1 and the key
    b2 = N.noise_bits((7 << 32) | 5, [3], 4)[0]
    assert [int(x) for x in b2] == [int(x) for x in N.philox4x32_10(0, 3, 0, 0, 5, 7)]


def test_uniform_from_bits():
    u = N.uniform_from_bits(np.array([0, 0xFFFFFFFF, 0x1FF, 0x200, 0x80000000], np.uint32))
    assert u.dtype == np.float32
    assert float(u[0]) == 2.0 ** -24 and float(u[1]) == 1.0 - 2.0 ** -24
    assert float(u[2]) == 2.0 ** -24 and float(u[3]) == 1.5 * 2.0 ** -23
    assert float(u[4]) == 0.5 + 2.0 ** -24
    assert np.all((u > 0) & (u < 1))


def test_log_against_library():
    x = np.concatenate([np.geomspace(2.0 ** -24, 64.0, 200001),
                        1.0 + np.arange(-3000, 3000) * 2.0 ** -24]).astype(np.float32)
    x = x[x > 0]
    got = N.log_f32(x).astype(np.float64)
    ref = np.array([math.log(float(v)) for v in x[::7]])
    g = got[::7]
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(g - ref) <= 2.0 * ulp + 1e-45)
    assert N.log_f32(np.float32(1.0)) == 0.0
    assert abs(float(N.log_f32(np.float32(2.0))) - math.log(2.0)) <= 2.0 ** -24


def test_gumbel_law_ks():
    from scipy import stats
    g = N.gumbel_rows(12345, np.arange(300), 2000).ravel().astype(np.float64)
    ks = stats.kstest(g, lambda t: np.exp(-np.exp(-t)))
    assert ks.pvalue > 1e-3
    n = g.size
    assert abs(g.mean() - 0.5772156649) < 4.5 * (math.pi / math.sqrt(6)) / math.sqrt(n)


@pytest.mark.parametrize("T", [0.7, 1.0, 1.5])
def test_proposition2_with_generated_noise(T):
    from scipy.special import softmax
    l = np.array([0.3, -1.2, 1.1, 0.0], np.float32)
    n = 400_000
    G = N.gumbel_rows(977 + int(10 * T), np.arange(n), 4)
    scores = A.gumbel_scores(l[None, :], G, T)
    counts = np.bincount(np.argmax(scores, axis=1), minlength=4)
    p = softmax(l.astype(np.float64) / float(np.float32(T)))
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < 16.27                                # chi2(3) 0.999 quantile
    assert np.all(np.abs(counts / n - p) < 4.5 * np.sqrt(p * (1 - p) / n))


def test_rows_are_reproducible_and_distinct():
    a = N.gumbel_rows(1, [10, 11], 4096)
    b = N.gumbel_rows(1, [10], 4096)
    c = N.gumbel_rows(2, [10], 4096)
    np.testing.assert_array_equal(a[0], b[0])
    assert not np.array_equal(a[0], a[1]) and not np.array_equal(a[0], c[0])
    assert abs(np.corrcoef(a[0], a[1])[0, 1]) < 0.06 and abs(np.corrcoef(a[0], c[0])[0, 1]) < 0.06
