"""Pins of the oracle's scalar rules: E2M1, E4M3, Philox4x32-10, stochastic rounding.

Each check compares the oracle with something other than itself: the format
facts of the OCP specifications, closed-form threshold tables, published
known-answer vectors, or the mathematics (fixed points, expectation).
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E2M1_SET = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_are_the_e2m1_set(oracle):
    # The E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; codes 8..15 are the negatives.
    vals = oracle.e2m1_values()
    assert list(vals[:8]) == E2M1_SET
    assert list(vals[8:]) == [-v for v in E2M1_SET]
    assert math.copysign(1.0, vals[8]) == -1.0


def _e2m1_threshold_rule(v: np.ndarray) -> np.ndarray:
    """Closed form of round-to-nearest-even on E2M1 written as thresholds:
    ties at .25 .75 1.25 1.75 2.5 3.5 5 go to the even code (0, 1, 1, 2, 2, 4, 4)."""
    a = np.abs(v.astype(np.float64))
    mag = np.select(
        [a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
        [0, 1, 2, 3, 4, 5, 6], default=7).astype(np.uint8)
    return mag | (np.signbit(v).astype(np.uint8) << 3)


def test_e2m1_rne_against_threshold_table_all_fp32_in_range(oracle):
    # Every FP32 bit pattern with magnitude in [2^-3, 2^4) (where all rounding
    # decisions happen), both signs; outside that range only the saturation
    # and the flush to zero remain, checked on a stride.
    for sign in (0, 1):
        lo = (127 - 3) << 23
        hi = (127 + 4) << 23
        bits = np.arange(lo, hi, dtype=np.uint32) | np.uint32(sign << 31)
        v = bits.view(np.float32)
        assert np.array_equal(oracle.e2m1_rne(v), _e2m1_threshold_rule(v))
        rest = np.concatenate([np.arange(0, lo, 4099, dtype=np.uint32),
                               np.arange(hi, 0x7f800000, 4099, dtype=np.uint32),
                               np.array([0x7f800000 - 1], dtype=np.uint32)]) | np.uint32(sign << 31)
        v = rest.view(np.float32)
        assert np.array_equal(oracle.e2m1_rne(v), _e2m1_threshold_rule(v))


def test_e2m1_rne_every_finite_fp32(oracle):
    # The rest of the 2^32 patterns: every finite FP32 below 2^-3 rounds to a
    # signed zero and every one from 2^4 up saturates to a signed 6 (checked
    # in 2^26-pattern chunks through the oracle's array form).
    lo, hi, step = (127 - 3) << 23, (127 + 4) << 23, 1 << 26
    for sign in (0, 1):
        for a, b, want in ((0, lo, 0), (hi, 0x7f800000, 7)):
            for c0 in range(a, b, step):
                bits = np.arange(c0, min(b, c0 + step), dtype=np.uint32) | np.uint32(sign << 31)
                codes = oracle.e2m1_rne(bits.view(np.float32))
                assert np.all(codes == (want | (sign << 3))), (sign, hex(c0))


def test_e2m1_threshold_rule_is_nearest_with_ties_to_even():
    # The threshold table used above equals "the nearest E2M1 magnitude, ties to
    # the even code" at every tie point, its FP32 neighbours and a dense grid.
    grid = np.array(E2M1_SET)
    mids = (grid[1:] + grid[:-1]) / 2
    pts = [np.float32(m) for m in mids]
    pts += [np.nextafter(np.float32(m), np.float32(0)) for m in mids]
    pts += [np.nextafter(np.float32(m), np.float32(9)) for m in mids]
    v = np.concatenate([np.array(pts, dtype=np.float32), np.linspace(0, 8, 100001, dtype=np.float32)])
    d = np.abs(v.astype(np.float64)[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best                                       # one nearest code, or two at a tie
    code = np.arange(8)[None, :]
    even = cand & (code % 2 == 0)                          # the even code of a tie (mantissa bit 0)
    want = np.where(cand.sum(axis=1) > 1, np.argmax(even, axis=1), np.argmax(cand, axis=1))
    assert np.array_equal(_e2m1_threshold_rule(v), want.astype(np.uint8))


def test_e2m1_rne_special_cases(oracle):
    v = np.array([0.0, -0.0, 6.0, -6.0, 1e30, -1e30, np.inf, -1e-40, 0.25, 0.2500001], dtype=np.float32)
    assert list(oracle.e2m1_rne(v)) == [0, 8, 7, 15, 7, 15, 7, 8, 0, 1]


def _read_e4m3_values():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                b, v = line.split()
                rows.append((int(b, 16), float(eval(v))))
    return rows


def test_e4m3_decode_golden(oracle):
    for b, v in _read_e4m3_values():
        got = oracle.e4m3_value(b)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (hex(b), got, v)
    assert math.isnan(oracle.e4m3_value(0x7f)) and math.isnan(oracle.e4m3_value(0xff))


def test_e4m3_decode_monotone_and_distinct(oracle):
    vals = oracle.e4m3_values()[:0x7f]          # finite non-negative codes in order
    assert np.all(np.diff(vals) > 0)
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9


def test_e4m3_rn_satfinite_against_midpoints(oracle):
    # Closed form: RNE onto the sorted grid g; a value strictly between g[i] and
    # g[i+1] goes to the nearer one; exact midpoints go to the even code.
    g = oracle.e4m3_values()[:0x7f]
    mids = (g[:-1] + g[1:]) / 2
    # midpoints are exact in float32 for this grid
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    codes = oracle.e4m3_rn_satfinite(m32)
    even = np.where(np.arange(0x7e) % 2 == 0, np.arange(0x7e), np.arange(1, 0x7f))
    assert np.array_equal(codes, even.astype(np.uint8))
    below = np.nextafter(m32, np.float32(0))
    above = np.nextafter(m32, np.float32(np.inf))
    assert np.array_equal(oracle.e4m3_rn_satfinite(below), np.arange(0x7e, dtype=np.uint8))
    assert np.array_equal(oracle.e4m3_rn_satfinite(above), np.arange(1, 0x7f, dtype=np.uint8))
    big = np.array([448.0, 464.0, 1e9, np.inf, -500.0], dtype=np.float32)
    assert list(oracle.e4m3_rn_satfinite(big)) == [0x7e, 0x7e, 0x7e, 0x7e, 0xfe]
    # every grid value is a fixed point
    assert np.array_equal(oracle.e4m3_rn_satfinite(g.astype(np.float32)), np.arange(0x7f, dtype=np.uint8))


def _read_kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                w = [int(t, 16) for t in line.split()]
                rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers(oracle):
    for ctr, key, out in _read_kat():
        assert list(oracle.philox4x32_10(ctr, key)) == out


def test_sr_words_follow_the_stream(oracle):
    # element i takes word (i mod 4) of the block with counter i // 4 (low, high, 0, 0)
    seed = 0x1234_5678_9abc
    w = oracle.sr_words(seed, (1 << 34) - 6, 12)
    for j in range(12):
        i = (1 << 34) - 6 + j
        blk = i >> 2
        ref = oracle.philox4x32_10([blk & 0xffffffff, blk >> 32, 0, 0], [seed & 0xffffffff, seed >> 32])
        assert w[j] == ref[i & 3]


def test_sr_fixed_points(oracle):
    # representable values never move, whatever the random word
    g = np.array(E2M1_SET + [-x for x in E2M1_SET], dtype=np.float32)
    for r in (0, 1, 2 ** 31, 2 ** 32 - 1):
        codes = oracle.e2m1_sr(g, np.full(g.shape, r, dtype=np.uint32))
        assert np.array_equal(oracle.e2m1_values()[codes], g.astype(np.float64))


def test_sr_threshold_is_exact(oracle):
    # round up iff r < frac * 2^32 (strict, as real numbers): the switch happens
    # between r = ceil(frac*2^32) - 1 and r = ceil(frac*2^32).
    rng = np.random.default_rng(11)
    v = rng.uniform(0, 6, 4000).astype(np.float32)
    grid = np.array(E2M1_SET)
    lo = np.array([grid[grid <= x].max() for x in v.astype(np.float64)])
    hi = np.array([grid[grid > x].min() if x < 6 else 6.0 for x in v.astype(np.float64)])
    frac = (v.astype(np.float64) - lo) / np.where(hi > lo, hi - lo, 1.0)
    t = np.ceil(frac * 2.0 ** 32)
    keep = (frac > 0) & (t < 2.0 ** 32)
    v, lo, hi, t = v[keep], lo[keep], hi[keep], t[keep]
    vals = oracle.e2m1_values()
    up = vals[oracle.e2m1_sr(v, (t - 1).astype(np.uint32))]
    down = vals[oracle.e2m1_sr(v, t.astype(np.uint32))]
    assert np.array_equal(up, hi) and np.array_equal(down, lo)


def test_sr_is_unbiased(oracle):
    # E[SR(v)] = v: 2^20 draws of the Philox stream per value, 5-sigma z-test,
    # and the up-probability equals frac to within the same bound.
    vals = oracle.e2m1_values()
    n = 1 << 20
    for k, v0 in enumerate([0.1, 0.37, 0.8, 1.3, 1.9, 2.2, 3.7, 4.9, 5.999, -2.6]):
        r = oracle.sr_words(1234 + k, 0, n)
        q = vals[oracle.e2m1_sr(np.full(n, v0, dtype=np.float32), r)]
        v = float(np.float32(v0))
        grid = np.array(E2M1_SET)
        a = abs(v)
        lo = grid[grid <= a].max()
        hi = grid[grid > a].min()
        p = (a - lo) / (hi - lo)
        sd = (hi - lo) * math.sqrt(p * (1 - p) / n)
        assert abs(q.mean() - v) < 5 * sd + 1e-12, (v0, q.mean())
        assert set(np.unique(np.abs(q))) <= {lo, hi}


def test_sr_saturates(oracle):
    v = np.array([6.0, 6.5, 100.0, -7.0], dtype=np.float32)
    assert list(oracle.e2m1_sr(v, np.zeros(4, dtype=np.uint32))) == [7, 7, 7, 15]
