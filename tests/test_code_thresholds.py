"""The write-path kernels decide each INT2 code by three compares instead of a division.

Per-token asymmetric INT2 (axbrief.com OSCAR page, section "attention-statistics rotation + Triton
kernels") defines the code of a clipped value as clamp(rint((x - m) / s), 0, 3) with the fp16 scale
s and minimum m.  The kernels compute d = fl(x - m) and count how many of 0.5 s, 1.5 s, 2.5 s it
passes (d > 0.5 s, d >= 1.5 s, d > 2.5 s): exact because s has at most 11 significant bits, so the
three products are exact fp32 numbers and the halfway points of the IEEE quotient fall strictly
inside one fp32 spacing of them.  This test checks that equivalence for every positive finite fp16
scale, at and around each threshold and over random quotients, with round-half-even ties.
"""
import numpy as np


def _by_division(d, s):
    with np.errstate(all="ignore"):
        q = np.rint(np.float32(d) / np.float32(s))       # IEEE fp32 quotient, ties to even
    return np.clip(q, 0, 3).astype(np.int32)


def _by_compares(d, s):
    return ((d > np.float32(0.5) * s).astype(np.int32) + (d >= np.float32(1.5) * s)
            + (d > np.float32(2.5) * s))


def test_compares_equal_division_for_every_fp16_scale():
    s = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)   # all s > 0
    checked = 0
    for k in (0.5, 1.5, 2.5, 3.0):
        t = (np.float32(k) * s).astype(np.float32)
        for off in range(-24, 25):                    # the threshold and 24 fp32 neighbours each side
            d = (t.view(np.int32) + np.int32(off)).view(np.float32)
            assert np.array_equal(_by_division(d, s), _by_compares(d, s)), (k, off)
            checked += d.size
    rng = np.random.default_rng(7)
    for _ in range(20):                               # quotients spread over [-1, 4)
        d = (s * rng.uniform(-1.0, 4.0, s.size).astype(np.float32)).astype(np.float32)
        assert np.array_equal(_by_division(d, s), _by_compares(d, s))
        checked += d.size
    for d0 in (0.0, -0.0, 1e-45, -1e-45, 3.0e38, -3.0e38):
        d = np.full(s.size, d0, np.float32)
        assert np.array_equal(_by_division(d, s), _by_compares(d, s)), d0
    assert checked > 5_000_000


def test_exact_ties_round_to_even():
    # d = 0.5 s, 1.5 s, 2.5 s exactly: rint gives 0, 2, 2
    s = np.float32(0.125)
    d = np.array([0.0625, 0.1875, 0.3125], np.float32)
    assert _by_division(d, s).tolist() == [0, 2, 2]
    assert _by_compares(d, s).tolist() == [0, 2, 2]
