"""Pins of the oracle's random numbers: Philox4x32-10 against its published
known-answer vectors, the exact uniform conversion, and uniformity."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w = [int(t, 16) for t in line.split()]
        yield w[0:4], w[4:6], w[6:10]


def test_philox_known_answers(orc):
    n = 0
    for ctr, key, want in _kat():
        assert orc.philox4x32_10(ctr, key) == want
        n += 1
    assert n == 3


def test_uniform_conversion_is_exact_24_bit(orc):
    assert orc.u01(0) == 0.0
    assert orc.u01(0xFF) == 0.0  # the low 8 bits are dropped
    assert orc.u01(0x100) == 2.0 ** -24
    assert orc.u01(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    # every value is a multiple of 2^-24, hence exact in fp32
    for w in (0x12345678, 0x9ABCDEF0, 0x80000000):
        u = orc.u01(w)
        assert u * 2 ** 24 == int(u * 2 ** 24)
        assert np.float32(u) == u


def test_round_uniforms_use_the_stated_counter_and_key(orc):
    seed, step, r, i = 0x1122334455667788, 0x0000000A0000000B, 3, 5
    u, u2 = orc.round_uniforms(seed, step, r, i)
    out = orc.philox4x32_10([r, i, step & 0xFFFFFFFF, step >> 32],
                            [seed & 0xFFFFFFFF, seed >> 32])
    assert u == orc.u01(out[0]) and u2 == orc.u01(out[1])


def test_uniforms_are_uniform(orc):
    # chi-square over 64 bins on 40k draws of each word; 1e-4 false-alarm level
    n = 20000
    us = np.array([orc.round_uniforms(0, 0, r, 1) for r in range(n)]).ravel()
    counts = np.bincount((us * 64).astype(int), minlength=64)
    exp = len(us) / 64
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 120.0, chi2  # chi2(63) 99.99th percentile ~ 115
    assert us.min() >= 0.0 and us.max() < 1.0
