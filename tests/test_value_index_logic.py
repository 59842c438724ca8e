"""Host model of the value encoder's fast index path (2 and 3 bits), checked on the CPU.

For a group of 32 rotated values y with den = rms + 1e-8 (finite), the encoder
never divides.  The codebook is antisymmetric with its middle boundary at 0.
So with s_k = [y^2 < fl(fl(b_k den)^2)] for the positive boundaries b_k,
m = s_0 + s_1 + ... counts the positive boundaries above |y|, and the index
is m for y <= 0 and 2^bits - 1 - m for y > 0.

The kernel reads these tests from the sign bits of fused multiply-adds:
- the index bits are m's bits xor [y > 0];
- for 3 bits, m's bits are s_1 and s_0 ^ s_1 ^ s_2, because the s_k rise
  together;
- each bit is shifted into the group's packed words with a funnel shift,
  highest stream bit first.

The model replays those steps.  The sign of each fused result is exact in
binary64: y^2 of a float32 is exact, and rounding keeps a sign.  The model
must give the codes of an exact count of boundaries below y / den (away from
the boundaries), packed little-endian at `bits` per code.  CPU only.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F32 = np.float32


def neg_sign(x):
    """Bit 31 of a float32 result, as the kernel reads it."""
    return 1 if np.signbit(F32(x)) else 0


def fast_path_words(y, den, bits, bnd):
    """The kernel's code bits and packed words for one group (y: 32 float32)."""
    H = 1 << (bits - 1)
    t = [F32(F32(bnd[H + k]) * den) for k in range(H - 1)]
    nq = [-float(F32(tk * tk)) for tk in t]
    w = [0] * bits
    for j in range(31, -1, -1):
        yj = float(y[j])
        e = [neg_sign(yj * yj + nqk) for nqk in nq]  # sign set iff y^2 < fl(t^2)
        n = neg_sign(-yj + 0.0)                      # sign set iff y > 0 (+0 for y = +-0)
        if bits == 3:
            ax = e[1] ^ n
            c = [n, ax, e[0] ^ e[2] ^ ax]            # index bits, highest first
        else:
            c = [n, e[0] ^ n]
        for q in range(bits):
            word = (j * bits + bits - 1 - q) >> 5
            w[word] = ((w[word] << 1) | c[q]) & 0xFFFFFFFF  # funnel shift left by one
    return w


def exact_index(yj, den, bnd):
    """Count of boundaries strictly below y / den, in exact rationals."""
    r = Fraction(float(yj)) / Fraction(float(den))
    return sum(1 for b in bnd if Fraction(float(b)) < r)


def pack_le(idx, bits):
    v = sum(int(c) << (i * bits) for i, c in enumerate(idx))
    return [(v >> (32 * k)) & 0xFFFFFFFF for k in range(bits)]


@pytest.mark.parametrize("bits", [2, 3])
def test_fast_index_matches_exact_count(bits):
    """Codes equal the exact count away from boundaries; within 1e-6 of one, either
    neighbouring cell (the squared test rounds fl(b den)^2); packing is exact."""
    _, bnd = oracle.codebook(bits)
    rng = np.random.default_rng(bits)
    near_seen = 0
    for trial in range(400):
        den = F32(np.exp(rng.normal(0, 3)))
        y = (rng.standard_normal(32) * float(den) * rng.choice([0.3, 1.0, 3.0])).astype(F32)
        if trial % 7 == 0:  # values on a threshold and signed zeros
            y[:4] = [F32(0.0), F32(-0.0), F32(F32(bnd[-1]) * den), -F32(F32(bnd[-1]) * den)]
        got = fast_path_words(y, den, bits, bnd)
        v = sum(wd << (32 * k) for k, wd in enumerate(got))
        got_idx = [(v >> (i * bits)) & ((1 << bits) - 1) for i in range(32)]
        want_idx = []
        for yj, gj in zip(y, got_idx):
            want = exact_index(yj, den, bnd)
            if min(abs(float(yj) / float(den) - float(b)) for b in bnd) < 1e-6:
                near_seen += 1
                assert abs(gj - want) <= 1
                want = gj
            want_idx.append(want)
        assert got == pack_le(want_idx, bits), trial
    assert near_seen > 0


def test_signed_zero_takes_the_lower_middle_cell():
    """y = +0 and -0 are not above the middle boundary 0: index 2^(bits-1) - 1."""
    for bits in (2, 3):
        _, bnd = oracle.codebook(bits)
        y = np.full(32, F32(0.0), dtype=F32)
        y[1::2] = F32(-0.0)
        H = 1 << (bits - 1)
        assert fast_path_words(y, F32(1.0), bits, bnd) == pack_le([H - 1] * 32, bits)
