"""Host model of the value encoder's fast index path (2, 3 and 4 bits), checked on the CPU.

For a group of 32 rotated values y with den = rms + 1e-8 (finite), the encoder
never divides.  The codebook is antisymmetric with its middle boundary at 0,
so with m = #{positive b_k : b_k den < |y|} the index is H-1-m for y <= 0 and
H+m for y > 0 (H = 2^(bits-1)), i.e. 2 idx = 2H-1 + s (2m+1), s = +1 iff y > 0.

The kernel's steps, replayed here:
- a power of two K per group with K den in [2^40, 2^41) (from den's exponent);
- kv = fma(y, -K, 0), whose sign bit is set iff y > 0 (+0 for y = +-0);
- threshold tests sat(fma(kv, kv, -fl(fl(K fl(b den)))^2)), which must come out
  exactly 0 or 1 (the model checks that no value lands strictly inside (0, 1));
- m by binary search: at 3 bits the middle threshold's test picks which outer
  threshold to test next, through nsel = fma(b1, fl(nt2 - nt0), nt0); at 4
  bits two levels of such picks (the last from two picked candidates);
- s (2m+1) summed into float chunks of C = 21 // bits codes weighted
  2^(bits i) on top of 1.5*2^23 + (2H-1) * (sum of weights), which must stay
  exact integers below 2^22 above 1.5*2^23;
- the chunks' low 22 bits (twice the chunk) placed at bit C*bits*c of the
  group's little-endian words.

The model must give the codes of an exact count of boundaries below y / den
(away from the boundaries), packed little-endian at `bits` per code.  CPU only.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F32 = np.float32
M = 12582912  # 1.5 * 2^23


def f32_bits(x):
    return int(np.array([x], dtype=F32).view(np.uint32)[0])


def sat_fma(a, b, c):
    """sat(a*b + c) of float32 operands; the kernel needs the exact value outside (0, 1)."""
    v = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    if v <= 0:
        return 0
    assert v >= 1, "a saturated test landed inside (0, 1)"
    return 1


def fast_path_words(y, den, bits, bnd):
    """The kernel's packed words for one group (y: 32 float32, den float32)."""
    H = 1 << (bits - 1)
    C = 21 // bits
    NC = (32 + C - 1) // C
    K = F32(np.array([(294 - (f32_bits(den) >> 23)) << 23], dtype=np.uint32).view(F32)[0])
    assert 2.0 ** 40 <= float(K) * float(den) < 2.0 ** 41
    t = [F32(F32(F32(bnd[H + k]) * den) * K) for k in range(H - 1)]
    nt = [F32(-F32(tk * tk)) for tk in t]
    acc = []
    for c in range(NC):
        wsum = sum((2 * H - 1) << (bits * i) for i in range(C) if c * C + i < 32)
        acc.append(M + wsum)
    for j in range(32):
        kv = F32(F32(y[j]) * F32(-K) + F32(0.0))  # fma(y, -K, 0): exact product (power of two)
        if bits == 4:
            b1 = sat_fma(kv, kv, nt[3])
            n2 = nt[1] if b1 == 0 else F32(F32(nt[5] - nt[1]) + nt[1])
            b2 = sat_fma(kv, kv, n2)
            lo = nt[0] if b1 == 0 else F32(F32(nt[4] - nt[0]) + nt[0])
            hi = nt[2] if b1 == 0 else F32(F32(nt[6] - nt[2]) + nt[2])
            n3 = lo if b2 == 0 else F32(F32(hi - lo) + lo)
            b3 = sat_fma(kv, kv, n3)
            q = 8 * b1 + 4 * b2 + 2 * b3 + 1
        elif bits == 3:
            b1 = sat_fma(kv, kv, nt[1])
            d = F32(nt[2] - nt[0])
            nsel = nt[0] if b1 == 0 else F32(d + nt[0])
            b2 = sat_fma(kv, kv, nsel)
            q = 4 * b1 + 2 * b2 + 1
        else:
            q = 2 * sat_fma(kv, kv, nt[0]) + 1
        s = 1 if np.signbit(kv) else -1  # sign bit of kv set iff y > 0
        acc[j // C] += s * q * (1 << (bits * (j % C)))
        assert M <= acc[j // C] < M + (1 << 22)  # exact in float32 (ulp 1 there)
    w = [0] * bits
    for c in range(NC):
        u = (acc[c] - M) & 0x3FFFFF  # the chunk's low 22 bits: twice the chunk
        bit = c * C * bits
        word, off = bit >> 5, bit & 31
        nbits = min(C, 32 - c * C) * bits
        w[word] += (u >> 1) if off == 0 else ((u << (off - 1)) & 0xFFFFFFFF)
        if off + nbits > 32:
            w[word + 1] += u >> (33 - off)
    return [x & 0xFFFFFFFF for x in w]


def exact_index(yj, den, bnd):
    """Count of boundaries strictly below y / den, in exact rationals."""
    r = Fraction(float(yj)) / Fraction(float(den))
    return sum(1 for b in bnd if Fraction(float(b)) < r)


def pack_le(idx, bits):
    v = sum(int(c) << (i * bits) for i, c in enumerate(idx))
    return [(v >> (32 * k)) & 0xFFFFFFFF for k in range(bits)]


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_fast_index_matches_exact_count(bits):
    """Codes equal the exact count away from boundaries; within 1e-6 of one, either
    neighbouring cell (the squared tests round fl(b den)^2, and at 3 bits the
    outer threshold comes from one more rounding); packing is exact."""
    _, bnd = oracle.codebook(bits)
    rng = np.random.default_rng(bits)
    near_seen = 0
    for trial in range(400):
        den = F32(np.exp(rng.normal(0, 3))) + F32(1e-8)
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
    for bits in (2, 3, 4):
        _, bnd = oracle.codebook(bits)
        y = np.full(32, F32(0.0), dtype=F32)
        y[1::2] = F32(-0.0)
        H = 1 << (bits - 1)
        assert fast_path_words(y, F32(1.0), bits, bnd) == pack_le([H - 1] * 32, bits)


@pytest.mark.parametrize("den", [1e-8, 3e-8, 1.0, 1e20, 3e37])
def test_extreme_scales(den):
    """The per-group power of two keeps every test saturating and every chunk exact
    from the smallest den (rms 0: den = 1e-8) to the largest finite ones."""
    for bits in (2, 3, 4):
        _, bnd = oracle.codebook(bits)
        d = F32(den)
        rng = np.random.default_rng(int(np.log10(den) + 20) * 10 + bits)
        y = (rng.standard_normal(32) * float(d)).astype(F32)
        y = np.clip(y, -5.6 * float(d), 5.6 * float(d)).astype(F32)  # |y| <= sqrt(32) rms
        got = fast_path_words(y, d, bits, bnd)
        want = [exact_index(yj, d, bnd) for yj in y]
        v = sum(wd << (32 * k) for k, wd in enumerate(got))
        got_idx = [(v >> (i * bits)) & ((1 << bits) - 1) for i in range(32)]
        for g, w_, yj in zip(got_idx, want, y):
            if min(abs(float(yj) / float(d) - float(b)) for b in bnd) >= 1e-6:
                assert g == w_
