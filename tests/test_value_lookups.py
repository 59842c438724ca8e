"""Host models of the attention kernels' value-centroid lookups, checked on the CPU.

The decode attention kernels turn value codes into f16 centroids inside
registers.  The A operand of P·V pairs two tokens of one dim in each 32-bit
register.  Two forms are modelled here:
- 3-bit codes: two tokens' 12-bit fields (4 dims each) are spread to one code
  per nibble, `e = y + (y & 0x38383838)`.  Each byte permute then reads the low
  (or high) bytes of 4 centroids from an 8-entry table held in two registers,
  and two more permutes interleave them into (token 1, token 2) f16 pairs.
- 2-bit codes: the selector `ab * 0x22 + 0x1010` (a, b the two tokens' codes)
  picks the f16 pair (c[a], c[b]) from the four centroids in two registers,
  in one permute.

The models restate those steps with the documented byte-permute semantics.
They compare every lookup with the table entry of each code, using random
16-bit table entries so that a swapped byte shows up.  CPU only.
"""
import numpy as np

from test_key_cuts import byte_perm


def tables_3bit(c):
    """(tl0, tl1, th0, th1): low bytes of c0..c3, of c4..c7, then the high bytes."""
    tl0 = sum((c[i] & 0xFF) << (8 * i) for i in range(4))
    tl1 = sum((c[4 + i] & 0xFF) << (8 * i) for i in range(4))
    th0 = sum((c[i] >> 8) << (8 * i) for i in range(4))
    th1 = sum((c[4 + i] >> 8) << (8 * i) for i in range(4))
    return tl0, tl1, th0, th1


def lookup_3bit(x_first, x_second, tabs):
    """A-operand registers for dims r = 0..3 of two tokens, each (c[first code], c[second code])."""
    tl0, tl1, th0, th1 = tabs
    w = byte_perm(x_first, x_second, 0x5410)
    y = ((w & 0x003F003F) | ((w & 0x0FC00FC0) * 4)) & 0xFFFFFFFF
    e = (y + (y & 0x38383838)) & 0xFFFFFFFF
    out = []
    for half in range(2):
        sel = byte_perm(e, 0, 0x0031 if half else 0x0020)
        lo, hi = byte_perm(tl0, tl1, sel), byte_perm(th0, th1, sel)
        out.append(byte_perm(lo, hi, 0x6240))  # dim 2 half
        out.append(byte_perm(lo, hi, 0x7351))  # dim 2 half + 1
    return out


def lookup_2bit(x_first, x_second, c):
    tl0, tl1 = c[0] | (c[1] << 16), c[2] | (c[3] << 16)
    u = x_first | (x_second << 8)
    out = []
    for r in range(4):
        ab = (u >> (2 * r)) & 0x0303
        out.append(byte_perm(tl0, tl1, (ab * 0x22 + 0x1010) & 0xFFFF))
    return out


def test_3bit_lookup_every_code_pair():
    rng = np.random.default_rng(3)
    for _ in range(20):
        c = [int(v) for v in rng.integers(0, 1 << 16, 8)]
        tabs = tables_3bit(c)
        for _ in range(200):
            a = [int(v) for v in rng.integers(0, 8, 4)]
            b = [int(v) for v in rng.integers(0, 8, 4)]
            junk = [int(v) for v in rng.integers(0, 1 << 20, 2)]  # bits above the 12-bit field are ignored
            xa = sum(a[r] << (3 * r) for r in range(4)) | (junk[0] << 12)
            xb = sum(b[r] << (3 * r) for r in range(4)) | (junk[1] << 12)
            got = lookup_3bit(xa & 0xFFFFFFFF, xb & 0xFFFFFFFF, tabs)
            assert got == [c[a[r]] | (c[b[r]] << 16) for r in range(4)]


def test_3bit_lookup_exhaustive_first_dims():
    """All 64 code pairs of dim 0 (the others fixed) select the right entries."""
    c = [0x3C00 + 17 * i for i in range(8)]
    tabs = tables_3bit(c)
    for a0 in range(8):
        for b0 in range(8):
            got = lookup_3bit(a0 | (5 << 3) | (2 << 6) | (7 << 9), b0 | (1 << 3) | (6 << 6) | (3 << 9), tabs)
            assert got[0] == c[a0] | (c[b0] << 16)
            assert got[1:] == [c[5] | (c[1] << 16), c[2] | (c[6] << 16), c[7] | (c[3] << 16)]


def test_2bit_lookup_every_code_pair():
    rng = np.random.default_rng(2)
    for _ in range(50):
        c = [int(v) for v in rng.integers(0, 1 << 16, 4)]
        for xa in range(256):
            xb = int(rng.integers(0, 256))
            got = lookup_2bit(xa, xb, c)
            assert got == [c[(xa >> (2 * r)) & 3] | (c[(xb >> (2 * r)) & 3] << 16) for r in range(4)]
