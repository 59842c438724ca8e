"""Host models of the generic attention kernel's key-code cuts, checked on the CPU.

The kernel turns the 8 key codes a lane needs (dims 32G + 8c .. +7 of a packed
row) into four f16 pairs (dims 2p, 2p + 1).  Each half is an exact f16
integer: koff + code, where koff is 1024 for unsigned codes and 1152 for int8
codes, which are stored offset by 128.  The scores then take the group affine.

The kernel has three cuts:
- 8-bit keys: one 64-bit word, spread with byte permutes;
- 4-bit keys: one 32-bit word, spread with constant shifts;
- every other width: a 64-bit window cut with run-time shifts.

These models restate each cut with the documented semantics of the byte
permute.  They check each half against the codes read straight from the
packed row, for random rows of every width and group.  CPU only.
"""
import numpy as np
import pytest

M32 = 0xFFFFFFFF


def byte_perm(x, y, s):
    """__byte_perm: result byte i is byte (nibble i of s) & 7 of the 8-byte value y:x."""
    src = (y << 32) | x
    return sum(((src >> (8 * ((s >> (4 * i)) & 7))) & 0xFF) << (8 * i) for i in range(4))


def f16_value(h):
    """Value of an f16 bit pattern with a normal exponent (enough for 0x64xx halves)."""
    e, m = (h >> 10) & 0x1F, h & 0x3FF
    assert 0 < e < 31 and not (h >> 15)
    return (1 + m / 1024) * 2.0 ** (e - 15)


def halves(pr):
    return [f16_value(v & 0xFFFF) for v in pr], [f16_value(v >> 16) for v in pr]


def word(row, byte_off, nbytes):
    return int.from_bytes(bytes(row[byte_off:byte_off + nbytes]), "little")


def cut_8bit(row, G, c):
    w = word(row, (4 * G + c) * 8, 8)
    lo, hi = (w & M32) ^ 0x80808080, (w >> 32) ^ 0x80808080
    return [byte_perm(lo, 0x64646464, 0x5140), byte_perm(lo, 0x64646464, 0x5342),
            byte_perm(hi, 0x64646464, 0x5140), byte_perm(hi, 0x64646464, 0x5342)]


def cut_4bit(row, G, c):
    x = word(row, (4 * G + c) * 4, 4)
    out = []
    for p in range(4):
        t = x >> (8 * p)
        out.append(((t & 0x0F) | ((t << 12) & 0x000F0000)) | 0x64006400)
    return out


def cut_window(row, G, c, kb):
    off = (4 * G + c) * kb
    a = off & ~3
    v = (word(row, a + 4, 4) << 32 | word(row, a, 4)) >> ((off & 3) * 8)
    mask = (1 << kb) - 1
    out = []
    for p in range(4):
        c0, c1 = (v >> (2 * p * kb)) & mask, (v >> ((2 * p + 1) * kb)) & mask
        out.append((c0 | (c1 << 16)) | 0x64006400)
    return out


def codes_of(row, d, kb):
    """Codes of a packed key row read straight from its layout (int8 bytes, else an LE bitstream)."""
    if kb == 8:
        return np.frombuffer(bytes(row[:d]), dtype=np.int8).astype(np.int64)
    bits = np.unpackbits(np.frombuffer(bytes(row), dtype=np.uint8), bitorder="little")
    return np.array([int("".join(map(str, bits[i * kb:(i + 1) * kb][::-1])), 2) for i in range(d)])


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("kb", [2, 4, 5, 8])
def test_cut_gives_offset_codes(d, kb):
    rng = np.random.default_rng(1000 * d + kb)
    for _ in range(3):
        # padded by 8 bytes: the 64-bit window may read past the last group's codes
        row = list(rng.integers(0, 256, d * kb // 8 + 8))
        codes = codes_of(row[:d * kb // 8], d, kb)
        koff = 1152 if kb == 8 else 1024
        for G in range(d // 32):
            for c in range(4):
                pr = cut_8bit(row, G, c) if kb == 8 else cut_4bit(row, G, c) if kb == 4 else cut_window(row, G, c, kb)
                lo, hi = halves(pr)
                want = codes[32 * G + 8 * c:32 * G + 8 * c + 8] + koff
                assert [lo[0], hi[0], lo[1], hi[1], lo[2], hi[2], lo[3], hi[3]] == list(map(float, want))


def test_4bit_cut_equals_the_window_cut():
    rng = np.random.default_rng(7)
    for _ in range(200):
        row = list(rng.integers(0, 256, 64 + 8))
        for G in range(4):
            for c in range(4):
                assert cut_4bit(row, G, c) == cut_window(row, G, c, 4)


def test_int8_extremes():
    """-128, -1, 0, 127 land on 1024, 1151, 1152 and 1279."""
    row = [0x80, 0xFF, 0x00, 0x7F, 0x80, 0xFF, 0x00, 0x7F] * 4 + [0] * 8
    lo, hi = halves(cut_8bit(row, 0, 0))
    assert [lo[0], hi[0], lo[1], hi[1]] == [1024.0, 1151.0, 1152.0, 1279.0]
