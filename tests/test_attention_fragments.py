"""Host model of the decode attention kernel's MMA fragments, checked on the CPU.

The head_dim-128 decode kernel reads key codes from a shared-memory tile that a
TMA copy wrote with a 128-byte (8-bit keys) or 64-byte (4-bit keys) swizzle:
the 16-byte chunk index of a row is xor-ed with shared-memory address bits 7..9
(or 7..8).  Each lane (g, c) of a warp reads its rows g and g + 8 at
precomputed swizzled offsets, turns two codes at a time into an f16 pair
(offset + code) with one 3-input logic op and a right shift, and feeds
them to mma.sync m16n8k16 against q fragments permuted the same way.  4-bit
codes in odd nibbles are read in place (1024 + 16 code) and meet q / 16.

This test builds the swizzled tile byte by byte.  It replays every lane's
offsets, loads, conversions and q permutation as the kernel states them, and
emulates the MMA from its documented fragment layout:
- A row-major: lane (g, c) holds A[g][2c..2c+1], A[g+8][2c..2c+1],
  A[g][2c+8..2c+9] and A[g+8][2c+8..2c+9];
- B column-major: lane (n, c) holds B[2c..2c+1][n] and B[2c+8..2c+9][n].

Each score must equal the plain dot product of the offset codes with q over
the key group.  The P V side is checked the same way: which dims and tokens
each lane's value fragments hold, P^T with the rms folded in, and the merge's
map from accumulator rows back to dims must give the plain weighted sum of the
value rows.  CPU only.
"""
import numpy as np
import pytest

from test_key_cuts import f16_value


def swizzled_tile(codes_bytes, krow, kb):
    """Shared-memory image of 16 rows of `krow` bytes under the TMA swizzle of the key map."""
    img = np.zeros(16 * krow, dtype=np.uint8)
    for r in range(16):
        for j in range(krow // 16):
            base = r * krow + 16 * j  # the unswizzled address of chunk j
            f = (base >> 7) & (7 if kb == 8 else 3)
            img[r * krow + 16 * (j ^ f):r * krow + 16 * (j ^ f) + 16] = codes_bytes[r, 16 * j:16 * j + 16]
    return img


def kcvt(w, kb):
    k_const, k_flip = (0xFF00FF00, 0x64806480) if kb == 8 else (0xFFF0FFF0, 0x64006400)
    return ((k_const & k_flip) | (~k_const & (w ^ k_flip))) & 0xFFFFFFFF


def pair(h):
    return f16_value(h & 0xFFFF), f16_value(h >> 16)


def u32(img, a):
    return int.from_bytes(img[a:a + 4].tobytes(), "little")


def lane_a_fragments(img, g, c, G, kb):
    """[mma][a0, a1, a2, a3] as pairs of values, rows g (a0, a2) and g + 8 (a1, a3)."""
    krow = 128 * kb // 8
    r0 = g  # warp 0, first tile
    if kb == 8:
        koff = r0 * krow + (((2 * G + (c >> 1)) ^ g) << 4) + ((c & 1) << 3)
        k0 = (u32(img, koff), u32(img, koff + 4))
        k1 = (u32(img, koff + 8 * krow), u32(img, koff + 8 * krow + 4))
        out = []
        for half in range(2):
            w0, w1 = k0[half], k1[half]
            out.append([pair(kcvt(w0, 8)), pair(kcvt(w1, 8)), pair(kcvt(w0 >> 8, 8)), pair(kcvt(w1 >> 8, 8))])
        return out
    koff = r0 * krow + ((G ^ ((g >> 1) & 3)) << 4) + 4 * c
    w0, w1 = u32(img, koff), u32(img, koff + 8 * krow)
    v0, v1 = w0 >> 8, w1 >> 8

    def odd(w):  # nibbles 1 and 5 of the word in place: 1024 + 16 code
        return (w & 0x00F000F0) | 0x64006400

    return [[pair(kcvt(w0, 4)), pair(kcvt(w1, 4)), pair(odd(w0)), pair(odd(w1))],
            [pair(kcvt(v0, 4)), pair(kcvt(v1, 4)), pair(odd(v0)), pair(odd(v1))]]


def lane_b_fragments(q, n, c, G, kb):
    """[mma][b0, b1] as pairs: q of head n at the dims the A fragments hold."""
    f = q[n, 32 * G + 8 * c:32 * G + 8 * c + 8]
    if kb == 8:  # a word's bytes pair as (0, 2), (1, 3)
        return [[(f[0], f[2]), (f[1], f[3])], [(f[4], f[6]), (f[5], f[7])]]
    # nibbles k and k + 4; the odd ones meet q / 16
    return [[(f[0], f[4]), (f[1] / 16, f[5] / 16)], [(f[2], f[6]), (f[3] / 16, f[7] / 16)]]


@pytest.mark.parametrize("kb", [8, 4])
def test_scores_equal_dot_products(kb):
    """The MMAs give code . q plus the offsets' share: the offset (1152 for
    8-bit keys, 1024 for 4-bit) times the sum of the q values the codes met,
    which is what the kernel subtracts."""
    rng = np.random.default_rng(kb)
    krow = 128 * kb // 8
    if kb == 8:
        codes = rng.integers(-128, 128, (16, 128))
        raw = codes.astype(np.int8).view(np.uint8).reshape(16, 128)
        offset = 1152.0
    else:
        codes = rng.integers(0, 16, (16, 128))
        raw = np.zeros((16, krow), dtype=np.uint8)
        for r in range(16):
            for dd in range(0, 128, 2):
                raw[r, dd // 2] = codes[r, dd] | (codes[r, dd + 1] << 4)
        offset = 1024.0
    img = swizzled_tile(raw, krow, kb)
    q = rng.integers(-8, 9, (8, 128)).astype(np.float64)
    for G in range(4):
        D = np.zeros((16, 8))
        share = np.zeros(8)  # per head: offset x the q values of the B fragments
        for m in range(2):  # the two MMAs of the group
            for g in range(8):
                for n in range(8):
                    for c in range(4):
                        a = lane_a_fragments(img, g, c, G, kb)[m]
                        b = lane_b_fragments(q, n, c, G, kb)[m]
                        # A[row][2c..2c+1] . B[2c..2c+1][n] + A[row][2c+8..+9] . B[2c+8..+9][n]
                        D[g, n] += a[0][0] * b[0][0] + a[0][1] * b[0][1] + a[2][0] * b[1][0] + a[2][1] * b[1][1]
                        D[g + 8, n] += a[1][0] * b[0][0] + a[1][1] * b[0][1] + a[3][0] * b[1][0] + a[3][1] * b[1][1]
                        if g == 0:
                            share[n] += offset * (b[0][0] + b[0][1] + b[1][0] + b[1][1])
        want = codes[:, 32 * G:32 * G + 32] @ q[:, 32 * G:32 * G + 32].T
        assert np.array_equal(D - share[None, :], want)


def test_swizzle_is_a_permutation_of_each_row():
    raw = np.arange(16 * 128, dtype=np.int64).reshape(16, 128).astype(np.uint8)
    for kb, krow in ((8, 128), (4, 64)):
        img = swizzled_tile(raw[:, :krow], krow, kb)
        for r in range(16):
            assert sorted(img[r * krow:(r + 1) * krow]) == sorted(raw[r, :krow])


def test_pv_fragments_and_merge_give_the_weighted_sum():
    """O^T += V^T (P * rms)^T per 32-dim group, then the merge's dim map, equals sum_t p v_hat.

    Per the kernel: lane (g, c) holds dims 32G + 4g + {0..3} of tokens 2c, 2c + 1, 2c + 8 and
    2c + 9.  m-tile 2G + half takes rows g -> dim 32G + 4g + 2 half and g + 8 -> that dim + 1.
    P^T comes from a transpose of the lane's (token g, heads 2c, 2c + 1) pair, so the lane
    gets (tokens 2c, 2c + 1; head g); the rms of those tokens' group multiplies it.
    """
    rng = np.random.default_rng(11)
    V = rng.integers(-7, 8, (16, 128)).astype(np.float64)   # centroid values, per token and dim
    rms = rng.integers(1, 5, (16, 4)).astype(np.float64)    # per token and 32-dim group
    P = rng.integers(0, 6, (16, 8)).astype(np.float64)      # weights, per token and head
    o = np.zeros((8, 4, 8, 4))  # [g][c][m-tile][c0..c3] accumulators of each lane
    for G in range(4):
        for half in range(2):
            mt = 2 * G + half
            for g in range(8):
                for c in range(4):
                    acc = np.zeros(4)
                    for cc in range(4):  # the MMA sums over the k (token) slots of all lanes
                        toks = (2 * cc, 2 * cc + 1, 2 * cc + 8, 2 * cc + 9)
                        d0 = 32 * G + 4 * g + 2 * half
                        # A of lane (g, cc): rows g (dim d0) and g + 8 (dim d0 + 1)
                        a_row_g = [V[t, d0] for t in toks]
                        a_row_g8 = [V[t, d0 + 1] for t in toks]
                        for j in range(2):  # B of lane (n = 2c + j, cc): (P * rms)[toks][n]
                            n = 2 * c + j
                            bcol = [P[t, n] * rms[t, G] for t in toks]
                            acc[j] += sum(x * y for x, y in zip(a_row_g, bcol))
                            acc[2 + j] += sum(x * y for x, y in zip(a_row_g8, bcol))
                    o[g, c, mt] += acc
    merged = np.zeros((8, 128))  # the merge: [head][dim]
    for g in range(8):
        for c in range(4):
            for mt in range(8):
                G, half = mt >> 1, mt & 1
                d0 = 32 * G + 4 * g + 2 * half
                for j in range(2):
                    merged[2 * c + j, d0] = o[g, c, mt, j]
                    merged[2 * c + j, d0 + 1] = o[g, c, mt, 2 + j]
    group_rms = np.repeat(rms, 32, axis=1)  # [token][dim]
    want = P.T @ (V * group_rms)
    assert np.array_equal(merged, want)


# ---------------------------------------------------------------- generic kernel: swizzled key stages
def tma_stage_image(codes_bytes, rb, boxb):
    """Shared-memory image of one 64-row stage of `rb`-byte key rows brought in by
    tensor copies of boxes of `boxb` bytes x 64 rows, box j at j * 64 * boxb, with
    the TMA swizzle of a `boxb`-byte span: bits 4.. of the offset inside the box
    (the 16-byte chunk) xor-ed with the same number of bits from bit 7 up."""
    nbits = {128: 3, 64: 2, 32: 1}[boxb]
    img = np.zeros(64 * rb, dtype=np.uint8)
    for j in range(rb // boxb):
        for r in range(64):
            for col in range(boxb):
                lin = r * boxb + col  # offset inside the box before the swizzle
                sw = lin ^ (((lin >> 7) & ((1 << nbits) - 1)) << 4)
                img[j * 64 * boxb + sw] = codes_bytes[r, j * boxb + col]
    return img


def ksw_addr(r, off, boxb, rows=64):
    """The kernel's read address of byte `off` of row r of a stage of `rows` rows
    (its per-mode form)."""
    box, col = off // boxb, off % boxb
    x = (r & 7) if boxb == 128 else ((r >> 1) & 3) if boxb == 64 else ((r >> 2) & 1)
    return box * rows * boxb + r * boxb + (((col >> 4) ^ x) << 4) + (col & 15)


@pytest.mark.parametrize("d,kb", [(d, kb) for d in (64, 128, 256, 512) for kb in (4, 8)])
def test_generic_swizzled_key_reads(d, kb):
    """Every key word a lane of the generic kernel reads, at every row of a stage,
    is the packed row's word at that offset; and the lanes served together
    (a half-warp for 8-byte loads, the warp for 4-byte ones; lane = 4 g + c,
    row g) conflict at most two ways per load."""
    rb = d * kb // 8
    boxb = min(rb, 128)
    rng = np.random.default_rng(d + kb)
    raw = rng.integers(0, 256, size=(64, rb), dtype=np.uint8)
    img = tma_stage_image(raw, rb, boxb)
    width = 8 if kb == 8 else 4  # bytes one lane loads per group
    for G in range(d // 32):
        for r in range(64):
            for c in range(4):
                off = (4 * G + c) * width
                a = ksw_addr(r, off, boxb)
                assert bytes(img[a:a + width]) == bytes(raw[r, off:off + width])
        groups = ((0, 4), (4, 8)) if width == 8 else ((0, 8),)
        for base in (0, 8, 16, 40):  # the rows of a tile: 16 warp + g (+ 8) + 32 tile
            for g0, g1 in groups:
                words = {}
                for g in range(g0, g1):
                    for c in range(4):
                        a = ksw_addr(base + g, (4 * G + c) * width, boxb)
                        for w in range(width // 4):
                            bank = (a // 4 + w) % 32
                            words.setdefault(bank, set()).add(a // 4 + w)
                assert max(len(v) for v in words.values()) <= 2


@pytest.mark.parametrize("d,kb", [(d, kb) for d in (64, 128, 256) for kb in (4, 8)])
def test_specialised_key_offsets(d, kb):
    """The specialised kernel's per-lane key offsets (one per group, computed once:
    koff[G] = box * ST * SW + r0 * SW + ((chunk ^ xr) << 4) + byte, with the second
    row of a tile 8 SW on and the warp's next tiles 32 SW apart) are the swizzled
    addresses of the lane's bytes of rows r0, r0 + 8, r0 + 32, r0 + 40, ... of a
    stage of ST rows (64 in two tiles per warp; 128 in four at head_dim 64; 96
    in three at head_dim 128 with 4-bit keys)."""
    rb = d * kb // 8
    sw = min(rb, 128)
    tiles = 4 if d == 64 else 3 if (d, kb) == (128, 4) else 2
    st = 32 * tiles
    for warp in range(2):
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            r0 = 16 * warp + g
            xr = g if sw == 128 else ((g >> 1) & 3) if sw == 64 else ((g >> 2) & 1)
            for G in range(d // 32):
                off = 32 * G + 8 * c if kb == 8 else 16 * G + 4 * c
                box, col = off // sw, off % sw
                koff = box * st * sw + r0 * sw + (((col >> 4) ^ xr) << 4) + (col & 15)
                for t2 in range(tiles):
                    for i in range(2):
                        r = r0 + 8 * i + 32 * t2
                        assert koff + t2 * 32 * sw + i * 8 * sw == ksw_addr(r, off, sw, st)
