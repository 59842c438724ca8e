"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than the oracle itself:
a value the pages print (fixtures under tests/golden/, each with its citation),
a closed form, a textbook table, an independent library routine (numpy, scipy,
torch), or brute force on tiny inputs.  CPU only.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.stats

import oracle
from conftest import golden_rows, read_golden

RNG = np.random.default_rng(20240601)


# --------------------------------------------------------------- generator
def test_splitmix64_published_vectors():
    g = read_golden("splitmix64_vectors.txt")
    want = [int(v) for v in g["seed_1234567"].split()]
    assert [oracle.splitmix64(1234567, i) for i in range(5)] == want
    counts = [0] * 5
    for i in range(100000):
        counts[int(oracle.splitmix64(987654321, i) / 2**64 * 5)] += 1
    assert counts == [int(v) for v in g["seed_987654321_floor5_counts"].split()]


def test_sign_vector_definition_and_prefix():
    for d in (64, 128, 256, 512):
        s = oracle.sign_vector(d)
        assert set(np.unique(s)) <= {-1, 1}
        want = [(-1 if (oracle.splitmix64(42, i) >> 63) else 1) for i in range(d)]
        assert s.tolist() == want
    # the smaller head dims use a prefix of the larger vectors
    assert np.array_equal(oracle.sign_vector(512)[:128], oracle.sign_vector(128))


# --------------------------------------------------------------- formats
def test_f16_conversion_matches_numpy():
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** RNG.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e5, -1e5, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
                  1e-10, np.inf, -np.inf, 1.0 + 2**-11, 1.0 + 3 * 2**-11], dtype=np.float32)])
    got = oracle.f32_to_f16_bits(x)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    back = oracle.f16_bits_to_f32(want)
    assert np.array_equal(back, want.view(np.float16).astype(np.float32))
    assert np.isnan(oracle.f16_bits_to_f32(oracle.f32_to_f16_bits(np.float32("nan"))))[0]


def test_bf16_conversion_matches_torch():
    torch = pytest.importorskip("torch")
    x = (RNG.standard_normal(20000) * 10.0 ** RNG.integers(-30, 30, 20000)).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-39, np.inf], dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16_bits(x), want)


# --------------------------------------------------------------- Lloyd-Max
def test_3bit_table_equals_printed_table():
    g = read_golden("codebook_3bit.txt")
    cpos = np.array([float(v) for v in g["centroids_positive"].split()])
    bpos = np.array([float(v) for v in g["boundaries_positive"].split()])
    c, b = oracle.codebook(3)
    assert np.max(np.abs(c[4:] - cpos)) <= 0.5e-5
    assert np.max(np.abs(c[:4] + cpos[::-1])) <= 0.5e-5
    assert np.max(np.abs(b[4:] - bpos)) <= 0.5e-5
    assert np.max(np.abs(b[:3] + bpos[::-1])) <= 0.5e-5
    assert b[3] == float(g["boundary_middle"])
    # rounded to the printed precision the tables agree digit for digit
    assert np.array_equal(np.round(c[4:].astype(np.float64), 5), cpos)
    assert np.array_equal(np.round(b[4:].astype(np.float64), 5), bpos)


def test_lloyd_max_textbook_levels_and_mse():
    for row in golden_rows("lloyd_max_textbook.txt"):
        n_s, lev_s, mse_s = [p.strip() for p in row.split(";")]
        n = int(n_s)
        bits = n.bit_length() - 1
        c, b = oracle.lloyd_max(bits)
        for got, printed in zip(c[n // 2:], lev_s.split()):
            one_digit = 10.0 ** -len(printed.split(".")[1])
            assert abs(got - float(printed)) <= one_digit * 1.0001, (n, got, printed)
        assert abs(oracle.normal_mse(c, b) - float(mse_s)) <= 1e-5 * max(1.0, float(mse_s) * 100)
    anchors = [float(v) for v in read_golden("lloyd_max_textbook.txt")["anchors"].split()]
    for bits, a in zip((1, 2, 3), anchors):
        c, b = oracle.lloyd_max(bits)
        assert abs(oracle.normal_mse(c, b) - a) < 0.01


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_lloyd_max_fixed_point_independent_check(bits):
    """The table satisfies both optimality conditions, evaluated with scipy."""
    c, b = oracle.lloyd_max(bits)
    n = 1 << bits
    assert np.all(np.diff(c) > 0)
    assert np.allclose(c, -c[::-1], atol=1e-12)  # symmetric density -> symmetric table
    assert np.allclose(b, 0.5 * (c[1:] + c[:-1]), atol=0, rtol=0)
    edges = np.concatenate([[-np.inf], b, [np.inf]])
    lo, hi = edges[:-1], edges[1:]
    # conditional mean of each cell, via scipy's truncated normal
    means = scipy.stats.truncnorm.mean(lo, hi)
    assert np.max(np.abs(means - c)) < 1e-9, np.max(np.abs(means - c))
    assert len(c) == n and len(b) == n - 1


def test_lloyd_max_3bit_mse_on_samples():
    """Pages: 3-bit distortion near 0.0345 on unit-normal inputs (10^6 samples)."""
    c, b = oracle.codebook(3)
    x = np.random.default_rng(7).standard_normal(1_000_000).astype(np.float32)
    idx = np.searchsorted(b, x, side="left")
    mse = float(np.mean((x - c[idx]) ** 2))
    assert abs(mse - 0.0345) < 0.001


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_codebook_exactly_symmetric_with_zero_middle(bits):
    """Pages print the middle 3-bit boundary as 0; the N(0,1) quantizer is symmetric."""
    c, b = oracle.codebook(bits)
    assert np.array_equal(c, -c[::-1]) and np.array_equal(b, -b[::-1])
    if bits > 1:
        assert b[len(b) // 2] == 0.0


def test_codebook_f32_is_rounded_binary64():
    for bits in (2, 3, 4, 5, 8):
        c64, b64 = oracle.lloyd_max(bits)
        c, b = oracle.codebook(bits)
        assert np.array_equal(c, c64.astype(np.float32))
        assert np.array_equal(b, b64.astype(np.float32))


# --------------------------------------------------------------- bitstream
def test_pack_worked_example():
    # element i at bits [3i, 3i+3), LSB first:
    # byte0 = 0 | 1<<3 | (2&3)<<6 = 0x88; byte1 = (2>>2) | 3<<1 | 4<<4 | (5&1)<<7 = 0xC6;
    # byte2 = (5>>1) | 6<<2 | 7<<5 = 0xFA.  The pages: 8 three-bit values fill 3 bytes.
    assert oracle.pack_bits(np.arange(8), 3).tolist() == [0x88, 0xC6, 0xFA]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_pack_matches_numpy_packbits(bits):
    for n in (8, 32, 64, 33):
        v = RNG.integers(0, 1 << bits, n).astype(np.uint32)
        bitarr = ((v[:, None] >> np.arange(bits)) & 1).astype(np.uint8).ravel()
        want = np.packbits(bitarr, bitorder="little")
        got = oracle.pack_bits(v, bits)
        assert np.array_equal(got, want)
        assert np.array_equal(oracle.unpack_bits(got, n, bits), v)


def test_pack_every_value_every_offset():
    for bits in (2, 3, 4, 5, 8):
        for off in range(8):
            for val in range(1 << bits):
                v = np.zeros(8 + off, dtype=np.uint32)
                v[off] = val
                packed = oracle.pack_bits(v, bits)
                assert oracle.unpack_bits(packed, len(v), bits)[off] == val
                bit0 = off * bits
                whole = int.from_bytes(packed.tobytes(), "little")
                assert (whole >> bit0) & ((1 << bits) - 1) == val


# --------------------------------------------------------------- FWHT
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_equals_sylvester_matrix(d):
    x = RNG.standard_normal(d).astype(np.float32)
    want = scipy.linalg.hadamard(d) @ x.astype(np.float64) / math.sqrt(d)
    got = oracle.fwht(x)
    assert np.max(np.abs(got - want)) < 4e-6 * np.max(np.abs(want))


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_involution_and_norm(d):
    x = RNG.standard_normal(d).astype(np.float32)
    y = oracle.fwht(x)
    assert abs(np.linalg.norm(y) / np.linalg.norm(x) - 1) < 1e-6
    assert np.max(np.abs(oracle.fwht(y) - x)) < 1e-5
    e0 = np.zeros(d, dtype=np.float32)
    e0[0] = 1.0
    assert np.allclose(oracle.fwht(e0), 1 / math.sqrt(d), rtol=1e-7)


# --------------------------------------------------------------- keys
def test_key_group_signed_worked_example():
    # min -127, max 127: scale = 254/254 = 1, zero = round(0/2) = 0 -> idx = round(x)
    x = np.array([-127, 127, 0, 1, -1, 5, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5, -126.5, 3.25, 3.75, -3.75]
                 + [10] * 16, dtype=np.float32)
    idx, s, z = oracle.key_group(x, 8)
    assert oracle.f16_bits_to_f32([s])[0] == 1.0 and oracle.f16_bits_to_f32([z])[0] == 0.0
    # half-to-even rounding (the reading of "round")
    assert idx[:16].tolist() == [-127, 127, 0, 1, -1, 5, 0, 2, 2, 0, -2, 126, -126, 3, 4, -4]


def test_key_group_unsigned_worked_example():
    for bits in (2, 4, 5):
        m = (1 << bits) - 1
        x = np.resize(np.arange(m + 1, dtype=np.float32), 32)
        idx, s, z = oracle.key_group(x, bits)
        assert oracle.f16_bits_to_f32([s])[0] == 1.0 and oracle.f16_bits_to_f32([z])[0] == 0.0
        assert np.array_equal(idx, x.astype(np.int32))
        # shifted: min 10 -> zero = round(10/1) = 10, indices unchanged
        idx2, s2, z2 = oracle.key_group(x + 10, bits)
        assert oracle.f16_bits_to_f32([z2])[0] == 10.0 and np.array_equal(idx2, idx)
        deq = oracle.key_group_dequant(idx2, s2, z2)
        assert np.array_equal(deq, x + 10)


@pytest.mark.parametrize("bits", [2, 4, 5, 8])
def test_key_group_error_bound(bits):
    """Affine round-to-nearest: an unclipped key is within half a step of its code.
    A code clipped at the end of the range (the zero point is itself rounded)
    can be up to one step away."""
    lo, hi = (-127, 127) if bits == 8 else (0, (1 << bits) - 1)
    for _ in range(300):
        x = (RNG.standard_normal(32) * math.exp(RNG.uniform(-3, 3))).astype(np.float32)
        idx, s, z = oracle.key_group(x, bits)
        assert idx.min() >= lo and idx.max() <= hi
        sf = oracle.f16_bits_to_f32([s])[0]
        zf = oracle.f16_bits_to_f32([z])[0]
        deq = oracle.key_group_dequant(idx, s, z)
        scale32 = (x.max() - x.min()) / (254.0 if bits == 8 else (1 << bits) - 1)
        # what storing the scale in fp16 can move, plus fp32 rounding
        slack = np.abs(idx + zf) * abs(sf - scale32) + 1e-6 * np.abs(x).max()
        inner = (idx > lo) & (idx < hi)
        err = np.abs(x - deq)
        assert np.all(err[inner] <= 0.5 * scale32 * (1 + 1e-5) + slack[inner])
        assert np.all(err[~inner] <= 1.0 * scale32 * (1 + 1e-5) + slack[~inner])


def test_key_group_constant_block_defect():
    """Pages: a constant-valued block overflows the zero point to +-Inf (kept on purpose)."""
    for bits in (8, 4):
        idx, s, z = oracle.key_group(np.full(32, 1.5, dtype=np.float32), bits)
        assert s == 0x0000 and z == 0x7C00
        assert np.all(np.isnan(oracle.key_group_dequant(idx, s, z)))
        idx, s, z = oracle.key_group(np.full(32, -2.0, dtype=np.float32), bits)
        assert s == 0x0000 and z == 0xFC00
    # all zeros: 0/0 -> NaN zero point
    idx, s, z = oracle.key_group(np.zeros(32, dtype=np.float32), 8)
    assert s == 0 and (z & 0x7C00) == 0x7C00 and (z & 0x3FF) != 0
    assert np.all(idx == -127)  # NaN clips to the low end (maxNum/minNum reading)


# --------------------------------------------------------------- values
def test_value_index_is_nearest_centroid_brute_force():
    for bits in (2, 3, 4, 5):
        c, b = oracle.codebook(bits)
        for d in (64, 128):
            x = RNG.standard_normal(d).astype(np.float32)
            idx, sc, yn = oracle.value_row(x, bits)
            brute = np.argmin(np.abs(yn[:, None].astype(np.float64) - c[None, :].astype(np.float64)), axis=1)
            away = np.min(np.abs(yn[:, None] - b[None, :]), axis=1) > 1e-6
            assert np.array_equal(idx[away], brute[away])


def test_value_scale_is_group_rms_of_rotated_row():
    d = 128
    x = RNG.standard_normal(d).astype(np.float32)
    s = oracle.sign_vector(d)
    y = scipy.linalg.hadamard(d) @ (x * s).astype(np.float64) / math.sqrt(d)
    rms = np.sqrt(np.mean(y.reshape(-1, 32) ** 2, axis=1))
    _, sc, yn = oracle.value_row(x, 3)
    assert np.allclose(oracle.f16_bits_to_f32(sc), rms, rtol=2 ** -10)
    assert np.allclose(yn, (y.reshape(-1, 32) / rms[:, None]).ravel(), atol=1e-5)


@pytest.mark.parametrize("bits,lo,hi", [(2, 0.10, 0.13), (3, 0.030, 0.038), (4, 0.0085, 0.0105)])
def test_value_roundtrip_mse_band(bits, lo, hi):
    """Pages: 3-bit roundtrip MSE on unit-normal data in the D_mse ~ 0.03 band."""
    err = tot = 0.0
    for _ in range(64):
        x = RNG.standard_normal(128).astype(np.float32)
        idx, sc, _ = oracle.value_row(x, bits)
        xh = oracle.value_row_dequant(idx, sc, bits)
        err += float(np.sum((x - xh) ** 2))
        tot += float(np.sum(x * x))
    assert lo < err / tot < hi, err / tot


def test_value_dequant_order_fwht_then_signs():
    """Earlier page: the inverse is 'apply FWHT then multiply signs'."""
    d = 64
    c, _ = oracle.codebook(3)
    idx = RNG.integers(0, 8, d).astype(np.int32)
    sc = oracle.f32_to_f16_bits(np.full(d // 32, 1.25, dtype=np.float32))
    got = oracle.value_row_dequant(idx, sc, 3)
    rot = c[idx].astype(np.float64) * 1.25
    want = oracle.sign_vector(d) * (scipy.linalg.hadamard(d) @ rot / math.sqrt(d))
    assert np.max(np.abs(got - want)) < 1e-5


# --------------------------------------------------------------- layout
def test_bytes_per_token_head_pages_figure():
    g = read_golden("bytes_per_token_head.txt")
    d, kb, vb = int(g["head_dim"]), int(g["k_bits"]), int(g["v_bits"])
    total = oracle.bytes_per_token_head(d, kb, vb)
    assert total == int(g["total"])
    assert total == int(g["k_codes"]) + int(g["k_scale_zero"]) + int(g["v_codes"]) + int(g["v_scale"])
    assert round(int(g["bf16_bytes"]) / total, 2) == float(g["ratio"])


def test_effective_bits_table():
    for row in golden_rows("effective_bits.txt"):
        name, kb, vb, eff = row.split()
        for d in (64, 128, 256, 512):
            bits = oracle.bytes_per_token_head(d, int(kb), int(vb)) * 8 / (2 * d)
            assert bits == float(eff), (name, d, bits)


# --------------------------------------------------------------- whole cache
def _bf16(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32)).reshape(np.shape(a))


def _small_cache(B=2, H=2, T=24, d=64, kb=8, vb=3, cap=32, t0=0):
    k = _bf16(RNG.standard_normal((B, H, T, d)))
    v = _bf16(RNG.standard_normal((B, H, T, d)))
    p = oracle.Planes(B, H, d, kb, vb, cap)
    oracle.encode(p, k, v, t0=t0)
    return p, k, v


def test_encode_rows_match_row_functions():
    p, k, v = _small_cache(kb=4, vb=3, t0=5)
    b, h, t = 1, 0, 7
    row = t + 5
    x = oracle.bf16_bits_to_f32(k[b, h, t])
    for g in range(2):
        idx, s, z = oracle.key_group(x[32 * g:32 * g + 32], 4)
        assert p.k_scale[b, h, row, g] == s and p.k_zero[b, h, row, g] == z
        assert np.array_equal(p.k_codes[b, h, row, 16 * g:16 * g + 16], oracle.pack_bits(idx, 4))
    idx, sc, _ = oracle.value_row(oracle.bf16_bits_to_f32(v[b, h, t]), 3)
    assert np.array_equal(p.v_scale[b, h, row], sc)
    assert np.array_equal(p.v_codes[b, h, row], oracle.pack_bits(idx, 3))
    # append writes rows [t0, t0+n) only
    assert not p.k_codes[:, :, :5].any() and not p.v_scale[:, :, 5 + 24:].any()


def test_decode_inverts_encode_within_quantization_error():
    p, k, v = _small_cache(d=128, T=16, cap=16)
    ko, vo = oracle.decode(p, 0, 16)
    kx = oracle.bf16_bits_to_f32(k)
    vx = oracle.bf16_bits_to_f32(v)
    assert np.max(np.abs(ko - kx)) < 0.05
    assert np.mean((vo - vx) ** 2) / np.mean(vx ** 2) < 0.05


def test_attention_single_token_returns_its_value():
    p, k, v = _small_cache(B=1, H=2, T=1, d=64, cap=16)
    q = _bf16(RNG.standard_normal((1, 4, 64)))
    out = oracle.attention(p, q, 1)
    _, vo = oracle.decode(p, 0, 1, want_k=False)
    for qh in range(4):
        assert np.allclose(out[0, qh], vo[0, qh // 2, 0], atol=1e-7)


def test_attention_identical_keys_average_values():
    B, H, T, d = 1, 1, 9, 64
    k1 = RNG.standard_normal(d)
    k = _bf16(np.broadcast_to(k1, (B, H, T, d)))
    v = _bf16(RNG.standard_normal((B, H, T, d)))
    p = oracle.Planes(B, H, d, 8, 3, 16)
    oracle.encode(p, k, v)
    q = _bf16(RNG.standard_normal((1, 2, d)))
    out = oracle.attention(p, q, T)
    _, vo = oracle.decode(p, 0, T, want_k=False)
    assert np.allclose(out[0, 0], vo[0, 0].astype(np.float64).mean(axis=0), atol=1e-6)


def test_attention_dominant_logit_selects_its_value():
    B, H, T, d = 1, 1, 12, 64
    k = RNG.standard_normal((B, H, T, d)) * 0.01
    q = RNG.standard_normal((1, 1, d))
    k[0, 0, 7] = 40.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    kb16, qb16 = _bf16(k), _bf16(q)
    v = _bf16(RNG.standard_normal((B, H, T, d)))
    p = oracle.Planes(B, H, d, 8, 3, 16)
    oracle.encode(p, kb16, v)
    out = oracle.attention(p, qb16, T)
    _, vo = oracle.decode(p, 0, T, want_k=False)
    assert np.allclose(out[0, 0], vo[0, 0, 7], atol=1e-6)


def _integer_key_rows(base_rows, d):
    """Key rows of integers whose every 32-group holds both 127 and -127, so
    the 8-bit affine has scale (127 - (-127)) / 254 = 1 and zero rint(0) = 0:
    the codes are the integers themselves and k_hat = x exactly."""
    k = np.array(base_rows, dtype=np.float64)
    for g in range(d // 32):
        k[:, 32 * g] = 127.0
        k[:, 32 * g + 1] = -127.0
    return k


def _closed_form_cache(k_rows, d=64, seed=0):
    """One sequence, one kv-head: integer key rows (exact k_hat) and random
    value rows; returns the planes, the exact keys and the decoded v_hat."""
    T = k_rows.shape[0]
    rng = np.random.default_rng(seed)
    v = _bf16(rng.standard_normal((1, 1, T, d)))
    p = oracle.Planes(1, 1, d, 8, 3, 16)
    oracle.encode(p, _bf16(k_rows.reshape(1, 1, T, d)), v)
    ko, vo = oracle.decode(p, 0, T)
    assert np.array_equal(ko[0, 0].astype(np.float64), k_rows)  # precondition: k_hat exact
    return p, vo[0, 0].astype(np.float64)


def test_attention_two_rows_closed_form():
    """Two cache rows: o = (v1 + e^D v2) / (1 + e^D), D = scale * q.(k2 - k1).

    The keys are integers the 8-bit affine reproduces exactly, so D is exact
    and needs no dequantisation; the weights are written out for two rows (no
    max subtraction, no running sums).  At the default scale 1/sqrt(d) D = 1;
    at scale ln(3)/8 the weights are exactly 1/4 and 3/4.  Dropping the scale
    from the oracle's scores (s_t = dot), or applying it twice, moves the
    output by more than 0.1 here, far outside the 1e-12 bound (checked by
    planting that change in the oracle on the CPU)."""
    d = 64
    rng = np.random.default_rng(77)
    base = rng.integers(-60, 61, size=(1, d)).astype(np.float64)
    k = _integer_key_rows(np.repeat(base, 2, axis=0), d)
    k[1, 10] = k[0, 10] + 8.0  # rows differ in one dim by 8
    q = np.zeros(d)
    q[10] = 1.0
    q[40] = -2.0  # same in both rows: shifts both logits alike
    qb = _bf16(q.reshape(1, 1, d))
    p, vh = _closed_form_cache(k, d, seed=5)
    dlt = float(q @ (k[1] - k[0]))
    assert dlt == 8.0
    # default scale 1/sqrt(64): D = 1
    e = math.exp(dlt / math.sqrt(d))
    want = (vh[0] + e * vh[1]) / (1.0 + e)
    got = oracle.attention(p, qb, 2)[0, 0]
    assert np.max(np.abs(got - want)) <= 1e-12
    # scale ln(3)/8: e^D = 3 exactly, so o = (v1 + 3 v2) / 4
    got = oracle.attention(p, qb, 2, softmax_scale=math.log(3.0) / 8.0)[0, 0]
    assert np.max(np.abs(got - (vh[0] + 3.0 * vh[1]) / 4.0)) <= 1e-12
    # the weighting is visible: the two rows' values differ
    assert np.max(np.abs(vh[0] - vh[1])) > 0.5


def test_attention_three_rows_distinct_weights():
    """Three rows whose scores differ by scale * (0, 8, 16): at scale ln(2)/8 the
    weights are exactly 1/7, 2/7, 4/7, so a wrong normaliser, a max subtracted
    from one row only, or a scale applied anywhere but the scores shows; the
    default scale 1/sqrt(d) is checked against the three-term closed form."""
    d = 64
    rng = np.random.default_rng(78)
    base = rng.integers(-60, 61, size=(1, d)).astype(np.float64)
    k = _integer_key_rows(np.repeat(base, 3, axis=0), d)
    k[1, 20] = k[0, 20] + 8.0
    k[2, 20] = k[0, 20] + 16.0
    q = np.zeros(d)
    q[20] = 1.0
    qb = _bf16(q.reshape(1, 1, d))
    p, vh = _closed_form_cache(k, d, seed=6)
    got = oracle.attention(p, qb, 3, softmax_scale=math.log(2.0) / 8.0)[0, 0]
    assert np.max(np.abs(got - (vh[0] + 2.0 * vh[1] + 4.0 * vh[2]) / 7.0)) <= 1e-12
    w = np.exp(np.array([0.0, 1.0, 2.0]))  # default scale 1/8: scores differ by 0, 1, 2
    want = (w[0] * vh[0] + w[1] * vh[1] + w[2] * vh[2]) / w.sum()
    got = oracle.attention(p, qb, 3)[0, 0]
    assert np.max(np.abs(got - want)) <= 1e-12


def test_attention_deferred_unrotation_equals_eager():
    """Pages, 'Deferred inverse FWHT': attention is linear in V, so un-rotating the
    weighted sum equals the weighted sum of un-rotated rows."""
    d, T = 128, 20
    c, _ = oracle.codebook(3)
    signs = oracle.sign_vector(d)
    w = RNG.random(T)
    w /= w.sum()
    rot = []
    eager = np.zeros(d)
    for t in range(T):
        idx, sc, _ = oracle.value_row(RNG.standard_normal(d).astype(np.float32), 3)
        r = c[idx].astype(np.float64) * np.repeat(oracle.f16_bits_to_f32(sc), 32)
        rot.append(r)
        eager += w[t] * oracle.value_row_dequant(idx, sc, 3)
    deferred = signs * oracle.fwht(np.sum([w[t] * rot[t] for t in range(T)], axis=0).astype(np.float32))
    assert np.max(np.abs(deferred - eager)) < 1e-5


# ---------------------------------------------------------------- deferred fetch (page: "Deferred inverse FWHT")
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_unrotate_basis_vectors_closed_form(d):
    """unrotate(e_k)_j = s_j * (-1)^popcount(j & k) * fl(1/sqrt d): the Sylvester
    index convention, the normalisation and signs applied last, exactly."""
    s = oracle.sign_vector(d).astype(np.float32)
    c = np.float32(1.0 / math.sqrt(d))
    for k in (0, 1, 5, d // 2, d - 1):
        e = np.zeros(d, dtype=np.float32)
        e[k] = 1.0
        want = np.array([s[j] * (-1.0 if bin(j & k).count("1") % 2 else 1.0) for j in range(d)], dtype=np.float32) * c
        assert np.array_equal(oracle.unrotate(e), want)


@pytest.mark.parametrize("d", [64, 128, 512])
def test_unrotate_inverts_the_encoder_rotation(d):
    """The encoder rotates y = FWHT(x * s)/sqrt(d); H H = d I and s * s = 1, so
    unrotate(y) = x up to fp32 rounding."""
    rng = np.random.default_rng(d)
    x = rng.standard_normal(d).astype(np.float32)
    y = oracle.fwht(x * oracle.sign_vector(d).astype(np.float32))
    back = oracle.unrotate(y)
    assert np.max(np.abs(back - x)) < 2e-6 * np.max(np.abs(x)) * math.log2(d)
    assert abs(np.linalg.norm(back) - np.linalg.norm(x)) < 1e-5 * np.linalg.norm(x)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_rotated_row_then_unrotate_is_the_dequantised_row(bits):
    """Deferred and eager paths split the same formula: centroid[idx]*rms, then
    signs * FWHT(.)/sqrt(d) -- identical arithmetic for a single row."""
    rng = np.random.default_rng(bits)
    d = 128
    idx = rng.integers(0, 1 << bits, d)
    sc = oracle.f32_to_f16_bits(rng.uniform(0.1, 3.0, d // 32).astype(np.float32))
    rot = oracle.value_row_rotated(idx, sc, bits)
    c = oracle.codebook(bits)[0]
    assert np.array_equal(rot, (c[idx] * np.repeat(oracle.f16_bits_to_f32(sc), 32)).astype(np.float32))
    assert np.array_equal(oracle.unrotate(rot), oracle.value_row_dequant(idx, sc, bits))


def test_deferred_weighted_sum_equals_eager():
    """The page's identity InvFWHT(sum w_i v_i) = sum w_i InvFWHT(v_i), in fp32."""
    rng = np.random.default_rng(7)
    d, n = 128, 50
    idx = rng.integers(0, 8, (n, d))
    sc = oracle.f32_to_f16_bits(rng.uniform(0.1, 3.0, (n, d // 32)).astype(np.float32)).reshape(n, d // 32)
    w = rng.dirichlet(np.ones(n))
    rot = np.stack([oracle.value_row_rotated(idx[i], sc[i], 3) for i in range(n)]).astype(np.float64)
    eager = np.stack([oracle.value_row_dequant(idx[i], sc[i], 3) for i in range(n)]).astype(np.float64)
    deferred = oracle.unrotate((w @ rot).astype(np.float32))
    assert np.max(np.abs(deferred - w @ eager)) < 1e-5 * np.max(np.abs(w @ eager))


# ---------------------------------------------------------------- cache lifecycle (token slices are byte-safe)
def test_copy_rows_then_decode_equals_source_rows():
    rng = np.random.default_rng(11)
    B, H, d, T = 2, 2, 64, 20
    k = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, T, d)).astype(np.float32)).reshape(B, H, T, d)
    v = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, T, d)).astype(np.float32)).reshape(B, H, T, d)
    src = oracle.Planes(B, H, d, 4, 3, 32)
    oracle.encode(src, k, v)
    dst = oracle.Planes(B, H, d, 4, 3, 48)  # larger capacity: growth
    oracle.copy_rows(dst, 7, src, 3, 12)
    for a, b in zip(oracle.decode(dst, 7, 12), oracle.decode(src, 3, 12)):
        assert np.array_equal(a, b)
    assert all(np.all(a[:, :, :7] == 0) and np.all(a[:, :, 19:] == 0) for a in dst.arrays())


def test_trim_then_reappend_equals_encoding_the_kept_and_new_tokens():
    rng = np.random.default_rng(12)
    B, H, d = 1, 3, 128
    k = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, 30, d)).astype(np.float32)).reshape(B, H, 30, d)
    v = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, 30, d)).astype(np.float32)).reshape(B, H, 30, d)
    cache = oracle.Planes(B, H, d, 8, 3, 32)
    oracle.encode(cache, k[:, :, :20], v[:, :, :20])
    oracle.clear_rows(cache, 12, 20)            # trim to 12 tokens
    oracle.encode(cache, k[:, :, 20:30], v[:, :, 20:30], t0=12)
    fresh = oracle.Planes(B, H, d, 8, 3, 32)
    keep = np.concatenate([k[:, :, :12], k[:, :, 20:30]], axis=2), np.concatenate([v[:, :, :12], v[:, :, 20:30]], axis=2)
    oracle.encode(fresh, *keep)
    for a, b in zip(cache.arrays(), fresh.arrays()):
        assert np.array_equal(a, b)


# ---------------------------------------------------------------- multi-token queries (causal)
def _mt_planes(seed, B=1, H=2, d=64, T=24):
    rng = np.random.default_rng(seed)
    k = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, T, d)).astype(np.float32)).reshape(B, H, T, d)
    v = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, T, d)).astype(np.float32)).reshape(B, H, T, d)
    p = oracle.Planes(B, H, d, 8, 3, 32)
    oracle.encode(p, k, v)
    return p, rng


def test_multi_token_one_query_is_decode_attention():
    p, rng = _mt_planes(21)
    q = oracle.f32_to_bf16_bits(rng.standard_normal((1, 1, 8, 64)).astype(np.float32)).reshape(1, 1, 8, 64)
    assert np.array_equal(oracle.attention_multi(p, q, 20)[:, 0], oracle.attention(p, q[:, 0], 20))


def test_multi_token_causality():
    """Query i must not see rows past its own position: changing those rows
    leaves it unchanged, while the last query (which sees them) changes."""
    p, rng = _mt_planes(22)
    M, T = 4, 20
    q = oracle.f32_to_bf16_bits(rng.standard_normal((1, M, 8, 64)).astype(np.float32)).reshape(1, M, 8, 64)
    base = oracle.attention_multi(p, q, T)
    p.v_codes[:, :, T - 1] ^= 0x5A   # the newest row, visible to query M-1 only
    p.k_codes[:, :, T - 1] ^= 0x33
    moved = oracle.attention_multi(p, q, T)
    assert np.array_equal(moved[:, :M - 1], base[:, :M - 1])
    assert not np.array_equal(moved[:, M - 1], base[:, M - 1])


def test_multi_token_first_query_sees_its_own_row():
    """With one visible key the output is that row's value (closed form, T = 1)."""
    p, rng = _mt_planes(23)
    M = 3
    q = oracle.f32_to_bf16_bits(rng.standard_normal((1, M, 8, 64)).astype(np.float32)).reshape(1, M, 8, 64)
    out = oracle.attention_multi(p, q, M)          # query 0 sees row 0 only
    _, v = oracle.decode(p, 0, 1)
    for qh in range(8):
        assert np.allclose(out[0, 0, qh], v[0, qh // 4, 0], rtol=0, atol=1e-6)
