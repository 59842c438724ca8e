"""Shared helpers of the GPU parity tests (conversions and comparisons only)."""
import numpy as np

import oracle


def to_device_bf16(bits: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def planes_from_device(cache) -> "oracle.Planes":
    p = oracle.Planes(cache.batch, cache.num_kv_heads, cache.head_dim, cache.k_bits, cache.v_bits, cache.capacity,
                      sign_seed=cache.sign_seed)
    p.k_codes[...] = cache.k_codes.cpu().numpy()
    p.k_scale[...] = cache.k_scale.cpu().numpy().view(np.uint16)
    p.k_zero[...] = cache.k_zero.cpu().numpy().view(np.uint16)
    p.v_codes[...] = cache.v_codes.cpu().numpy()
    p.v_scale[...] = cache.v_scale.cpu().numpy().view(np.uint16)
    return p


def f16_equal(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Bitwise equality of fp16 bit patterns, any NaN equal to any NaN."""
    a = a.astype(np.uint16)
    b = b.astype(np.uint16)
    nan_a = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
    nan_b = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    return (a == b) | (nan_a & nan_b)


def f16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in fp16 ulps (ordered integer distance); NaN pairs count 0."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - x, x)
    d = np.abs(ordered(a.astype(np.uint16)) - ordered(b.astype(np.uint16)))
    return np.where(f16_equal(a, b), 0, d)


def value_indices(codes_row_bytes: np.ndarray, d: int, vb: int) -> np.ndarray:
    return oracle.unpack_bits(codes_row_bytes, d, vb).astype(np.int64)


def compare_value_codes(gpu: "oracle.Planes", ref: "oracle.Planes", v_bits_f32: np.ndarray, rows, t0: int):
    """Value indices must match exactly except where the oracle's normalised input
    lies within 1e-5 of a boundary.  rows: iterable of (b, h, t) with t relative to
    t0; v_bits_f32: the fp32 value inputs [B][H][n][d].  Returns (mismatches outside
    the exemption, exempt mismatches)."""
    d, vb = ref.d, ref.vb
    bnd = oracle.codebook(vb)[1].astype(np.float64)
    signs = oracle.sign_vector(d, ref.sign_seed)
    bad = exempt = 0
    for (b, h, t) in rows:
        g = gpu.v_codes[b, h, t0 + t]
        r = ref.v_codes[b, h, t0 + t]
        if np.array_equal(g, r):
            continue
        gi, ri = value_indices(g, d, vb), value_indices(r, d, vb)
        _, _, yn = oracle.value_row(v_bits_f32[b, h, t], vb, signs=signs)
        near = np.min(np.abs(yn.astype(np.float64)[:, None] - bnd[None, :]), axis=1) < 1e-5
        diff = gi != ri
        exempt += int(np.sum(diff & near))
        bad += int(np.sum(diff & ~near))
    return bad, exempt


def bf16_rne(x: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)
