"""CPU oracle of the TurboQuant rotated KV-cache codec (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product library never loads it; it shares no code
with the CUDA path.  The arithmetic lives in ``tq_oracle.c`` (plain C, fp32 in
program order, no FMA contraction); this module only marshals numpy arrays.

Every function cites the page passage it follows in ``tq_oracle.c``; the pins
that tie it to the pages and to textbook values are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libtq_oracle.so")

SIGN_SEED = 42  # the sign vector's seed (SplitMix64), fixed like the pages' key(42)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp32 in program order: no contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64


@lru_cache(maxsize=1)
def lib() -> ctypes.CDLL:
    so = ctypes.CDLL(build())
    so.tqo_splitmix64.restype = ctypes.c_uint64
    so.tqo_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    so.tqo_sign_vector.argtypes = [_I, ctypes.c_uint64, _P]
    so.tqo_lloyd_max.argtypes = [_I, _P, _P]
    so.tqo_codebook_f32.argtypes = [_I, _P, _P]
    so.tqo_normal_mse.restype = ctypes.c_double
    so.tqo_normal_mse.argtypes = [_I, _P, _P]
    so.tqo_f32_to_f16.restype = ctypes.c_uint16
    so.tqo_f32_to_f16.argtypes = [ctypes.c_float]
    so.tqo_f16_to_f32.restype = ctypes.c_float
    so.tqo_f16_to_f32.argtypes = [ctypes.c_uint16]
    so.tqo_f32_to_bf16.restype = ctypes.c_uint16
    so.tqo_f32_to_bf16.argtypes = [ctypes.c_float]
    so.tqo_pack_bits.argtypes = [_P, _I, _I, _P]
    so.tqo_unpack_bits.argtypes = [_P, _I, _I, _P]
    so.tqo_fwht.argtypes = [_P, _I]
    so.tqo_key_group.argtypes = [_P, _I, _P, _P, _P]
    so.tqo_key_group_dequant.argtypes = [_P, ctypes.c_uint16, ctypes.c_uint16, _P]
    so.tqo_value_row.argtypes = [_P, _I, _P, _I, _P, _P, _P, _P]
    so.tqo_value_row_dequant.argtypes = [_P, _P, _I, _P, _P, _P]
    so.tqo_value_row_rotated.argtypes = [_P, _P, _I, _P, _P]
    so.tqo_unrotate.argtypes = [_P, _I, _P, _P]
    so.tqo_decode_rotated.argtypes = [_I, _I, _I, _I, _L, _L, _L, _P, _P, _P, _P]
    so.tqo_bytes_per_token_head.restype = _L
    so.tqo_bytes_per_token_head.argtypes = [_I, _I, _I]
    so.tqo_encode.argtypes = [_I, _I, _I, _I, _I, _L, _L, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    so.tqo_decode.argtypes = [_I, _I, _I, _I, _I, _L, _L, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    so.tqo_attention.argtypes = [_I, _I, _I, _I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _P, _I, _L,
                                 ctypes.c_double, _P, _P]
    return so


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


# ---------------------------------------------------------------- formats
def f32_to_f16_bits(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib().tqo_f32_to_f16(float(v)) for v in x], dtype=np.uint16)


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib().tqo_f16_to_f32(int(v)) for v in h], dtype=np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib().tqo_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- tables
def splitmix64(seed: int, i: int) -> int:
    return int(lib().tqo_splitmix64(seed, i))


@lru_cache(maxsize=None)
def _signs(d: int, seed: int) -> bytes:
    out = np.zeros(d, dtype=np.int8)
    lib().tqo_sign_vector(d, seed, _ptr(out))
    return out.tobytes()


def sign_vector(d: int, seed: int = SIGN_SEED) -> np.ndarray:
    return np.frombuffer(_signs(d, seed), dtype=np.int8).copy()


@lru_cache(maxsize=None)
def _lloyd(bits: int):
    n = 1 << bits
    c = np.zeros(n, dtype=np.float64)
    b = np.zeros(max(n - 1, 1), dtype=np.float64)
    steps = lib().tqo_lloyd_max(bits, _ptr(c), _ptr(b))
    if steps < 0:
        raise ValueError(f"bad bit width {bits}")
    return c.tobytes(), b[: n - 1].tobytes()


def lloyd_max(bits: int):
    """(centroids, boundaries) in float64 for N(0,1)."""
    c, b = _lloyd(bits)
    return np.frombuffer(c, dtype=np.float64).copy(), np.frombuffer(b, dtype=np.float64).copy()


def codebook(bits: int):
    """(centroids, boundaries) as the fp32 values the codec uses."""
    n = 1 << bits
    c = np.zeros(n, dtype=np.float32)
    b = np.zeros(max(n - 1, 1), dtype=np.float32)
    if lib().tqo_codebook_f32(bits, _ptr(c), _ptr(b)) != 0:
        raise ValueError(f"bad bit width {bits}")
    return c, b[: n - 1]


def normal_mse(centroids, boundaries) -> float:
    c = np.ascontiguousarray(centroids, dtype=np.float64)
    b = np.ascontiguousarray(boundaries, dtype=np.float64)
    return float(lib().tqo_normal_mse(len(c), _ptr(c), _ptr(b)))


# ---------------------------------------------------------------- primitives
def pack_bits(vals, bits: int) -> np.ndarray:
    v = np.ascontiguousarray(vals, dtype=np.uint32)
    out = np.zeros((len(v) * bits + 7) // 8, dtype=np.uint8)
    lib().tqo_pack_bits(_ptr(v), len(v), bits, _ptr(out))
    return out


def unpack_bits(buf, n: int, bits: int) -> np.ndarray:
    b = np.ascontiguousarray(buf, dtype=np.uint8)
    out = np.zeros(n, dtype=np.uint32)
    lib().tqo_unpack_bits(_ptr(b), n, bits, _ptr(out))
    return out


def fwht(x) -> np.ndarray:
    y = np.array(x, dtype=np.float32, copy=True)
    lib().tqo_fwht(_ptr(y), len(y))
    return y


def key_group(x, bits: int):
    """32 fp32 keys -> (int32 codes, fp16 scale bits, fp16 zero bits)."""
    xx = np.ascontiguousarray(x, dtype=np.float32)
    assert xx.size == 32
    idx = np.zeros(32, dtype=np.int32)
    s = np.zeros(1, dtype=np.uint16)
    z = np.zeros(1, dtype=np.uint16)
    lib().tqo_key_group(_ptr(xx), bits, _ptr(idx), _ptr(s), _ptr(z))
    return idx, int(s[0]), int(z[0])


def key_group_dequant(idx, scale_bits: int, zero_bits: int) -> np.ndarray:
    i = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.zeros(32, dtype=np.float32)
    lib().tqo_key_group_dequant(_ptr(i), scale_bits, zero_bits, _ptr(out))
    return out


def value_row(x, bits: int, signs=None, boundaries=None):
    """d fp32 values -> (int32 codes, fp16 scale bits per group, normalised inputs)."""
    xx = np.ascontiguousarray(x, dtype=np.float32)
    d = xx.size
    s = sign_vector(d) if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    b = codebook(bits)[1] if boundaries is None else np.ascontiguousarray(boundaries, dtype=np.float32)
    idx = np.zeros(d, dtype=np.int32)
    sc = np.zeros(d // 32, dtype=np.uint16)
    yn = np.zeros(d, dtype=np.float32)
    lib().tqo_value_row(_ptr(xx), d, _ptr(s), bits, _ptr(b), _ptr(idx), _ptr(sc), _ptr(yn))
    return idx, sc, yn


def value_row_dequant(idx, scale_bits, bits: int, signs=None, centroids=None) -> np.ndarray:
    i = np.ascontiguousarray(idx, dtype=np.int32)
    d = i.size
    sc = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    s = sign_vector(d) if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    c = codebook(bits)[0] if centroids is None else np.ascontiguousarray(centroids, dtype=np.float32)
    out = np.zeros(d, dtype=np.float32)
    lib().tqo_value_row_dequant(_ptr(i), _ptr(sc), d, _ptr(s), _ptr(c), _ptr(out))
    return out


def value_row_rotated(idx, scale_bits, bits: int, centroids=None) -> np.ndarray:
    """centroid[idx] * rms: a value row before the inverse transform (deferred fetch)."""
    i = np.ascontiguousarray(idx, dtype=np.int32)
    sc = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    c = codebook(bits)[0] if centroids is None else np.ascontiguousarray(centroids, dtype=np.float32)
    out = np.zeros(i.size, dtype=np.float32)
    lib().tqo_value_row_rotated(_ptr(i), _ptr(sc), i.size, _ptr(c), _ptr(out))
    return out


def unrotate(x, signs=None) -> np.ndarray:
    """signs * FWHT(x)/sqrt(d) for each row of x ([..., d], fp32)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    d = a.shape[-1]
    s = sign_vector(d) if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    rows = a.reshape(-1, d)
    out = np.zeros_like(rows)
    for r in range(rows.shape[0]):
        lib().tqo_unrotate(_ptr(rows[r]), d, _ptr(s), _ptr(out[r]))
    return out.reshape(a.shape)


def bytes_per_token_head(d: int, kb: int, vb: int) -> int:
    return int(lib().tqo_bytes_per_token_head(d, kb, vb))


# ---------------------------------------------------------------- whole cache
class Planes:
    """Host copy of the five cache planes, [B][H][cap][...] each."""

    def __init__(self, B, H, d, kb, vb, cap, sign_seed=SIGN_SEED):
        g = d // 32
        self.B, self.H, self.d, self.kb, self.vb, self.cap = B, H, d, kb, vb, cap
        self.sign_seed = sign_seed  # the cache's sign vector: sign_vector(d, sign_seed)
        self.k_codes = np.zeros((B, H, cap, d * kb // 8), dtype=np.uint8)
        self.k_scale = np.zeros((B, H, cap, g), dtype=np.uint16)
        self.k_zero = np.zeros((B, H, cap, g), dtype=np.uint16)
        self.v_codes = np.zeros((B, H, cap, d * vb // 8), dtype=np.uint8)
        self.v_scale = np.zeros((B, H, cap, g), dtype=np.uint16)

    def arrays(self):
        return self.k_codes, self.k_scale, self.k_zero, self.v_codes, self.v_scale


def encode(planes: Planes, k_bf16: np.ndarray, v_bf16: np.ndarray, t0: int = 0) -> Planes:
    """Encode bf16 bits [B][H][n][d] into rows [t0, t0+n) of `planes`."""
    p = planes
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
    n = k.shape[2]
    signs = sign_vector(p.d, p.sign_seed)
    bnd = codebook(p.vb)[1]
    rc = lib().tqo_encode(p.B, p.H, p.d, p.kb, p.vb, p.cap, t0, n, _ptr(k), _ptr(v), _ptr(signs),
                          _ptr(bnd), *[_ptr(a) for a in p.arrays()])
    if rc != 0:
        raise ValueError("oracle encode: bad arguments")
    return p


def decode(planes: Planes, t0: int, n: int, want_k: bool = True, want_v: bool = True):
    """Rows [t0, t0+n) -> fp32 K, V [B][H][n][d] (None where not wanted)."""
    p = planes
    ko = np.zeros((p.B, p.H, n, p.d), dtype=np.float32) if want_k else None
    vo = np.zeros((p.B, p.H, n, p.d), dtype=np.float32) if want_v else None
    signs = sign_vector(p.d, p.sign_seed)
    cen = codebook(p.vb)[0]
    rc = lib().tqo_decode(p.B, p.H, p.d, p.kb, p.vb, p.cap, t0, n, *[_ptr(a) for a in p.arrays()],
                          _ptr(signs), _ptr(cen), _ptr(ko), _ptr(vo))
    if rc != 0:
        raise ValueError("oracle decode: bad arguments")
    return ko, vo


def decode_rotated(planes: Planes, t0: int, n: int) -> np.ndarray:
    """Value rows [t0, t0+n) in the rotated domain, fp32 [B][H][n][d]."""
    p = planes
    vo = np.zeros((p.B, p.H, n, p.d), dtype=np.float32)
    cen = codebook(p.vb)[0]  # held for the duration of the call
    rc = lib().tqo_decode_rotated(p.B, p.H, p.d, p.vb, p.cap, t0, n, _ptr(p.v_codes), _ptr(p.v_scale), _ptr(cen),
                                  _ptr(vo))
    if rc != 0:
        raise ValueError("oracle decode_rotated: bad arguments")
    return vo


def copy_rows(dst: Planes, dst_t0: int, src: Planes, src_t0: int, n: int) -> None:
    """Token rows of every plane, byte for byte (token slices are byte-safe:
    quantisation groups run along head_dim only)."""
    for a, b in zip(dst.arrays(), src.arrays()):
        a[:, :, dst_t0:dst_t0 + n] = b[:, :, src_t0:src_t0 + n]


def clear_rows(planes: Planes, t0: int, n: int) -> None:
    for a in planes.arrays():
        a[:, :, t0:t0 + n] = 0


def attention(planes: Planes, q_bf16: np.ndarray, seq_len: int, softmax_scale: float | None = None,
              want: np.ndarray | None = None) -> np.ndarray:
    """softmax(q k_hat^T * scale) v_hat over tokens [0, seq_len); q bf16 bits [B][QH][d].
    Returns float64 [B][QH][d]; rows with want == 0 are left at zero."""
    p = planes
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    QH = q.shape[1]
    scale = 1.0 / np.sqrt(p.d) if softmax_scale is None else float(softmax_scale)
    out = np.zeros((p.B, QH, p.d), dtype=np.float64)
    w = None if want is None else np.ascontiguousarray(want, dtype=np.uint8)
    signs = sign_vector(p.d, p.sign_seed)
    cen = codebook(p.vb)[0]
    rc = lib().tqo_attention(p.B, p.H, p.d, p.kb, p.vb, p.cap, *[_ptr(a) for a in p.arrays()],
                             _ptr(signs), _ptr(cen), _ptr(q), QH, seq_len, scale, _ptr(w), _ptr(out))
    if rc != 0:
        raise ValueError("oracle attention: bad arguments")
    return out



def attention_multi(planes: Planes, q_bf16: np.ndarray, seq_len: int, softmax_scale: float | None = None) -> np.ndarray:
    """M query rows per sequence: q bf16 bits [B][M][QH][d], the M newest cache
    rows being the queries' own.  Query i attends causally to rows
    [0, seq_len - M + i] -- the plain attention of each query over its visible
    prefix (the page's multi-token forward shapes).  Returns float64 [B][M][QH][d]."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    M = q.shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    for i in range(M):
        out[:, i] = attention(planes, np.ascontiguousarray(q[:, i]), seq_len - M + i + 1, softmax_scale)
    return out
