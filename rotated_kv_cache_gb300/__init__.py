"""GB300-native TurboQuant rotated KV-cache codec: thin Python binding.

Every function here marshals torch tensors into the C ABI declared in
``include/tq.h`` (library ``_build/libtq.so``, built by ``build.py``) and
calls the entry point of the same name.  All arithmetic runs in the CUDA
kernels; there is no fallback path.  If the library or a CUDA device is
missing, the calls raise.

Cache planes are ordinary torch tensors owned by :class:`Cache`; the library
itself never allocates.
"""
from __future__ import annotations

import ctypes
import os
from functools import lru_cache

import torch

from . import build as _build

__all__ = [
    "Cache", "TQError", "lib", "tq_bytes_per_token_head", "tq_sign_vector", "tq_codebook",
    "tq_encode_append", "tq_decode", "tq_attention_workspace_bytes", "tq_decode_attention",
    "tq_attention_supported", "tq_device_error", "tq_plane_bytes", "tq_decode_attention_noalloc",
    "tq_decode_values_rotated", "tq_unrotate", "tq_cache_copy_rows", "tq_cache_clear_rows",
    "tq_multi_token_workspace_bytes", "tq_multi_token_attention", "tq_check_wait_timeout",
    "TQ_DEVICE_ERR_WAIT_TIMEOUT", "TQ_DEFAULT_SIGN_SEED",
]

HEAD_DIMS = (64, 128, 256, 512)
K_BITS = (2, 4, 5, 8)
V_BITS = (2, 3, 4, 5, 8)
TQ_BF16, TQ_F32 = 0, 1
TQ_DEVICE_ERR_WAIT_TIMEOUT = 1  # device error word: a bounded wait gave up
TQ_DEFAULT_SIGN_SEED = 42  # the codec's sign-vector seed unless a cache states another

EXPORTS = (
    "tq_status_string", "tq_bytes_per_token_head", "tq_plane_bytes", "tq_sign_vector", "tq_codebook",
    "tq_encode_append", "tq_decode", "tq_attention_workspace_bytes", "tq_decode_attention",
    "tq_attention_supported", "tq_device_error", "tq_decode_attention_noalloc", "tq_decode_values_rotated",
    "tq_unrotate", "tq_cache_copy_rows", "tq_cache_clear_rows", "tq_multi_token_workspace_bytes",
    "tq_multi_token_attention", "tq_check_wait_timeout",
)


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().tq_status_string(status).decode()} (status {status})")


class _CacheStruct(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32), ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("batch", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("capacity", ctypes.c_int64),
        ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("k_zero", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("sign_seed", ctypes.c_uint64),
    ]


_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_CP = ctypes.POINTER(_CacheStruct)


def library_path() -> str:
    return _build.LIB


@lru_cache(maxsize=1)
def lib() -> ctypes.CDLL:
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run rotated_kv_cache_gb300/build.py)")
    so = ctypes.CDLL(path)
    so.tq_status_string.restype = ctypes.c_char_p
    so.tq_status_string.argtypes = [ctypes.c_int]
    so.tq_bytes_per_token_head.restype = _SZ
    so.tq_bytes_per_token_head.argtypes = [_I32, _I32, _I32]
    so.tq_plane_bytes.argtypes = [_CP, ctypes.POINTER(_SZ)]
    so.tq_sign_vector.argtypes = [_I32, ctypes.c_uint64, _P]
    so.tq_codebook.argtypes = [_I32, _P, _P]
    so.tq_encode_append.argtypes = [_CP, _P, ctypes.POINTER(_I64), _P, ctypes.POINTER(_I64), _I64, _I64, _P]
    so.tq_decode.argtypes = [_CP, _I64, _I64, ctypes.c_int, _P, _P, _P]
    so.tq_attention_workspace_bytes.restype = _SZ
    so.tq_attention_workspace_bytes.argtypes = [_CP, _I32, _I64]
    so.tq_decode_attention.argtypes = [_CP, _P, _I32, _I64, ctypes.c_float, _P, _P, _SZ, _P]
    so.tq_attention_supported.argtypes = [_I32, _I32, _I32, _I32]
    so.tq_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    so.tq_check_wait_timeout.argtypes = [_P]
    so.tq_decode_attention_noalloc.argtypes = [_CP, _P, _I32, _I64, ctypes.c_float, _P, _P]
    so.tq_decode_values_rotated.argtypes = [_CP, _I64, _I64, ctypes.c_int, _P, _P]
    so.tq_unrotate.argtypes = [_I32, ctypes.c_uint64, ctypes.c_int, _P, _I64, ctypes.c_int, _P, _P]
    so.tq_cache_copy_rows.argtypes = [_CP, _I64, _CP, _I64, _I64, _P]
    so.tq_cache_clear_rows.argtypes = [_CP, _I64, _I64, _P]
    so.tq_multi_token_workspace_bytes.restype = _SZ
    so.tq_multi_token_workspace_bytes.argtypes = [_CP, _I32, _I64, _I64]
    so.tq_multi_token_attention.argtypes = [_CP, _P, _I32, _I64, _I64, ctypes.c_float, _P, _P, _SZ, _P]
    for name in EXPORTS:
        if name not in ("tq_status_string", "tq_bytes_per_token_head", "tq_attention_workspace_bytes",
                        "tq_attention_supported", "tq_multi_token_workspace_bytes"):
            getattr(so, name).restype = ctypes.c_int
    so.tq_attention_supported.restype = ctypes.c_int
    return so


def _check(status: int, what: str) -> None:
    if status != 0:
        raise TQError(status, what)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


class Cache:
    """The five packed planes of one KV cache, [batch][H][capacity][row] each.

    capacity is rounded up to a multiple of 16 (the library's row alignment).
    sign_seed picks the value sign vector (tq_sign_vector); every call on the
    cache uses it.
    """

    def __init__(self, batch: int, num_kv_heads: int, head_dim: int, capacity: int, k_bits: int = 8,
                 v_bits: int = 3, device="cuda", sign_seed: int = TQ_DEFAULT_SIGN_SEED):
        cap = (int(capacity) + 15) // 16 * 16
        g = head_dim // 32
        self.batch, self.num_kv_heads, self.head_dim = int(batch), int(num_kv_heads), int(head_dim)
        self.k_bits, self.v_bits, self.capacity = int(k_bits), int(v_bits), cap
        self.sign_seed = int(sign_seed)
        shape = (self.batch, self.num_kv_heads, cap)
        kw = dict(device=device)
        self.k_codes = torch.zeros(*shape, head_dim * k_bits // 8, dtype=torch.uint8, **kw)
        self.k_scale = torch.zeros(*shape, g, dtype=torch.int16, **kw)
        self.k_zero = torch.zeros(*shape, g, dtype=torch.int16, **kw)
        self.v_codes = torch.zeros(*shape, head_dim * v_bits // 8, dtype=torch.uint8, **kw)
        self.v_scale = torch.zeros(*shape, g, dtype=torch.int16, **kw)

    def planes(self):
        return self.k_codes, self.k_scale, self.k_zero, self.v_codes, self.v_scale

    def struct(self) -> _CacheStruct:
        return _CacheStruct(self.head_dim, self.k_bits, self.v_bits, self.num_kv_heads, self.batch, 0,
                            self.capacity, *[t.data_ptr() for t in self.planes()], self.sign_seed)

    def batch_slice(self, b0: int, nb: int) -> "Cache":
        """A view of sequences [b0, b0+nb) sharing this cache's storage."""
        v = Cache.__new__(Cache)
        v.__dict__.update(self.__dict__)
        for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale"):
            setattr(v, name, getattr(self, name)[b0:b0 + nb])
        v.batch = int(nb)
        return v

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.planes())


# ------------------------------------------------------------------ host-side queries
def tq_bytes_per_token_head(head_dim: int, k_bits: int, v_bits: int) -> int:
    return int(lib().tq_bytes_per_token_head(head_dim, k_bits, v_bits))


def tq_plane_bytes(cache: Cache) -> list:
    out = (_SZ * 5)()
    s = cache.struct()
    _check(lib().tq_plane_bytes(ctypes.byref(s), out), "tq_plane_bytes")
    return list(out)


def tq_sign_vector(head_dim: int, seed: int = TQ_DEFAULT_SIGN_SEED):
    import numpy as np

    out = np.zeros(head_dim, dtype=np.int8)
    _check(lib().tq_sign_vector(head_dim, int(seed), out.ctypes.data), "tq_sign_vector")
    return out


def tq_codebook(v_bits: int):
    import numpy as np

    c = np.zeros(1 << v_bits, dtype=np.float32)
    b = np.zeros((1 << v_bits) - 1, dtype=np.float32)
    _check(lib().tq_codebook(v_bits, c.ctypes.data, b.ctypes.data), "tq_codebook")
    return c, b


def tq_attention_supported(head_dim: int, k_bits: int, v_bits: int, group: int) -> bool:
    return bool(lib().tq_attention_supported(head_dim, k_bits, v_bits, group))


# ------------------------------------------------------------------ device work
def _strides3(x: torch.Tensor):
    if x.dim() != 4 or x.stride(3) != 1:
        raise ValueError("K/V must be [batch][heads][tokens][head_dim] with head_dim contiguous")
    return (_I64 * 3)(x.stride(0), x.stride(1), x.stride(2))


def tq_encode_append(cache: Cache, k: torch.Tensor, v: torch.Tensor, t0: int, stream=None) -> None:
    """Quantise K, V (bf16 [B][H][n][d], any strides with d contiguous) into rows [t0, t0+n)."""
    _require_cuda(k, v)
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("K and V must be bfloat16")
    if k.shape != v.shape or k.shape[0] != cache.batch or k.shape[1] != cache.num_kv_heads or \
            k.shape[3] != cache.head_dim:
        raise ValueError(f"K/V shape {tuple(k.shape)} does not match the cache")
    s = cache.struct()
    _check(lib().tq_encode_append(ctypes.byref(s), k.data_ptr(), _strides3(k), v.data_ptr(), _strides3(v),
                                  int(t0), int(k.shape[2]), _stream(stream)), "tq_encode_append")


def tq_decode(cache: Cache, t0: int, n: int, dtype=torch.bfloat16, want_k: bool = True, want_v: bool = True,
              k_out: torch.Tensor | None = None, v_out: torch.Tensor | None = None, stream=None):
    """Dequantise rows [t0, t0+n) -> (K, V) as [B][H][n][d] of `dtype` (bf16 or fp32)."""
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dtype must be bfloat16 or float32")
    dev = cache.k_codes.device
    shape = (cache.batch, cache.num_kv_heads, int(n), cache.head_dim)
    if want_k and k_out is None:
        k_out = torch.empty(shape, dtype=dtype, device=dev)
    if want_v and v_out is None:
        v_out = torch.empty(shape, dtype=dtype, device=dev)
    for t in (k_out, v_out):
        if t is not None and (t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous()):
            raise ValueError("decode outputs must be contiguous [B][H][n][d] of the requested dtype")
    s = cache.struct()
    _check(lib().tq_decode(ctypes.byref(s), int(t0), int(n), TQ_F32 if dtype == torch.float32 else TQ_BF16,
                           k_out.data_ptr() if want_k else None, v_out.data_ptr() if want_v else None,
                           _stream(stream)), "tq_decode")
    return (k_out if want_k else None), (v_out if want_v else None)


def _dtype_code(dtype) -> int:
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dtype must be bfloat16 or float32")
    return TQ_F32 if dtype == torch.float32 else TQ_BF16


def tq_decode_values_rotated(cache: Cache, t0: int, n: int, dtype=torch.float32, out: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """Value rows [t0, t0+n) in the rotated domain (centroid[code] * rms) as [B][H][n][d]."""
    shape = (cache.batch, cache.num_kv_heads, int(n), cache.head_dim)
    if out is None:
        out = torch.empty(shape, dtype=dtype, device=cache.k_codes.device)
    if out.dtype != dtype or tuple(out.shape) != shape or not out.is_contiguous():
        raise ValueError("output must be contiguous [B][H][n][d] of the requested dtype")
    s = cache.struct()
    _check(lib().tq_decode_values_rotated(ctypes.byref(s), int(t0), int(n), _dtype_code(dtype), out.data_ptr(),
                                          _stream(stream)), "tq_decode_values_rotated")
    return out


def tq_unrotate(x: torch.Tensor, out: torch.Tensor | None = None, dtype=None, stream=None,
                sign_seed: int = TQ_DEFAULT_SIGN_SEED) -> torch.Tensor:
    """signs * FWHT(x)/sqrt(d) for every row of x ([..., d] contiguous, fp32 or bf16);
    signs = tq_sign_vector(d, sign_seed), the seed of the cache the rows came from."""
    _require_cuda(x)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    dtype = x.dtype if dtype is None else dtype
    if out is None:
        out = torch.empty(x.shape, dtype=dtype, device=x.device)
    if out.dtype != dtype or out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be contiguous, shaped like x, of the requested dtype")
    d = x.shape[-1]
    _check(lib().tq_unrotate(int(d), int(sign_seed), _dtype_code(x.dtype), x.data_ptr(), int(x.numel() // d),
                             _dtype_code(dtype), out.data_ptr(), _stream(stream)), "tq_unrotate")
    return out


def tq_cache_copy_rows(dst: Cache, dst_t0: int, src: Cache, src_t0: int, n: int, stream=None) -> None:
    """Token rows [src_t0, src_t0+n) of every (sequence, kv-head) of src -> rows [dst_t0, ...) of dst, byte for byte."""
    a, b = dst.struct(), src.struct()
    _check(lib().tq_cache_copy_rows(ctypes.byref(a), int(dst_t0), ctypes.byref(b), int(src_t0), int(n),
                                    _stream(stream)), "tq_cache_copy_rows")


def tq_cache_clear_rows(cache: Cache, t0: int, n: int, stream=None) -> None:
    """Zero token rows [t0, t0+n) of every (sequence, kv-head), all planes (trim)."""
    s = cache.struct()
    _check(lib().tq_cache_clear_rows(ctypes.byref(s), int(t0), int(n), _stream(stream)), "tq_cache_clear_rows")


def tq_attention_workspace_bytes(cache: Cache, q_heads: int, seq_len: int) -> int:
    s = cache.struct()
    return int(lib().tq_attention_workspace_bytes(ctypes.byref(s), int(q_heads), int(seq_len)))


def tq_decode_attention(cache: Cache, q: torch.Tensor, seq_len: int, softmax_scale: float | None = None,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """softmax(q k_hat^T * scale) v_hat over rows [0, seq_len); q bf16 [B][QH][d] -> fp32 [B][QH][d]."""
    _require_cuda(q)
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous bfloat16 [batch][q_heads][head_dim]")
    B, QH, d = q.shape
    if B != cache.batch or d != cache.head_dim:
        raise ValueError("q does not match the cache")
    if out is None:
        out = torch.empty((B, QH, d), dtype=torch.float32, device=q.device)
    need = tq_attention_workspace_bytes(cache, QH, seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    s = cache.struct()
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().tq_decode_attention(ctypes.byref(s), q.data_ptr(), int(QH), int(seq_len), scale,
                                     out.data_ptr(), ws_ptr, ws_bytes, _stream(stream)), "tq_decode_attention")
    return out


def tq_decode_attention_noalloc(cache: Cache, q: torch.Tensor, seq_len: int, softmax_scale: float | None = None,
                                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """tq_decode_attention without a workspace: for callers that cannot allocate
    device memory.  The library's built-in 16 MiB scratch holds the partials;
    concurrent calls race on it (see include/tq.h)."""
    _require_cuda(q)
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous bfloat16 [batch][q_heads][head_dim]")
    B, QH, d = q.shape
    if out is None:
        out = torch.empty((B, QH, d), dtype=torch.float32, device=q.device)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    s = cache.struct()
    _check(lib().tq_decode_attention_noalloc(ctypes.byref(s), q.data_ptr(), int(QH), int(seq_len), scale,
                                             out.data_ptr(), _stream(stream)), "tq_decode_attention_noalloc")
    return out


def tq_multi_token_workspace_bytes(cache: Cache, q_heads: int, m_queries: int, seq_len: int) -> int:
    s = cache.struct()
    return int(lib().tq_multi_token_workspace_bytes(ctypes.byref(s), int(q_heads), int(m_queries), int(seq_len)))


def tq_multi_token_attention(cache: Cache, q: torch.Tensor, seq_len: int, softmax_scale: float | None = None,
                             out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """Causal attention of M query rows per sequence over cache rows [0, seq_len):
    q bf16 [B][M][QH][d] -> fp32 [B][M][QH][d]; row i sees rows [0, seq_len - M + i]."""
    _require_cuda(q)
    if q.dtype != torch.bfloat16 or q.dim() != 4 or not q.is_contiguous():
        raise ValueError("q must be contiguous bfloat16 [batch][m_queries][q_heads][head_dim]")
    B, M, QH, d = q.shape
    if B != cache.batch or d != cache.head_dim:
        raise ValueError("q does not match the cache")
    if out is None:
        out = torch.empty((B, M, QH, d), dtype=torch.float32, device=q.device)
    need = tq_multi_token_workspace_bytes(cache, QH, M, seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    s = cache.struct()
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().tq_multi_token_attention(ctypes.byref(s), q.data_ptr(), int(QH), int(M), int(seq_len), scale,
                                          out.data_ptr(), ws_ptr, ws_bytes, _stream(stream)),
           "tq_multi_token_attention")
    return out


def tq_check_wait_timeout(stream=None) -> None:
    """Enqueue the failure-path check: one warp whose bounded wait on a barrier
    nothing completes gives up after ~2 s and records TQ_DEVICE_ERR_WAIT_TIMEOUT
    (read it with tq_device_error())."""
    _check(lib().tq_check_wait_timeout(_stream(stream)), "tq_check_wait_timeout")


def tq_device_error() -> int:
    """Synchronise, return and clear the device error word (0 = no bounded wait gave up)."""
    code = ctypes.c_uint32(0)
    _check(lib().tq_device_error(ctypes.byref(code)), "tq_device_error")
    return int(code.value)
