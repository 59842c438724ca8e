"""The C-ABI library on the host: symbols, host-side tables, argument refusal.

CPU only: nothing here launches a kernel.  Every refusal below is decided by
the host validation before any CUDA call.
"""
import ctypes
import re

import numpy as np
import pytest

import oracle
from conftest import ROOT


def _declared_functions():
    src = open(f"{ROOT}/include/tq.h").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_function_is_exported(tqlib):
    so = tqlib.lib()
    names = _declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(tqlib.EXPORTS)


def test_bytes_per_token_head_matches_oracle(tqlib):
    for d in tqlib.HEAD_DIMS:
        for kb in tqlib.K_BITS:
            for vb in tqlib.V_BITS:
                assert tqlib.tq_bytes_per_token_head(d, kb, vb) == oracle.bytes_per_token_head(d, kb, vb)
    assert tqlib.tq_bytes_per_token_head(128, 8, 3) == 200
    assert tqlib.tq_bytes_per_token_head(96, 8, 3) == 0
    assert tqlib.tq_bytes_per_token_head(128, 3, 3) == 0


def test_sign_vector_matches_oracle(tqlib):
    for d in tqlib.HEAD_DIMS:
        assert np.array_equal(tqlib.tq_sign_vector(d), oracle.sign_vector(d))
        for seed in (0, 7, 2**64 - 1):
            assert np.array_equal(tqlib.tq_sign_vector(d, seed), oracle.sign_vector(d, seed))
    assert not np.array_equal(tqlib.tq_sign_vector(128, 7), tqlib.tq_sign_vector(128))


@pytest.mark.parametrize("vb", [2, 3, 4, 5, 8])
def test_codebook_bit_identical_to_oracle(tqlib, vb):
    c, b = tqlib.tq_codebook(vb)
    oc, ob = oracle.codebook(vb)
    assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(b.view(np.uint32), ob.view(np.uint32))
    # exact symmetry (the kernels may rely on it)
    assert np.array_equal(c, -c[::-1]) and np.array_equal(b, -b[::-1])


def _struct(tqlib, **kw):
    f = dict(head_dim=128, k_bits=8, v_bits=3, num_kv_heads=2, batch=1, reserved=0, capacity=32,
             k_codes=0x1000, k_scale=0x2000, k_zero=0x3000, v_codes=0x4000, v_scale=0x5000, sign_seed=42)
    f.update(kw)
    return tqlib._CacheStruct(*[f[n] for n, _ in tqlib._CacheStruct._fields_])


def test_plane_bytes(tqlib):
    s = _struct(tqlib, batch=2, num_kv_heads=3, capacity=48)
    out = (ctypes.c_size_t * 5)()
    assert tqlib.lib().tq_plane_bytes(ctypes.byref(s), out) == 0
    rows = 2 * 3 * 48
    assert list(out) == [rows * 128, rows * 8, rows * 8, rows * 48, rows * 8]


def _encode_status(tqlib, s, k=0x10000, v=0x20000, ks=(4096, 2048, 128), vs=(4096, 2048, 128), t0=0, n=4):
    L = tqlib.lib()
    return L.tq_encode_append(ctypes.byref(s) if s is not None else None, k, (ctypes.c_int64 * 3)(*ks), v,
                              (ctypes.c_int64 * 3)(*vs), t0, n, None)


def test_refusals_before_launch(tqlib):
    S = {name: i for i, name in enumerate(
        ["TQ_OK", "TQ_ERR_NULL", "TQ_ERR_HEAD_DIM", "TQ_ERR_BITS", "TQ_ERR_SHAPE", "TQ_ERR_CAPACITY",
         "TQ_ERR_ALIGN", "TQ_ERR_WORKSPACE", "TQ_ERR_CUDA", "TQ_ERR_UNSUPPORTED"])}
    assert _encode_status(tqlib, None) == S["TQ_ERR_NULL"]
    assert _encode_status(tqlib, _struct(tqlib, head_dim=96)) == S["TQ_ERR_HEAD_DIM"]
    assert _encode_status(tqlib, _struct(tqlib, k_bits=3)) == S["TQ_ERR_BITS"]
    assert _encode_status(tqlib, _struct(tqlib, v_bits=6)) == S["TQ_ERR_BITS"]
    assert _encode_status(tqlib, _struct(tqlib, capacity=40)) == S["TQ_ERR_SHAPE"]
    assert _encode_status(tqlib, _struct(tqlib, reserved=1)) == S["TQ_ERR_SHAPE"]
    assert _encode_status(tqlib, _struct(tqlib, batch=0)) == S["TQ_ERR_SHAPE"]
    assert _encode_status(tqlib, _struct(tqlib, v_scale=0)) == S["TQ_ERR_NULL"]
    assert _encode_status(tqlib, _struct(tqlib, k_codes=0x1008)) == S["TQ_ERR_ALIGN"]
    assert _encode_status(tqlib, _struct(tqlib), t0=30, n=4) == S["TQ_ERR_CAPACITY"]
    assert _encode_status(tqlib, _struct(tqlib), t0=-1) == S["TQ_ERR_SHAPE"]
    assert _encode_status(tqlib, _struct(tqlib), k=0x10008) == S["TQ_ERR_ALIGN"]
    assert _encode_status(tqlib, _struct(tqlib), ks=(4096, 2048, 100)) == S["TQ_ERR_ALIGN"]
    assert _encode_status(tqlib, _struct(tqlib), k=0) == S["TQ_ERR_NULL"]
    assert _encode_status(tqlib, _struct(tqlib), n=0) == S["TQ_OK"]  # empty append: no-op
    L = tqlib.lib()
    s = _struct(tqlib)
    assert L.tq_decode(ctypes.byref(s), 0, 40, 0, 0x10000, None, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_decode(ctypes.byref(s), 0, 4, 7, 0x10000, None, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_decode(ctypes.byref(s), 0, 4, 0, 0x10004, None, None) == S["TQ_ERR_ALIGN"]
    # the fetch moves 32-byte words: 16-byte alignment is not enough for its outputs
    assert L.tq_decode(ctypes.byref(s), 0, 4, 0, 0x10010, None, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_decode(ctypes.byref(s), 0, 4, 0, None, 0x10010, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_decode(ctypes.byref(s), 0, 0, 0, 0x10000, None, None) == S["TQ_OK"]
    assert L.tq_decode_attention(ctypes.byref(s), 0x10000, 3, 8, 1.0, 0x20000, None, 0, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_decode_attention(ctypes.byref(s), 0x10000, 4, 33, 1.0, 0x20000, None, 0, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_decode_attention(ctypes.byref(s), None, 4, 8, 1.0, 0x20000, None, 0, None) == S["TQ_ERR_NULL"]
    assert L.tq_attention_workspace_bytes(ctypes.byref(s), 3, 8) == 0
    for st in range(11):
        assert L.tq_status_string(st)


def test_lifecycle_and_deferred_refusals(tqlib):
    """Argument checks of the deferred fetch, un-rotation and row copy/clear
    return before any launch (fake, never-read pointers)."""
    S = {name: i for i, name in enumerate(
        ["TQ_OK", "TQ_ERR_NULL", "TQ_ERR_HEAD_DIM", "TQ_ERR_BITS", "TQ_ERR_SHAPE", "TQ_ERR_CAPACITY",
         "TQ_ERR_ALIGN", "TQ_ERR_WORKSPACE", "TQ_ERR_CUDA", "TQ_ERR_UNSUPPORTED"])}
    L = tqlib.lib()
    a, b = _struct(tqlib), _struct(tqlib)
    c = _struct(tqlib, k_codes=0x11000, k_scale=0x12000, k_zero=0x13000, v_codes=0x14000, v_scale=0x15000)
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 40, 1, 0x10000, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 4, 5, 0x10000, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 4, 1, None, None) == S["TQ_ERR_NULL"]
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 4, 1, 0x10008, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 4, 1, 0x10010, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_decode_values_rotated(ctypes.byref(a), 0, 0, 1, None, None) == S["TQ_OK"]
    assert L.tq_unrotate(96, 42, 1, 0x10000, 4, 1, 0x20000, None) == S["TQ_ERR_HEAD_DIM"]
    assert L.tq_unrotate(128, 42, 2, 0x10000, 4, 1, 0x20000, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_unrotate(128, 42, 1, 0x10000, -1, 1, 0x20000, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_unrotate(128, 42, 1, 0x10000, 4, 0, 0x10000, None) == S["TQ_ERR_SHAPE"]  # in place, different sizes
    assert L.tq_unrotate(128, 42, 1, 0x10004, 4, 1, 0x20000, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_unrotate(128, 42, 1, 0x10010, 4, 1, 0x20000, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_unrotate(128, 42, 1, 0x10000, 4, 1, 0x20010, None) == S["TQ_ERR_ALIGN"]
    assert L.tq_unrotate(128, 42, 1, None, 4, 1, 0x20000, None) == S["TQ_ERR_NULL"]
    assert L.tq_unrotate(128, 42, 1, None, 0, 1, None, None) == S["TQ_OK"]
    big = _struct(tqlib, capacity=64)
    other = _struct(tqlib, head_dim=64)
    assert L.tq_cache_copy_rows(ctypes.byref(c), 0, ctypes.byref(other), 0, 4, None) == S["TQ_ERR_SHAPE"]
    reseeded = _struct(tqlib, sign_seed=7)  # rows of another sign vector cannot be mixed in
    assert L.tq_cache_copy_rows(ctypes.byref(c), 0, ctypes.byref(reseeded), 0, 4, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_cache_copy_rows(ctypes.byref(c), 30, ctypes.byref(b), 0, 4, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_cache_copy_rows(ctypes.byref(c), 0, ctypes.byref(big), 40, 30, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_cache_copy_rows(ctypes.byref(a), 4, ctypes.byref(b), 0, 8, None) == S["TQ_ERR_SHAPE"]  # overlap
    assert L.tq_cache_copy_rows(ctypes.byref(a), 5, ctypes.byref(b), 5, 8, None) == S["TQ_OK"]        # identical
    assert L.tq_cache_copy_rows(ctypes.byref(a), -1, ctypes.byref(b), 0, 8, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_cache_copy_rows(ctypes.byref(c), 0, ctypes.byref(b), 0, 0, None) == S["TQ_OK"]
    assert L.tq_cache_clear_rows(ctypes.byref(a), 30, 4, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_cache_clear_rows(ctypes.byref(a), 3, -1, None) == S["TQ_ERR_SHAPE"]
    assert L.tq_cache_clear_rows(ctypes.byref(a), 3, 0, None) == S["TQ_OK"]


def test_multi_token_refusals(tqlib):
    """Argument checks of the multi-token attention return before any launch."""
    S = {name: i for i, name in enumerate(
        ["TQ_OK", "TQ_ERR_NULL", "TQ_ERR_HEAD_DIM", "TQ_ERR_BITS", "TQ_ERR_SHAPE", "TQ_ERR_CAPACITY",
         "TQ_ERR_ALIGN", "TQ_ERR_WORKSPACE", "TQ_ERR_CUDA", "TQ_ERR_UNSUPPORTED"])}
    L = tqlib.lib()
    s = _struct(tqlib)  # 2 kv-heads, capacity 32
    call = lambda qh, m, T, q=0x10000, out=0x20000: L.tq_multi_token_attention(  # noqa: E731
        ctypes.byref(s), q, qh, m, T, 1.0, out, None, 0, None)
    assert call(3, 2, 8) == S["TQ_ERR_SHAPE"]          # q_heads not a multiple of kv-heads
    assert call(4, 0, 8) == S["TQ_ERR_SHAPE"]          # no query rows
    assert call(4, 9, 8) == S["TQ_ERR_SHAPE"]          # more query rows than cache rows
    assert call(4, 2, 33) == S["TQ_ERR_CAPACITY"]
    assert call(4, 2, 8, q=None) == S["TQ_ERR_NULL"]
    assert call(4, 2, 8, out=0x20008) == S["TQ_ERR_ALIGN"]
    big = _struct(tqlib, capacity=1 << 20)
    assert L.tq_multi_token_attention(ctypes.byref(big), 0x10000, 2 * 4096, 1 << 18, 1 << 18, 1.0, 0x20000, None, 0,
                                      None) == S["TQ_ERR_SHAPE"]  # 2^31 output rows
    assert L.tq_multi_token_workspace_bytes(ctypes.byref(s), 4, 9, 8) == 0
    assert L.tq_multi_token_workspace_bytes(ctypes.byref(s), 3, 2, 8) == 0
