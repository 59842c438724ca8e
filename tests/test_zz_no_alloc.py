"""tq_decode_attention_noalloc (decode attention with the library's own fixed
scratch, for callers that cannot allocate device memory) against
tq_decode_attention on the same cache and queries, and against the oracle on
a sampled (sequence, kv-head) pair where the split plan is the reduced one.

Collected last on purpose: the scratch is shared process state, so a run of
the whole suite exercises it after every other test.  Run on its own
(``pytest tests/test_zz_no_alloc.py``) the first call of the file is the
process's first, which covers the scratch address lookup on a fresh context.
Each case makes two calls in a row with different queries, so a second call
that read the first call's partials would show.  Tolerance: the attention
tests' 2e-3 max-abs (both entry points run the same kernels, so the outputs
agree far more closely unless the split count differs).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import to_device_bf16

TOL = 2e-3
SCRATCH_BYTES = 16 << 20


def _noalloc(tq, cache, q, T, scale):
    """One call through the C ABI; returns the fp32 output."""
    B, QH, d = q.shape
    out = torch.full((B, QH, d), float("nan"), dtype=torch.float32, device=q.device)
    s = cache.struct()
    st = tq.lib().tq_decode_attention_noalloc(ctypes.byref(s), q.data_ptr(), QH, T, scale, out.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 0, tq.lib().tq_status_string(st)
    return out


def _two_calls_match(tq, cache, qs, T):
    scale = 1.0 / np.sqrt(qs[0].shape[-1])
    got = [_noalloc(tq, cache, q, T, scale) for q in qs]  # back to back, same scratch
    for q, g in zip(qs, got):
        want = tq.tq_decode_attention(cache, q, T, softmax_scale=scale)
        err = (g - want).abs().max().item()
        assert err < TOL, err
    assert tq.tq_device_error() == 0
    return got


def _oracle_pair(cache, q, T, b, h, G):
    """The oracle's attention for sequence b, kv-head h (its G q-heads), on the
    packed rows read back from the device."""
    p = oracle.Planes(1, 1, cache.head_dim, cache.k_bits, cache.v_bits, cache.capacity, sign_seed=cache.sign_seed)
    for dst, src in zip(p.arrays(), cache.planes()):
        dst[0, 0] = src[b, h].cpu().numpy().view(dst.dtype)
    qb = q[b:b + 1, h * G:(h + 1) * G].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return oracle.attention(p, qb, T)[0]


@pytest.mark.gpu
@pytest.mark.parametrize("kb", [8, 4])
def test_noalloc_small_ragged(cuda, kb):
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 2, 2, 1000
    k, v = tq_synth.host_kv(w, B=B, H=H, n=T)
    cache = cuda.Cache(B, H, w.d, T, k_bits=kb, v_bits=w.vb)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    qs = [to_device_bf16(tq_synth.host_q(w, step, B=B, QH=8 * H)) for step in (0, 1)]
    _two_calls_match(cuda, cache, qs, T)


@pytest.mark.gpu
@pytest.mark.parametrize("d,kb", [(64, 8), (256, 4)])
def test_noalloc_other_head_dims(cuda, d, kb):
    """The specialised kernel's other head_dims (partials merged by the generic
    kernel's merge), against tq_decode_attention and the oracle."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 2, 2, 777
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T)
    cache = cuda.Cache(B, H, d, T + 7, k_bits=kb, v_bits=w.vb)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    qs = [to_device_bf16(tq_synth.host_q(w, step, B=B, QH=8 * H, d=d)) for step in (0, 1)]
    got = _two_calls_match(cuda, cache, qs, T)
    want = _oracle_pair(cache, qs[1], T, 1, 1, 8)
    err = np.abs(got[1][1, 8:16].cpu().numpy().astype(np.float64) - want).max()
    assert err < TOL, err


@pytest.mark.gpu
def test_noalloc_group_of_four(cuda):
    """4 q-heads per kv-head (half the specialised kernel's columns)."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 3, 2, 1500
    k, v = tq_synth.host_kv(w, B=B, H=H, n=T)
    cache = cuda.Cache(B, H, w.d, T, k_bits=8, v_bits=w.vb)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    qs = [to_device_bf16(tq_synth.host_q(w, step, B=B, QH=4 * H)) for step in (0, 1)]
    _two_calls_match(cuda, cache, qs, T)


@pytest.mark.gpu
@pytest.mark.parametrize("d,G", [(128, 16), (64, 12)])
def test_noalloc_two_column_blocks(cuda, d, G):
    """More than 8 q-heads per kv-head at head_dims 64 and 128: each CTA of the
    specialised kernel takes two blocks of 8 columns (at G = 12 the second is
    half padding), against tq_decode_attention and the oracle."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 2, 2, 1234
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T)
    cache = cuda.Cache(B, H, d, T + 14, k_bits=8, v_bits=w.vb)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    qs = [to_device_bf16(tq_synth.host_q(w, step, B=B, QH=G * H, d=d)) for step in (0, 1)]
    got = _two_calls_match(cuda, cache, qs, T)
    want = _oracle_pair(cache, qs[1], T, 1, 1, G)
    err = np.abs(got[1][1, G:2 * G].cpu().numpy().astype(np.float64) - want).max()
    assert err < TOL, err


@pytest.mark.gpu
@pytest.mark.parametrize("kb", [8, 4])
def test_noalloc_fewer_splits_than_usual(cuda, kb):
    """8 kv-heads x 8193 rows and the smallest batch (64 to 512 sequences) whose
    usual split plan needs more than the 16 MiB scratch, so this entry point
    runs with fewer splits; both key widths (their kernels differ in CTAs per
    SM, hence in split plans)."""
    w = tq_synth.WORKLOADS["decode"]
    H, T = 8, 8193

    def usual_workspace(B):  # the size query reads no device memory
        s = cuda._CacheStruct(w.d, kb, w.vb, H, B, 0, T + 15, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 42)
        return cuda.lib().tq_attention_workspace_bytes(ctypes.byref(s), 8 * H, T)

    B = next(b for b in (64, 128, 256, 512) if usual_workspace(b) > SCRATCH_BYTES)
    cache = cuda.Cache(B, H, w.d, T, k_bits=kb, v_bits=w.vb)
    assert cuda.tq_attention_workspace_bytes(cache, 8 * H, T) > SCRATCH_BYTES
    for b0 in range(0, B, 64):
        nb = min(64, B - b0)
        k = torch.empty((nb, H, T, w.d), dtype=torch.int16, device="cuda")
        v = torch.empty_like(k)
        tq_synth.device_kv(w, k, v, B=nb, H=H, n=T, b_offset=b0)
        cuda.tq_encode_append(cache.batch_slice(b0, nb), k.view(torch.bfloat16), v.view(torch.bfloat16), 0)
        del k, v
    qs = []
    for step in (0, 1):
        q = torch.empty((B, 8 * H, w.d), dtype=torch.int16, device="cuda")
        tq_synth.device_q(w, step, q, B=B, QH=8 * H)
        qs.append(q.view(torch.bfloat16))
    got = _two_calls_match(cuda, cache, qs, T)
    b, h = B - 3, 5  # one sampled pair, checked against the oracle for both calls
    for q, g in zip(qs, got):
        want = _oracle_pair(cache, q, T, b, h, 8)
        err = np.abs(g[b, 8 * h:8 * h + 8].cpu().numpy().astype(np.float64) - want).max()
        assert err < TOL, err


def test_noalloc_rejects_problems_beyond_the_scratch(tqlib):
    """batch x kv-heads above 4032 cannot fit even one split: refused before
    any CUDA call (so this runs without a GPU; the pointers are never read)."""
    L = tqlib.lib()
    S = {n: i for i, n in enumerate(["TQ_OK", "TQ_ERR_NULL", "TQ_ERR_HEAD_DIM", "TQ_ERR_BITS", "TQ_ERR_SHAPE",
                                     "TQ_ERR_CAPACITY", "TQ_ERR_ALIGN", "TQ_ERR_WORKSPACE", "TQ_ERR_CUDA",
                                     "TQ_ERR_UNSUPPORTED", "TQ_ERR_SCRATCH"])}
    def status(B, H):
        s = tqlib._CacheStruct(128, 8, 3, H, B, 0, 16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 42)
        return L.tq_decode_attention_noalloc(ctypes.byref(s), 0x10000, 8 * H, 16, 1.0, 0x20000, None)
    assert status(4033, 1) == S["TQ_ERR_SCRATCH"]
    assert status(1, 4033) == S["TQ_ERR_SCRATCH"]
    assert status(37, 109) == S["TQ_ERR_SCRATCH"]  # 4033 units
    assert "16 MiB" in L.tq_status_string(S["TQ_ERR_SCRATCH"]).decode()
    # the usual argument checks still come first
    s = tqlib._CacheStruct(128, 8, 3, 1, 1, 0, 16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 42)
    assert L.tq_decode_attention_noalloc(ctypes.byref(s), 0x10000, 8, 17, 1.0, 0x20000, None) == S["TQ_ERR_CAPACITY"]
    assert L.tq_decode_attention_noalloc(ctypes.byref(s), 0x10000, 8, 16, 1.0, 0x20004, None) == S["TQ_ERR_ALIGN"]
    # value widths other than 2, 3 and 4 bits are outside the specialised kernel
    s2 = tqlib._CacheStruct(128, 8, 5, 1, 1, 0, 16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 42)
    assert L.tq_decode_attention_noalloc(ctypes.byref(s2), 0x10000, 8, 16, 1.0, 0x20000, None) == S["TQ_ERR_UNSUPPORTED"]
    # a group of 16 takes two column blocks: 2016 sequence-heads already overflow
    s3 = tqlib._CacheStruct(128, 8, 3, 1, 2017, 0, 16, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 42)
    assert L.tq_decode_attention_noalloc(ctypes.byref(s3), 0x10000, 16, 16, 1.0, 0x20000, None) == S["TQ_ERR_SCRATCH"]
