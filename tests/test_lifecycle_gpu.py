"""Deferred fetch (rotated-domain values, un-rotation) and cache row copy /
clear against the CPU oracle.

Rotated values are one fp32 multiply per element and the un-rotation runs
the definition's butterfly order, so both are compared bit for bit; copies
and clears are byte work, compared byte for byte.  The deferred attention
check (an attention formed outside the library on rotated values, then
un-rotated) uses the attention tests' 2e-3 max-abs tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import bf16_rne, planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu


def _cache(tq, B, H, d, T, kb, vb, cap=None, seed_w="sweep", t0=0):
    w = tq_synth.WORKLOADS[seed_w]
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T)
    cache = tq.Cache(B, H, d, cap or T, k_bits=kb, v_bits=vb)
    for t in cache.planes():
        t.fill_(0x5B if t.element_size() == 1 else 0x5B5B)
    tq.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), t0)
    return cache, k, v


@pytest.mark.parametrize("d,vb", [(64, 2), (128, 3), (128, 4), (256, 5), (512, 8), (128, 8)])
def test_rotated_fetch_bitexact(cuda, d, vb):
    cache, _, _ = _cache(cuda, 2, 3, d, 45, 8, vb, cap=64)
    planes = planes_from_device(cache)
    for t0, n in ((0, 45), (7, 20), (44, 1)):
        got = cuda.tq_decode_values_rotated(cache, t0, n, dtype=torch.float32).cpu().numpy()
        want = oracle.decode_rotated(planes, t0, n)
        assert np.array_equal(got, want)
        gb = cuda.tq_decode_values_rotated(cache, t0, n, dtype=torch.bfloat16)
        assert np.array_equal(gb.view(torch.int16).cpu().numpy().view(np.uint16), bf16_rne(want))


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_unrotate_bitexact(cuda, d):
    rng = np.random.default_rng(d)
    x = (rng.standard_normal((37, d)) * rng.uniform(0.01, 100.0, (37, 1))).astype(np.float32)
    xg = torch.from_numpy(x).cuda()
    want = oracle.unrotate(x)
    assert np.array_equal(cuda.tq_unrotate(xg).cpu().numpy(), want)
    # bf16 output is the rounding of the fp32 result; bf16 input is read exactly
    assert np.array_equal(cuda.tq_unrotate(xg, dtype=torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16),
                          bf16_rne(want))
    xb = xg.to(torch.bfloat16)
    want_b = oracle.unrotate(xb.float().cpu().numpy())
    assert np.array_equal(cuda.tq_unrotate(xb, dtype=torch.float32).cpu().numpy(), want_b)
    # in place
    y = xg.clone()
    cuda.tq_unrotate(y, out=y)
    assert np.array_equal(y.cpu().numpy(), want)


def test_unrotate_of_rotated_fetch_is_the_fetch(cuda):
    cache, _, _ = _cache(cuda, 2, 2, 128, 33, 8, 3, cap=48)
    rot = cuda.tq_decode_values_rotated(cache, 0, 33, dtype=torch.float32)
    _, v = cuda.tq_decode(cache, 0, 33, dtype=torch.float32, want_k=False)
    assert torch.equal(cuda.tq_unrotate(rot), v)


def test_deferred_attention_outside_the_library(cuda):
    """softmax(q k^T) v_rot formed in torch on the rotated fetch, then one
    un-rotation per query row, equals the fused attention."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T, G = 2, 2, 300, 8
    cache, _, _ = _cache(cuda, B, H, 128, T, 8, 3, cap=304, seed_w="decode")
    q = to_device_bf16(tq_synth.host_q(w, 0, B=B, QH=G * H))
    k, _ = cuda.tq_decode(cache, 0, T, dtype=torch.float32, want_v=False)
    vr = cuda.tq_decode_values_rotated(cache, 0, T, dtype=torch.float32)
    kq = k.repeat_interleave(G, dim=1).double()
    vq = vr.repeat_interleave(G, dim=1).double()
    s = torch.einsum("bhd,bhtd->bht", q.double(), kq) / 128 ** 0.5
    o_rot = torch.einsum("bht,bhtd->bhd", torch.softmax(s, dim=-1), vq).float().contiguous()
    got = cuda.tq_unrotate(o_rot)
    want = cuda.tq_decode_attention(cache, q, T)
    assert (got - want).abs().max().item() < 2e-3


def test_copy_rows_between_caches_and_growth(cuda):
    src, _, _ = _cache(cuda, 2, 3, 128, 40, 4, 3, cap=48)
    dst = cuda.Cache(2, 3, 128, 96, k_bits=4, v_bits=3)
    for t in dst.planes():
        t.fill_(0x5B if t.element_size() == 1 else 0x5B5B)
    cuda.tq_cache_copy_rows(dst, 33, src, 5, 35)
    a, b = planes_from_device(dst), planes_from_device(src)
    for x, y in zip(a.arrays(), b.arrays()):
        assert np.array_equal(x[:, :, 33:68], y[:, :, 5:40])
        out = np.concatenate([x[:, :, :33].ravel(), x[:, :, 68:].ravel()]).view(np.uint8)
        assert np.all(out == 0x5B)
    # the copy decodes exactly like the source rows
    for u, v in zip(cuda.tq_decode(dst, 33, 35, dtype=torch.float32), cuda.tq_decode(src, 5, 35, dtype=torch.float32)):
        assert torch.equal(u, v)


def test_copy_rows_within_one_cache(cuda):
    cache, _, _ = _cache(cuda, 1, 2, 64, 30, 5, 2, cap=64)   # 5-bit keys: rows of 40 bytes (4-byte words)
    before = planes_from_device(cache)
    cuda.tq_cache_copy_rows(cache, 31, cache, 0, 29)
    after = planes_from_device(cache)
    for x, y in zip(after.arrays(), before.arrays()):
        assert np.array_equal(x[:, :, 31:60], y[:, :, 0:29])
        assert np.array_equal(x[:, :, :31], y[:, :, :31])
    with pytest.raises(cuda.TQError):
        cuda.tq_cache_copy_rows(cache, 10, cache, 0, 20)   # overlapping ranges are refused


def test_trim_then_reappend_equals_fresh_encode(cuda):
    """Trim to 17 rows, append 10 more: the bytes equal a cache that only ever
    held those 27 tokens (same kernels, so byte for byte), and rows past them
    are zero."""
    w = tq_synth.WORKLOADS["prefill"]
    B, H, d = 2, 2, 128
    k, v = tq_synth.host_kv(w, B=B, H=H, n=50)
    cache = cuda.Cache(B, H, d, 64)
    cuda.tq_encode_append(cache, to_device_bf16(k[:, :, :40]), to_device_bf16(v[:, :, :40]), 0)
    cuda.tq_cache_clear_rows(cache, 17, 64 - 17)
    cuda.tq_encode_append(cache, to_device_bf16(k[:, :, 40:50]), to_device_bf16(v[:, :, 40:50]), 17)
    fresh = cuda.Cache(B, H, d, 64)
    for t in fresh.planes():
        t.zero_()
    cuda.tq_encode_append(fresh, to_device_bf16(np.concatenate([k[:, :, :17], k[:, :, 40:50]], axis=2)),
                          to_device_bf16(np.concatenate([v[:, :, :17], v[:, :, 40:50]], axis=2)), 0)
    assert all(torch.equal(a, b) for a, b in zip(cache.planes(), fresh.planes()))


def test_snapshot_restore_full_prefill_cache(cuda):
    """Snapshot a full prefill-size cache (4 x 8 kv-heads x 8192 rows) and restore it."""
    w = tq_synth.WORKLOADS["prefill"]
    B, H, T, d = w.B, w.H, w.T, w.d
    k = torch.empty((B, H, T, d), dtype=torch.int16, device="cuda")
    v = torch.empty_like(k)
    tq_synth.device_kv(w, k, v)
    cache = cuda.Cache(B, H, d, T)
    cuda.tq_encode_append(cache, k.view(torch.bfloat16), v.view(torch.bfloat16), 0)
    snap = cuda.Cache(B, H, d, T)
    cuda.tq_cache_copy_rows(snap, 0, cache, 0, T)
    orig = [t.clone() for t in cache.planes()]
    cuda.tq_cache_clear_rows(cache, 4000, T - 4000)
    cuda.tq_cache_copy_rows(cache, 4000, snap, 4000, T - 4000)
    assert all(torch.equal(a, b) for a, b in zip(cache.planes(), orig))
    assert cuda.tq_device_error() == 0
