"""Fused dequantise-on-fetch GQA decode attention against the CPU oracle.

The oracle computes softmax(q k_hat^T / sqrt(d)) v_hat in binary64 over its own
encoding of the same inputs (after checking that the GPU's packed cache equals
that encoding byte for byte).  Tolerance: 2e-3 max-abs on the fp32 output.
"""
import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import compare_value_codes, f16_equal, planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _cache_and_oracle(tq, w, B, H, T, kb, cap=None, QH=None, step=0):
    k, v = tq_synth.host_kv(w, B=B, H=H, n=T)
    cache = tq.Cache(B, H, w.d, cap or T, k_bits=kb, v_bits=w.vb)
    tq.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    ref = oracle.Planes(B, H, w.d, kb, w.vb, cache.capacity)
    oracle.encode(ref, k, v)
    QH = QH or 8 * H
    q = tq_synth.host_q(w, step, B=B, QH=QH)
    return cache, ref, q


@pytest.mark.parametrize("kb", [8, 4])
@pytest.mark.parametrize("T", [1, 15, 64, 65, 200, 1000, 4133])
def test_attention_small_ragged(cuda, kb, T):
    w = tq_synth.WORKLOADS["decode"]
    B, H = 2, 2
    cache, ref, q = _cache_and_oracle(cuda, w, B, H, T, kb)
    gpu = planes_from_device(cache)
    assert np.array_equal(gpu.k_codes[:, :, :T], ref.k_codes[:, :, :T])
    out = cuda.tq_decode_attention(cache, to_device_bf16(q), T)
    want = oracle.attention(ref, q, T)
    err = np.abs(out.cpu().numpy().astype(np.float64) - want).max()
    assert err < TOL, err


def test_attention_decode_step_flow(cuda):
    """Per step: append the new token (n = 1), then attend over all rows."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T0 = 3, 1, 300
    k, v = tq_synth.host_kv(w, B=B, H=H, n=T0 + 3)
    cache = cuda.Cache(B, H, w.d, T0 + 16)
    cuda.tq_encode_append(cache, to_device_bf16(k[:, :, :T0]), to_device_bf16(v[:, :, :T0]), 0)
    ref = oracle.Planes(B, H, w.d, 8, 3, cache.capacity)
    for s in range(3):
        t = T0 + s
        cuda.tq_encode_append(cache, to_device_bf16(k[:, :, t:t + 1]), to_device_bf16(v[:, :, t:t + 1]), t)
        oracle.encode(ref, k[:, :, :t + 1], v[:, :, :t + 1])
        q = tq_synth.host_q(w, s, B=B, QH=8 * H)
        out = cuda.tq_decode_attention(cache, to_device_bf16(q), t + 1)
        want = oracle.attention(ref, q, t + 1)
        assert np.abs(out.cpu().numpy() - want).max() < TOL


def test_attention_softmax_scale_and_large_q(cuda):
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 1, 2, 333
    cache, ref, q = _cache_and_oracle(cuda, w, B, H, T, 8)
    qf = oracle.bf16_bits_to_f32(q) * np.float32(3000.0)  # beyond fp16's comfortable range
    qb = oracle.f32_to_bf16_bits(qf).reshape(q.shape)
    for scale in (0.5 / np.sqrt(128), 1e-4):
        out = cuda.tq_decode_attention(cache, to_device_bf16(qb), T, softmax_scale=float(scale))
        want = oracle.attention(ref, qb, T, softmax_scale=float(scale))
        assert np.abs(out.cpu().numpy() - want).max() < TOL


def test_attention_nan_key_group_propagates(cuda):
    """A constant key group dequantises to NaN (the reference defect the pages keep);
    the output of the heads reading it is NaN on both sides."""
    B, H, T, d = 1, 1, 40, 128
    rng = np.random.default_rng(3)
    kx = rng.standard_normal((B, H, T, d)).astype(np.float32)
    kx[0, 0, 17, :32] = 1.25
    k = oracle.f32_to_bf16_bits(kx).reshape(kx.shape)
    v = oracle.f32_to_bf16_bits(rng.standard_normal((B, H, T, d)).astype(np.float32)).reshape(kx.shape)
    cache = cuda.Cache(B, H, d, T)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    ref = oracle.Planes(B, H, d, 8, 3, cache.capacity)
    oracle.encode(ref, k, v)
    q = oracle.f32_to_bf16_bits(rng.standard_normal((B, 8, d)).astype(np.float32)).reshape(B, 8, d)
    out = cuda.tq_decode_attention(cache, to_device_bf16(q), T).cpu().numpy()
    want = oracle.attention(ref, q, T)
    assert np.array_equal(np.isnan(out), np.isnan(want)) and np.isnan(want).all()


def test_attention_refusals(cuda):
    w = tq_synth.WORKLOADS["decode"]
    cache = cuda.Cache(1, 2, 128, 64, k_bits=8, v_bits=3)
    q = torch.zeros((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda.TQError) as e:
        cuda.tq_decode_attention(cache, q, 40, workspace=small)
    assert e.value.status == 7
    # every valid (head_dim, k_bits, v_bits) and group >= 1 is covered; nothing else
    assert all(cuda.tq_attention_supported(d, kb, vb, g) for d in (64, 128, 256, 512) for kb in (2, 4, 5, 8)
               for vb in (2, 3, 4, 5, 8) for g in (1, 8, 16))
    assert not any(cuda.tq_attention_supported(*a) for a in ((96, 8, 3, 8), (128, 3, 3, 8), (128, 8, 6, 8), (128, 8, 3, 0)))


def _full_size_check(tq, w, B, samples, chunk_b=4):
    """Encode the workload on the device in batch chunks, run one decode step
    (append token T, attend over T + 1 rows), and compare sampled (sequence,
    kv-head) pairs with the oracle."""
    H, T, d = w.H, w.T, w.d
    cache = tq.Cache(B, H, d, T + 1, k_bits=w.kb, v_bits=w.vb)
    for b0 in range(0, B, chunk_b):
        nb = min(chunk_b, B - b0)
        kd = torch.empty((nb, H, T + 1, d), dtype=torch.bfloat16, device="cuda")
        vd = torch.empty_like(kd)
        tq_synth.device_kv(w, kd, vd, B=nb, H=H, n=T + 1, b_offset=b0)  # sequences b0 .. b0+nb-1
        view = cache.batch_slice(b0, nb)
        tq.tq_encode_append(view, kd[:, :, :T], vd[:, :, :T], 0)      # the cached context
        tq.tq_encode_append(view, kd[:, :, T:], vd[:, :, T:], T)      # the appended token
        del kd, vd
    q = torch.empty((B, w.QH, d), dtype=torch.bfloat16, device="cuda")
    tq_synth.device_q(w, 0, q, B=B, QH=w.QH, d=d)
    out = tq.tq_decode_attention(cache, q, T + 1)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    qh = q.cpu().view(torch.int16).numpy().view(np.uint16)
    G = w.QH // H
    for (b, h) in samples:
        kd = torch.empty((1, H, T + 1, d), dtype=torch.bfloat16, device="cuda")
        vd = torch.empty_like(kd)
        tq_synth.device_kv(w, kd, vd, B=1, H=H, n=T + 1, b_offset=b)
        k = kd[:, h:h + 1].cpu().view(torch.int16).numpy().view(np.uint16)
        v = vd[:, h:h + 1].cpu().view(torch.int16).numpy().view(np.uint16)
        ref = oracle.Planes(1, 1, d, w.kb, w.vb, cache.capacity)
        oracle.encode(ref, k, v)
        g = oracle.Planes(1, 1, d, w.kb, w.vb, cache.capacity)
        for a, ga, src in zip(ref.arrays(), g.arrays(), cache.planes()):
            got = src[b, h, :T + 1].cpu().numpy().view(a.dtype)
            ga[0, 0, :T + 1] = got
            if a is ref.v_codes:
                continue
            assert (f16_equal(got, a[0, 0, :T + 1]).all() if a.dtype == np.uint16
                    else np.array_equal(got, a[0, 0, :T + 1])), "device cache differs from the oracle encoding"
        rows = [(0, 0, int(t)) for t in np.nonzero(np.any(g.v_codes[0, 0, :T + 1] != ref.v_codes[0, 0, :T + 1],
                                                             axis=-1))[0]]
        bad, exempt = compare_value_codes(g, ref, oracle.bf16_bits_to_f32(v), rows, 0) if rows else (0, 0)
        assert bad == 0 and exempt <= 1e-5 * v.size, (bad, exempt)
        want = oracle.attention(ref, qh[b:b + 1, h * G:(h + 1) * G], T + 1)
        err = np.abs(out[b, h * G:(h + 1) * G] - want[0]).max()
        assert err < TOL, (b, h, err)


@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_workload_full_size(cuda, B):
    """64 q-heads over 8 kv-heads, 32768 cached tokens + 1 appended, k8v3."""
    w = tq_synth.WORKLOADS["decode"]
    samples = [(0, 0), (B - 1, 7), (B // 2, 3)]
    _full_size_check(cuda, w, B, samples)


def test_longctx_workload_full_size(cuda):
    """32 sequences x 131072 tokens x 8 kv-heads, k4v3 (4.56 GB packed), one step."""
    w = tq_synth.WORKLOADS["longctx"]
    _full_size_check(cuda, w, w.B, [(0, 0), (31, 5)], chunk_b=2)


def test_no_bounded_wait_gave_up(cuda):
    assert cuda.tq_device_error() == 0
