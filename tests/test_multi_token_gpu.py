"""Causal multi-token attention (M query rows per sequence, row i seeing
cache rows [0, seq_len - M + i]) against the binary64 oracle.  Tolerance:
2e-3 max-abs on the fp32 output, as for decode attention.

Shapes: the page's forward shapes M = 1, 4 and 128 plus ragged ones (M * G
not a multiple of 8, one column block short), every head_dim (1, 2 or 4
blocks of 8 columns per CTA), long contexts with several splits, and M equal
to the whole cache (query 0 sees one row).
"""
import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _queries(B, M, QH, d, step=0):
    """[B][M][QH][d] bf16 bits from the seeded decode-query stream, one step per row."""
    w = tq_synth.WORKLOADS["decode"]
    return np.stack([tq_synth.host_q(w, step + i, B=B, QH=QH, d=d) for i in range(M)], axis=1)


def _run(tq, d, kb, vb, B, H, G, M, T, cap=None, step=0):
    w = tq_synth.WORKLOADS["sweep"]
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T)
    cache = tq.Cache(B, H, d, cap or T, k_bits=kb, v_bits=vb)
    tq.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    q = _queries(B, M, G * H, d, step)
    out = tq.tq_multi_token_attention(cache, to_device_bf16(q), T)
    want = oracle.attention_multi(planes_from_device(cache), q, T)
    assert tq.tq_device_error() == 0
    return np.abs(out.cpu().numpy().astype(np.float64) - want).max()


@pytest.mark.parametrize("d,kb,vb,G,M", [
    (128, 8, 3, 8, 1), (128, 8, 3, 8, 4), (128, 8, 3, 8, 128), (128, 4, 3, 8, 4),
    (64, 2, 2, 8, 4), (64, 5, 8, 3, 5), (64, 8, 4, 1, 128),
    (256, 4, 2, 4, 4), (256, 8, 5, 8, 3), (256, 5, 3, 2, 128),
    (512, 8, 3, 2, 4), (512, 2, 4, 8, 7),
    (128, 2, 5, 6, 4), (128, 5, 4, 16, 4), (128, 8, 8, 1, 1), (128, 4, 2, 12, 3),
])
def test_shapes(cuda, d, kb, vb, G, M):
    err = _run(cuda, d, kb, vb, B=2, H=2, G=G, M=M, T=301, step=7 * M)
    assert err < TOL, err


@pytest.mark.parametrize("d,kb,vb,G,M,T", [(128, 8, 3, 8, 4, 5000), (128, 4, 3, 8, 128, 3000),
                                           (64, 8, 4, 4, 16, 9000), (256, 4, 3, 8, 4, 4100)])
def test_long_contexts_split(cuda, d, kb, vb, G, M, T):
    """Several splits per (sequence, kv-head); the causal edge falls in the last split."""
    err = _run(cuda, d, kb, vb, B=1, H=2, G=G, M=M, T=T, cap=T + 21 + (16 - (T + 21) % 16) % 16)
    assert err < TOL, err


@pytest.mark.parametrize("d,G,T", [(128, 8, 37), (64, 3, 70), (512, 1, 19)])
def test_whole_cache_is_the_chunk(cuda, d, G, T):
    """M = seq_len: a prefill from empty, query 0 attending to row 0 only."""
    err = _run(cuda, d, 8, 3, B=2, H=2, G=G, M=T, T=T)
    assert err < TOL, err


def test_one_row_matches_decode_attention(cuda):
    """M = 1 through the multi-token entry equals tq_decode_attention (the
    specialised kernel at these parameters) within the shared tolerance."""
    B, H, G, d, T = 3, 2, 8, 128, 777
    k, v = tq_synth.host_kv(tq_synth.WORKLOADS["sweep"], B=B, H=H, d=d, n=T)
    cache = cuda.Cache(B, H, d, T)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    q = _queries(B, 1, G * H, d, 3)
    multi = cuda.tq_multi_token_attention(cache, to_device_bf16(q), T)[:, 0]
    single = cuda.tq_decode_attention(cache, to_device_bf16(q[:, 0]), T)
    assert (multi - single).abs().max().item() < TOL


def test_verify_flow_append_then_attend(cuda):
    """Speculative-verify shape: a cache of 500 rows, then chunks of 4 and 128
    rows appended and attended to, each chunk checked against the oracle."""
    B, H, G, d = 2, 2, 8, 128
    k, v = tq_synth.host_kv(tq_synth.WORKLOADS["sweep"], B=B, H=H, d=d, n=632)
    cache = cuda.Cache(B, H, d, 640)
    cuda.tq_encode_append(cache, to_device_bf16(k[:, :, :500]), to_device_bf16(v[:, :, :500]), 0)
    t = 500
    for M in (4, 128):
        cuda.tq_encode_append(cache, to_device_bf16(k[:, :, t:t + M]), to_device_bf16(v[:, :, t:t + M]), t)
        t += M
        q = _queries(B, M, G * H, d, t)
        out = cuda.tq_multi_token_attention(cache, to_device_bf16(q), t)
        want = oracle.attention_multi(planes_from_device(cache), q, t)
        assert np.abs(out.cpu().numpy() - want).max() < TOL
    assert cuda.tq_device_error() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kb,vb", [(kb, vb) for kb in (2, 4, 5, 8) for vb in (2, 3, 4, 5, 8)])
def test_tensor_core_path_every_width(cuda, d, kb, vb):
    """Chunks of 16 rows x 8 q-heads (128 columns per kv-head): the tcgen05
    kernel at head_dim 64 and 128, every key/value width."""
    err = _run(cuda, d, kb, vb, B=1, H=2, G=8, M=16, T=333, step=kb * 10 + vb)
    assert err < TOL, err


@pytest.mark.parametrize("d,G,M,T", [(128, 8, 15, 260), (128, 8, 16, 64), (128, 6, 50, 700), (64, 16, 40, 2100),
                                     (128, 1, 300, 300), (256, 8, 16, 290)])
def test_around_the_tensor_core_threshold(cuda, d, G, M, T):
    """Just below 128 columns (generic kernel), exactly 128, ragged column
    blocks of 256, one q-head per kv-head, and head_dim 256 (generic)."""
    err = _run(cuda, d, 8, 3, B=2, H=2, G=G, M=M, T=T, step=M)
    assert err < TOL, err


def _slab(cache, b, h):
    """One (sequence, kv-head) of a device cache as a 1 x 1 oracle cache."""
    g = oracle.Planes(1, 1, cache.head_dim, cache.k_bits, cache.v_bits, cache.capacity)
    for ga, src in zip(g.arrays(), cache.planes()):
        ga[0, 0] = src[b, h].cpu().numpy().view(ga.dtype)
    return g


@pytest.mark.parametrize("kb,M", [(8, 128), (4, 16)])
def test_full_size_chunk_sampled(cuda, kb, M):
    """The measured shape: 8 sequences x 8 kv-heads x 32769 rows (d128, 64
    q-heads, the decode workload's heavy-tailed keys), a chunk of M rows at the
    end; sampled (sequence, kv-head, query row) outputs against the oracle."""
    w = tq_synth.WORKLOADS["decode"]
    B, H, T, d, G = 8, 8, 32769, 128, 8
    cache = cuda.Cache(B, H, d, T, k_bits=kb, v_bits=3)
    for b0 in range(B):
        k = torch.empty((1, H, T, d), dtype=torch.int16, device="cuda")
        v = torch.empty_like(k)
        tq_synth.device_kv(w, k, v, B=1, H=H, d=d, n=T, b_offset=b0)
        cuda.tq_encode_append(cache.batch_slice(b0, 1), k.view(torch.bfloat16), v.view(torch.bfloat16), 0)
        del k, v
    q = torch.empty((B, M * G * H, d), dtype=torch.int16, device="cuda")
    tq_synth.device_q(w, 0, q, B=B, QH=M * G * H, d=d)
    out = cuda.tq_multi_token_attention(cache, q.view(torch.bfloat16).view(B, M, G * H, d), T).cpu().numpy()
    qh = q.cpu().numpy().view(np.uint16).reshape(B, M, G * H, d)
    assert cuda.tq_device_error() == 0
    for (b, h) in [(0, 0), (B - 1, 5)]:
        g = _slab(cache, b, h)
        for i in (0, 1, M // 2, M - 1):
            want = oracle.attention(g, np.ascontiguousarray(qh[b:b + 1, i, h * G:(h + 1) * G]), T - M + i + 1)
            err = np.abs(out[b, i, h * G:(h + 1) * G] - want[0]).max()
            assert err < TOL, (b, h, i, err)
