"""The data-parallel split on one GPU: the shards of a world-2 plan (rank r owns
sequences [r B, (r + 1) B) of the global batch) run one after the other,
each into its own cache with its own queries, as two ranks would.

Joined in rank order, the shards' cache bytes must equal one rank's encoding
of the global batch byte for byte.  The attention outputs must agree with the
global run within 2e-3 (the split plan depends on the batch, so the summation
order may differ) and with the oracle on sampled (sequence, kv-head) pairs.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import tq_synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _encode(tq, w, B, H, T, kb, b_offset):
    cache = tq.Cache(B, H, w.d, T, k_bits=kb, v_bits=w.vb)
    k = torch.empty((B, H, T, w.d), dtype=torch.int16, device="cuda")
    v = torch.empty_like(k)
    tq_synth.device_kv(w, k, v, B=B, H=H, n=T, b_offset=b_offset)
    tq.tq_encode_append(cache, k.view(torch.bfloat16), v.view(torch.bfloat16), 0)
    return cache


@pytest.mark.parametrize("kb", [8, 4])
def test_two_shards_equal_the_global_batch(cuda, kb):
    w = tq_synth.WORKLOADS["decode"]
    world, per_rank, H, T = 2, 3, 8, 4097
    QH = w.QH
    glob = _encode(cuda, w, world * per_rank, H, T, kb, 0)
    q = torch.empty((world * per_rank, QH, w.d), dtype=torch.int16, device="cuda")
    tq_synth.device_q(w, 0, q, B=world * per_rank, QH=QH)
    qb = q.view(torch.bfloat16)
    out_g = cuda.tq_decode_attention(glob, qb, T)
    for r in range(world):
        start, n = bench.rank_shard(r, world, per_rank)
        shard = _encode(cuda, w, n, H, T, kb, start)
        for a, b in zip(shard.planes(), glob.planes()):
            assert torch.equal(a, b[start:start + n]), "shard bytes differ from the global encoding"
        out = cuda.tq_decode_attention(shard, qb[start:start + n].contiguous(), T)
        assert (out - out_g[start:start + n]).abs().max().item() < TOL
        # one sampled (sequence, kv-head) pair of this shard against the oracle
        b, h = n - 1, 3 + r
        p = oracle.Planes(1, 1, w.d, kb, w.vb, shard.capacity)
        for dst, src in zip(p.arrays(), shard.planes()):
            dst[0, 0] = src[b, h].cpu().numpy().view(dst.dtype)
        G = QH // H
        qs = qb[start + b:start + b + 1, h * G:(h + 1) * G].contiguous().view(torch.int16).cpu().numpy()
        want = oracle.attention(p, qs.view(np.uint16), T)[0]
        got = out[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
        assert np.abs(got - want).max() < TOL
    assert cuda.tq_device_error() == 0
