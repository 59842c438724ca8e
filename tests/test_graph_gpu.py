"""The calls are capturable in a CUDA graph: one decode step (append the
token, attend over the cache including it), a fetch and a multi-token
attention are captured once and replayed with new data written into the
captured input buffers; each replay is checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3


def test_decode_step_replayed_from_a_graph(cuda):
    B, H, G, d, T, M = 2, 2, 8, 128, 300, 4
    w = tq_synth.WORKLOADS["sweep"]
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T + 3)
    cache = cuda.Cache(B, H, d, T + 1)
    cuda.tq_encode_append(cache, to_device_bf16(k[:, :, :T]), to_device_bf16(v[:, :, :T]), 0)
    # captured inputs / outputs / workspaces
    knew = torch.empty((B, H, 1, d), dtype=torch.bfloat16, device="cuda")
    vnew = torch.empty_like(knew)
    q = torch.empty((B, G * H, d), dtype=torch.bfloat16, device="cuda")
    qm = torch.empty((B, M, G * H, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, G * H, d), dtype=torch.float32, device="cuda")
    outm = torch.empty((B, M, G * H, d), dtype=torch.float32, device="cuda")
    kf = torch.empty((B, H, T + 1, d), dtype=torch.float32, device="cuda")
    vf = torch.empty_like(kf)
    ws = torch.empty(cuda.tq_attention_workspace_bytes(cache, G * H, T + 1), dtype=torch.uint8, device="cuda")
    wsm = torch.empty(cuda.tq_multi_token_workspace_bytes(cache, G * H, M, T + 1), dtype=torch.uint8, device="cuda")

    def step():
        cuda.tq_encode_append(cache, knew, vnew, T)
        cuda.tq_decode_attention(cache, q, T + 1, out=out, workspace=ws)
        cuda.tq_decode(cache, 0, T + 1, dtype=torch.float32, k_out=kf, v_out=vf)
        cuda.tq_multi_token_attention(cache, qm, T + 1, out=outm, workspace=wsm)

    def load(r):
        knew.copy_(to_device_bf16(k[:, :, T + r:T + r + 1]))
        vnew.copy_(to_device_bf16(v[:, :, T + r:T + r + 1]))
        qh = tq_synth.host_q(tq_synth.WORKLOADS["decode"], r, B=B, QH=G * H, d=d)
        qmh = np.stack([tq_synth.host_q(tq_synth.WORKLOADS["decode"], 10 + r + i, B=B, QH=G * H, d=d)
                        for i in range(M)], axis=1)
        q.copy_(to_device_bf16(qh))
        qm.copy_(to_device_bf16(qmh))
        return qh, qmh

    load(0)
    step()  # eager first: one-time set-up (function attributes, symbol lookups) stays out of the graph
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for r in (1, 2):
        qh, qmh = load(r)
        g.replay()
        torch.cuda.synchronize()
        got = planes_from_device(cache)
        ref = oracle.Planes(B, H, d, 8, 3, cache.capacity)
        oracle.encode(ref, k[:, :, T + r:T + r + 1], v[:, :, T + r:T + r + 1], T)
        assert np.array_equal(got.k_codes[:, :, T], ref.k_codes[:, :, T])  # this replay's token was appended
        want = oracle.attention(got, qh, T + 1)
        assert np.abs(out.cpu().numpy() - want).max() < TOL
        ko, vo = oracle.decode(got, 0, T + 1)
        assert np.array_equal(kf.cpu().numpy(), ko)
        assert np.allclose(vf.cpu().numpy(), vo, rtol=0, atol=1e-3 * np.abs(vo).max())
        wantm = oracle.attention_multi(got, qmh, T + 1)
        assert np.abs(outm.cpu().numpy() - wantm).max() < TOL
    assert cuda.tq_device_error() == 0
