"""Decode attention for every head_dim, bit pair and GQA group size (the
generic kernel; head_dims 64, 128 and 256 with 8- or 4-bit keys and 2-, 3-
or 4-bit values take the specialised kernel, in blocks of 8 q-heads) against
the binary64 oracle.  Tolerance: 2e-3
max-abs on the fp32 output, as for the specialised kernel.
"""
import numpy as np
import pytest
import torch

import oracle
import tq_synth
from tqtest import planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3
COMBOS = [(d, kb, vb) for d in (64, 128, 256, 512) for kb in (2, 4, 5, 8) for vb in (2, 3, 4, 5, 8)]


def _run(tq, d, kb, vb, B, H, G, T, cap=None, step=0, w=None):
    w = w or tq_synth.WORKLOADS["sweep"]
    k, v = tq_synth.host_kv(w, B=B, H=H, d=d, n=T)
    cache = tq.Cache(B, H, d, cap or T, k_bits=kb, v_bits=vb)
    tq.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    q = tq_synth.host_q(tq_synth.WORKLOADS["decode"], step, B=B, QH=G * H, d=d)
    out = tq.tq_decode_attention(cache, to_device_bf16(q), T)
    # the oracle attends over the GPU's own bytes (the codec is checked separately)
    want = oracle.attention(planes_from_device(cache), q, T)
    return np.abs(out.cpu().numpy().astype(np.float64) - want).max()


@pytest.mark.parametrize("d,kb,vb", COMBOS)
def test_every_width_and_head_dim(cuda, d, kb, vb):
    err = _run(cuda, d, kb, vb, B=2, H=2, G=8, T=137)
    assert err < TOL, err


@pytest.mark.parametrize("G", [1, 2, 3, 6, 12, 16])
def test_group_sizes(cuda, G):
    err = _run(cuda, 128, 8, 3, B=2, H=3, G=G, T=201, step=G)
    assert err < TOL, err


@pytest.mark.parametrize("kb,G,T", [(8, 4, 5000), (4, 4, 3001), (8, 7, 2050), (4, 1, 777), (8, 5, 64),
                                    (8, 16, 4000), (4, 12, 2500), (8, 24, 900), (4, 9, 1234)])
def test_specialised_kernel_group_sizes(cuda, kb, G, T):
    """Groups other than 8 on the specialised kernel (blocks of the MMA's 8
    columns, those past G dropped): several splits, ragged stage tails, ragged
    combine blocks, one to three column blocks per kv-head (two per CTA above
    8, the last CTA of G = 24 holding one real block and one of padding)."""
    err = _run(cuda, 128, kb, 3, B=3, H=3, G=G, T=T, cap=T + (16 - T % 16) % 16 + 16, step=G)
    assert err < TOL, err


@pytest.mark.parametrize("d,kb,G,T", [(64, 8, 8, 5000), (64, 4, 12, 3001), (256, 8, 4, 4133), (256, 4, 16, 2050),
                                      (256, 8, 8, 777), (64, 8, 1, 64)])
def test_specialised_kernel_head_dims(cuda, d, kb, G, T):
    """The specialised kernel at head_dims 64 and 256 (one 32-byte, 64-byte or
    128-byte swizzled key box per row, or two at d256 k8; the generic kernel's
    merge): several splits, ragged stage tails, one or two column blocks per
    kv-head, padding columns."""
    err = _run(cuda, d, kb, 3, B=3, H=2, G=G, T=T, cap=T + (16 - T % 16) % 16 + 16, step=G)
    assert err < TOL, err


@pytest.mark.parametrize("d,kb,vb,G,T", [(128, 8, 4, 8, 5000), (128, 4, 2, 12, 3001), (256, 8, 4, 4, 4133),
                                         (64, 4, 2, 8, 2050), (256, 4, 2, 16, 777), (64, 8, 4, 3, 1234),
                                         (128, 8, 4, 16, 2222), (64, 4, 4, 16, 1500), (64, 8, 2, 10, 999)])
def test_specialised_kernel_value_widths(cuda, d, kb, vb, G, T):
    """2- and 4-bit values on the specialised kernel (one permute per f16 pair
    out of the four 2-bit centroids; 4-bit codes as a magnitude index and a
    sign, the table being odd): several splits, ragged tails, padding columns."""
    err = _run(cuda, d, kb, vb, B=3, H=2, G=G, T=T, cap=T + (16 - T % 16) % 16 + 16, step=G)
    assert err < TOL, err


@pytest.mark.parametrize("d,kb,vb,G,T", [(256, 8, 3, 8, 8200), (256, 4, 4, 8, 8200), (64, 8, 3, 8, 16400),
                                         (64, 4, 2, 8, 16400), (128, 4, 3, 16, 8200), (64, 8, 3, 12, 16400),
                                         (128, 4, 3, 8, 8200), (128, 4, 4, 8, 8200)])
def test_specialised_kernel_many_stages_per_split(cuda, d, kb, vb, G, T):
    """Enough (sequence, kv-head) pairs (4 x 8) that the split plan fills the
    GPU with few splits, so each CTA walks several stages (64 rows, 128 at
    head_dim 64) and its running max rises after the first: every output
    m-tile (2 head_dim / 32 of them, per column block) must be rescaled then,
    not only the first eight; two column blocks per CTA at G = 12 and 16; three
    tiles per warp (96-row stages) at d128 with 4-bit keys."""
    err = _run(cuda, d, kb, vb, B=4, H=8, G=G, T=T, step=d + kb + G)
    assert err < TOL, err


@pytest.mark.parametrize("d,kb,vb,G,T", [(256, 4, 2, 4, 5000), (64, 8, 4, 8, 9000), (512, 5, 3, 2, 1500)])
def test_long_contexts_split(cuda, d, kb, vb, G, T):
    """Several splits per (sequence, kv-head) and ragged stage tails."""
    err = _run(cuda, d, kb, vb, B=1, H=2, G=G, T=T, cap=T + 11 + (16 - (T + 11) % 16) % 16)
    assert err < TOL, err


def test_single_row_and_decode_step_flow(cuda):
    w = tq_synth.WORKLOADS["decode"]
    d, kb, vb, B, H, G = 256, 8, 2, 2, 2, 4
    k, v = tq_synth.host_kv(tq_synth.WORKLOADS["sweep"], B=B, H=H, d=d, n=40)
    cache = cuda.Cache(B, H, d, 48, k_bits=kb, v_bits=vb)
    ref = oracle.Planes(B, H, d, kb, vb, cache.capacity)
    for t in (0, 1, 2, 39):
        if t == 39:
            cuda.tq_encode_append(cache, to_device_bf16(k[:, :, 3:39]), to_device_bf16(v[:, :, 3:39]), 3)
        cuda.tq_encode_append(cache, to_device_bf16(k[:, :, t:t + 1]), to_device_bf16(v[:, :, t:t + 1]), t)
        q = tq_synth.host_q(w, t, B=B, QH=G * H, d=d)
        out = cuda.tq_decode_attention(cache, to_device_bf16(q), t + 1)
        want = oracle.attention(planes_from_device(cache), q, t + 1)
        assert np.abs(out.cpu().numpy() - want).max() < TOL
    assert cuda.tq_device_error() == 0
