"""Failure path of the bounded waits, made without a fault: a kernel waits on a
barrier that nothing completes, gives up at its limit, records the timeout code
in the device error word, and the context stays usable for the next calls."""
import time

import numpy as np
import pytest

import oracle
import tq_synth
from tqtest import planes_from_device, to_device_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(cuda):
    assert cuda.tq_device_error() == 0  # nothing pending from earlier calls
    t = time.perf_counter()
    cuda.tq_check_wait_timeout()
    code = cuda.tq_device_error()  # synchronises
    waited = time.perf_counter() - t
    assert code == cuda.TQ_DEVICE_ERR_WAIT_TIMEOUT
    assert 1.0 < waited < 60.0, waited  # the limit is ~2 s of device time
    assert cuda.tq_device_error() == 0  # reading the word cleared it

    # the context is still usable: an append and a decode attention afterwards
    # match the oracle and report no error
    w = tq_synth.WORKLOADS["decode"]
    B, H, T = 2, 2, 300
    k, v = tq_synth.host_kv(w, B=B, H=H, n=T)
    cache = cuda.Cache(B, H, w.d, T + 4, k_bits=w.kb, v_bits=w.vb)
    cuda.tq_encode_append(cache, to_device_bf16(k), to_device_bf16(v), 0)
    q = tq_synth.host_q(w, 0, B=B, QH=8 * H)
    out = cuda.tq_decode_attention(cache, to_device_bf16(q), T)
    want = oracle.attention(planes_from_device(cache), q, T)
    assert np.abs(out.cpu().numpy().astype(np.float64) - want).max() < 2e-3
    assert cuda.tq_device_error() == 0
