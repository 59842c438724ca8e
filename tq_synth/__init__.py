"""Seeded synthetic inputs for the KV codec (shared by tests, oracle checks and bench).

This module holds none of the codec's arithmetic: it only draws bf16 K, V and q
values from counter-based SplitMix64 streams (definitions in ``synth.h``).  The
host implementation feeds CPU checks and small GPU cases; the device
implementation fills the multi-gigabyte workloads directly in device memory.

Workloads (shapes and distributions of the serving workloads the pages discuss):
  tiny        1 x 4 kv-heads x 256 tokens x d128, k8v3; K ~ N(0,1) x logN(0,1) per channel; V ~ N(0,1)
  prefill     4 x 8 kv-heads x 8192 tokens x d128, k8v3; K ~ N(0,1) x logN(0,1.5); V ~ t5 (unit var)
  decode      B in {1,8,32} x 8 kv-heads, 64 q-heads, 32768 cached tokens + 1 appended per step,
              d128, k8v3, K/V as prefill; q ~ N(0,1)
  sweep       8 kv-heads x 16384 tokens, d in {64,256,512}, kb in {2,4,5,8}, vb in {2,3,4};
              K ~ N(0,1) x logN(0,1), V ~ N(0,1)
  longctx     32 x 8 kv-heads x 131072 tokens x d128, k4v3, 64 q-heads; K/V as prefill
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libtq_synth.so")
_CUDA_SO = os.path.join(_BUILD, "libtq_synth_cuda.so")

V_NORMAL, V_T5 = 0, 1


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    H: int
    T: int
    d: int
    kb: int
    vb: int
    k_log_sigma: float
    v_dist: int
    QH: int = 0


WORKLOADS = {
    "tiny": Workload("tiny", 1001, 1, 4, 256, 128, 8, 3, 1.0, V_NORMAL),
    "prefill": Workload("prefill", 1002, 4, 8, 8192, 128, 8, 3, 1.5, V_T5),
    "decode": Workload("decode", 1003, 32, 8, 32768, 128, 8, 3, 1.5, V_T5, QH=64),
    "sweep": Workload("sweep", 1004, 1, 8, 16384, 128, 8, 3, 1.0, V_NORMAL),
    "longctx": Workload("longctx", 1005, 32, 8, 131072, 128, 4, 3, 1.5, V_T5, QH=64),
}


def _newer(target: str, *srcs: str) -> bool:
    return os.path.exists(target) and all(os.path.getmtime(target) >= os.path.getmtime(s) for s in srcs)


def build_host(force: bool = False) -> str:
    src, hdr = os.path.join(_HERE, "synth.c"), os.path.join(_HERE, "synth.h")
    if not force and _newer(_HOST_SO, src, hdr):
        return _HOST_SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _HOST_SO + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_cuda(force: bool = False) -> str:
    src, hdr = os.path.join(_HERE, "synth_cuda.cu"), os.path.join(_HERE, "synth.h")
    if not force and _newer(_CUDA_SO, src, hdr):
        return _CUDA_SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _CUDA_SO + f".{os.getpid()}.tmp"
    subprocess.run(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-gencode",
                    "arch=compute_103a,code=sm_103a", "-o", tmp, src], check=True)
    os.replace(tmp, _CUDA_SO)
    return _CUDA_SO


_P, _I, _L, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64


@lru_cache(maxsize=1)
def _host():
    so = ctypes.CDLL(build_host())
    so.tqs_host_kv.argtypes = [_U, _I, _I, _I, _L, _L, _I, ctypes.c_double, _I, _P, _P]
    so.tqs_host_q.argtypes = [_U, _L, _I, _I, _I, _P]
    so.tqs_splitmix64.restype = _U
    so.tqs_splitmix64.argtypes = [_U, _U]
    return so


@lru_cache(maxsize=1)
def _cuda():
    so = ctypes.CDLL(build_cuda())
    so.tqs_device_kv.argtypes = [_U, _I, _I, _I, _L, _L, _I, ctypes.c_double, _I, _P, _P, _P]
    so.tqs_device_kv.restype = _I
    so.tqs_device_q.argtypes = [_U, _L, _I, _I, _I, _P, _P]
    so.tqs_device_q.restype = _I
    return so


def host_kv(w: Workload, B=None, H=None, d=None, t_begin: int = 0, n: int | None = None,
            want_k: bool = True, want_v: bool = True, b_offset: int = 0):
    """bf16 bits K, V [B][H][n][d] for tokens [t_begin, t_begin+n)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    d = w.d if d is None else d
    n = w.T if n is None else n
    k = np.zeros((B, H, n, d), dtype=np.uint16) if want_k else None
    v = np.zeros((B, H, n, d), dtype=np.uint16) if want_v else None
    _host().tqs_host_kv(w.seed, B, H, d, t_begin, n, b_offset, w.k_log_sigma, w.v_dist,
                        None if k is None else k.ctypes.data, None if v is None else v.ctypes.data)
    return k, v


def host_q(w: Workload, step: int, B=None, QH=None, d=None):
    B = w.B if B is None else B
    QH = w.QH if QH is None else QH
    d = w.d if d is None else d
    q = np.zeros((B, QH, d), dtype=np.uint16)
    _host().tqs_host_q(w.seed, step, B, QH, d, q.ctypes.data)
    return q


def device_kv(w: Workload, k_out, v_out, B=None, H=None, d=None, t_begin: int = 0, n=None, stream=None,
              b_offset: int = 0):
    """Fill device tensors (torch, bf16/int16 [B][H][n][d] contiguous) in place."""
    import torch

    B = w.B if B is None else B
    H = w.H if H is None else H
    d = w.d if d is None else d
    n = w.T if n is None else n
    for t in (k_out, v_out):
        if t is not None:
            assert t.is_cuda and t.is_contiguous() and t.numel() == B * H * n * d and t.element_size() == 2
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = _cuda().tqs_device_kv(w.seed, B, H, d, t_begin, n, b_offset, w.k_log_sigma, w.v_dist,
                               None if k_out is None else k_out.data_ptr(),
                               None if v_out is None else v_out.data_ptr(), s)
    if rc != 0:
        raise RuntimeError(f"synthetic KV fill failed (cuda error {rc})")


def device_q(w: Workload, step: int, q_out, B=None, QH=None, d=None, stream=None):
    import torch

    B = w.B if B is None else B
    QH = w.QH if QH is None else QH
    d = w.d if d is None else d
    assert q_out.is_cuda and q_out.is_contiguous() and q_out.numel() == B * QH * d
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = _cuda().tqs_device_q(w.seed, step, B, QH, d, q_out.data_ptr(), s)
    if rc != 0:
        raise RuntimeError(f"synthetic q fill failed (cuda error {rc})")
