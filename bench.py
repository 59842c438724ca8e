#!/usr/bin/env python3
"""Benchmark of the TurboQuant KV-codec hot path on GB300.

One step is one pass of the whole path over one batch of synthetic input:
  1. append  -- quantise a prefill batch (4 seq x 8 kv-heads x 8192 tokens x d128,
                k8v3) into a packed cache (tq_encode_append);
  2. fetch   -- dequantise a prefill cache back to bf16 K, V (tq_decode); two
                caches alternate, so the fetch reads rows written a step earlier,
                never rows the append just left in L2;
  3. decode  -- one decode step of the serving workload (32 seq x 64 q-heads over
                8 kv-heads, 32768 cached tokens): append the new token of every
                sequence, then fused dequantise-on-fetch attention over 32769
                rows (tq_decode_attention).
Every input of a step (134 MB + 134 MB bf16, a 52 MB cache, the 1.68 GB decode
cache) is larger than L2 or was evicted by the rest of the step.

value = algorithmic bytes of the whole step / step time (GB/s), the bytes being
the codec's format traffic: bf16 K/V in and packed rows out for the append,
packed rows in and bf16 out for the fetch, every cached row (200 B per
token-head) plus q and the output for the attention.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       python bench.py --sweep   (one JSON line per path beyond the headline step:
                                  attention at other widths/head dims/groups, the
                                  deferred fetch, the un-rotation, row copies)
Under torchrun each rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV codec encode/decode GB/s and fused dequant-attn µs/step, % of HBM roofline"
PREFILL = dict(B=4, H=8, T=8192, d=128, kb=8, vb=3)
DECODE = dict(B=32, H=8, QH=64, T=32768, d=128, kb=8, vb=3)
BYTES_PER_TH = 200  # k8v3, d128 (page section "Algorithm", bytes per token-head)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0  # dense bf16, one earlier GB300 measurement
NOMINAL_HBM_GBS = 8000.0  # the codec's stated roofline: bytes moved / 8 TB/s
# decode attention at other head_dims and widths: (head_dim, key bits, value bits, sequences), ~0.4 GB each
OTHER_ATTN = ((256, 8, 3, 4), (64, 8, 3, 15), (128, 8, 4, 7), (128, 5, 2, 11))
LONGCTX = dict(B=32, H=8, QH=64, T=131072, d=128, kb=4, vb=3)
SWEEP = dict(H=8, T=16384, ds=(64, 256, 512), kbs=(2, 4, 5, 8), vbs=(2, 3, 4))


# ------------------------------------------------------------------ helpers
def algorithmic_bytes(prefill=PREFILL, decode=DECODE):
    th_pre = prefill["B"] * prefill["H"] * prefill["T"]
    bf16_row = 2 * prefill["d"] * 2  # K and V bf16
    enc = th_pre * (bf16_row + BYTES_PER_TH)
    dec = th_pre * (BYTES_PER_TH + bf16_row)
    th_new = decode["B"] * decode["H"]
    app = th_new * (2 * decode["d"] * 2 + BYTES_PER_TH)
    attn = decode["B"] * decode["H"] * (decode["T"] + 1) * BYTES_PER_TH \
        + decode["B"] * decode["QH"] * decode["d"] * (2 + 4)  # q in (bf16), out (fp32)
    return dict(encode=enc, decode=dec, append=app, attention=attn, total=enc + dec + app + attn)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak (cuBLAS, burst) from MEASURED_PEAKS.json, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


PRIME_CYCLES = 4_000_000  # ~2 ms of device spin before a timed region starts


def rate(nbytes, us, peak):
    """A part's time with its throughput and its fraction of both rooflines:
    the measured copy bandwidth (frac) and the nominal 8 TB/s (frac_8tbs)."""
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
            "frac_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "bytes": int(nbytes)}


def attention_traffic(kernel_hash: str):
    """DRAM bytes per launch of the attention kernel at this workload, from the
    committed ncu summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "attention_decode_traffic.txt")
    try:
        kv = {}
        with open(p) as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_hash:
            return None
        return float(kv["dram_bytes_per_launch_full_workload"])
    except Exception:
        return None


def kernel_source_hash() -> str:
    p = os.path.join(ROOT, "rotated_kv_cache_gb300", "csrc", "tq_attention.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        busy = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ranks
def rank_shard(rank: int, world: int, per_rank: int) -> tuple[int, int]:
    """Weak scaling over ranks: rank r owns the global units (sequences here)
    [r * per_rank, (r + 1) * per_rank) of a batch of world * per_rank.  The
    units are independent (encode, fetch and attention never mix sequences),
    so the ranks share no data and need no collective on the data path."""
    if world < 1 or not 0 <= rank < world or per_rank < 0:
        raise ValueError("bad rank / world / per_rank")
    return rank * per_rank, per_rank


def max_over_ranks(values, world: int, device="cpu"):
    """Every entry replaced by its maximum over the ranks (the slowest rank's
    time); all ranks receive the result.  One small all-reduce, outside the
    timed region."""
    values = [float(v) for v in values]
    if world == 1:
        return values
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from rotated_kv_cache_gb300 import build as libbuild

    libbuild.build()
    import rotated_kv_cache_gb300 as tq
    import tq_synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    P, D = PREFILL, DECODE
    wp, wd = tq_synth.WORKLOADS["prefill"], tq_synth.WORKLOADS["decode"]
    off_p, _ = rank_shard(rank, world, P["B"])  # this rank's sequences of the global batches
    off_d, _ = rank_shard(rank, world, D["B"])

    # --- prefill inputs and two caches
    kp = torch.empty((P["B"], P["H"], P["T"], P["d"]), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    tq_synth.device_kv(wp, kp, vp, b_offset=off_p)
    pre = [tq.Cache(P["B"], P["H"], P["d"], P["T"], P["kb"], P["vb"], device=dev) for _ in range(2)]
    for c in pre:
        tq.tq_encode_append(c, kp, vp, 0)
    ko = torch.empty_like(kp)
    vo = torch.empty_like(kp)

    # --- decode cache: the context is generated and encoded in chunks of sequences
    T = D["T"]
    dcache = tq.Cache(D["B"], D["H"], D["d"], T + 1, D["kb"], D["vb"], device=dev)
    for b0 in range(0, D["B"], 4):
        nb = min(4, D["B"] - b0)
        kc = torch.empty((nb, D["H"], T + 1, D["d"]), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        tq_synth.device_kv(wd, kc, vc, B=nb, n=T + 1, b_offset=off_d + b0)
        tq.tq_encode_append(dcache.batch_slice(b0, nb), kc[:, :, :T], vc[:, :, :T], 0)
        del kc, vc
    knew = torch.empty((D["B"], D["H"], 1, D["d"]), dtype=torch.bfloat16, device=dev)
    vnew = torch.empty_like(knew)
    tq_synth.device_kv(wd, knew, vnew, B=D["B"], t_begin=T, n=1, b_offset=off_d)
    q = torch.empty((D["B"], D["QH"], D["d"]), dtype=torch.bfloat16, device=dev)
    tq_synth.device_q(wd, rank, q, B=D["B"])  # one query stream per rank
    out = torch.empty((D["B"], D["QH"], D["d"]), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_attention_workspace_bytes(dcache, D["QH"], T + 1), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()

    def step(s, ev=None):
        if ev is not None:
            ev[0].record(stream)
        tq.tq_encode_append(pre[s % 2], kp, vp, 0)
        if ev is not None:
            ev[1].record(stream)
        tq.tq_decode(pre[(s + 1) % 2], 0, P["T"], dtype=torch.bfloat16, k_out=ko, v_out=vo)
        if ev is not None:
            ev[2].record(stream)
        tq.tq_encode_append(dcache, knew, vnew, T)  # the step's new token, row T
        if ev is not None:
            ev[3].record(stream)
        tq.tq_decode_attention(dcache, q, T + 1, out=out, workspace=ws)
        if ev is not None:
            ev[4].record(stream)

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        # keep the GPU busy (outside the timed region) while the host queues the
        # first steps, so no host launch latency lands between the device marks
        torch.cuda._sleep(PRIME_CYCLES)
        t0.record(stream)
        for s in range(K):
            step(s, evs[s])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    parts = {"encode": 0.0, "decode": 0.0, "append": 0.0, "attention": 0.0}
    for e in evs:
        parts["encode"] += e[0].elapsed_time(e[1])
        parts["decode"] += e[1].elapsed_time(e[2])
        parts["append"] += e[2].elapsed_time(e[3])
        parts["attention"] += e[3].elapsed_time(e[4])
    parts = {k: v / K for k, v in parts.items()}
    assert tq.tq_device_error() == 0

    # --- end to end through the public API with pinned host buffers.  Steps
    # are independent, so they are pipelined the way a serving loop would run
    # them: step s's host-to-device copies (copy-in stream), compute (the
    # compute stream) and device-to-host reads (copy-out stream) overlap with
    # the neighbouring steps', on two sets of device buffers.  Every step still
    # copies all of its inputs in and its results out inside the timed region.
    # A step's inputs (prefill K, V, the new token's K, V, q) live in one pinned
    # host buffer and one device buffer per set, its results (fetched K, V,
    # attention output) likewise, so each step is one copy in and one copy out.
    def packing(tensors):
        offs, o = [], 0
        for t in tensors:
            offs.append(o)
            o += (t.numel() * t.element_size() + 511) // 512 * 512
        return offs, o

    def views(buf, offs, like):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, like)]

    ins, outs = (kp, vp, knew, vnew, q), (ko, vo, out)
    in_offs, in_bytes = packing(ins)
    out_offs, out_bytes = packing(outs)
    in_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for hv, t in zip(views(in_h, in_offs, ins), ins):
        hv.copy_(t.cpu())
    out_h = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    sets = []
    for _ in range(2):
        ib = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        ob = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        sets.append(dict(inb=ib, outb=ob, **dict(zip(("kp", "vp", "knew", "vnew", "q"), views(ib, in_offs, ins))),
                         **dict(zip(("ko", "vo", "out"), views(ob, out_offs, outs)))))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    for e in comp_done + out_done:
        e.record(stream)

    def e2e_step(s):
        i = s % 2
        bs = sets[i]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[i])  # set i's inputs were read by step s - 2
            bs["inb"].copy_(in_h, non_blocking=True)
            in_done[i].record(s_in)
        stream.wait_event(in_done[i])
        stream.wait_event(out_done[i])  # set i's outputs were read back by step s - 2
        tq.tq_encode_append(pre[s % 2], bs["kp"], bs["vp"], 0)
        tq.tq_decode(pre[(s + 1) % 2], 0, P["T"], dtype=torch.bfloat16, k_out=bs["ko"], v_out=bs["vo"])
        tq.tq_encode_append(dcache, bs["knew"], bs["vnew"], T)
        tq.tq_decode_attention(dcache, bs["q"], T + 1, out=bs["out"], workspace=ws)
        comp_done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i])
            out_h.copy_(bs["outb"], non_blocking=True)
            out_done[i].record(s_out)

    Ke = 20  # pipelined steps: enough that filling and draining the pipeline stay small
    for s in range(2):
        e2e_step(s)
    torch.cuda.synchronize()
    a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(PRIME_CYCLES)  # as above: the host runs ahead of the device marks
    a.record(stream)
    s_in.wait_event(a)  # no copy of the timed steps starts before the start mark
    for s in range(Ke):
        e2e_step(s)
    for e in out_done:  # the last reads back are inside the timed region
        stream.wait_event(e)
    bb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(bb) / Ke
    h2d, d2h = in_h.numel(), out_h.numel()  # the bytes each step copies (padding included)

    # --- the other configurations (outside the headline's timed region)
    ctimes, cbytes = ({}, {}) if args.no_configs else \
        measure_configs(tq, tq_synth, torch, dev, dcache, knew, vnew, q, T, rank)

    # --- aggregate over ranks (max time)
    names = ("encode", "decode", "append", "attention")
    cnames = sorted(ctimes)
    tt = max_over_ranks([elapsed_ms / K, e2e_ms] + [parts[k] for k in names] + [ctimes[k] for k in cnames],
                        world, dev)
    ms, e2e_ms = tt[0], tt[1]
    parts = dict(zip(names, tt[2:2 + len(names)]))
    ctimes = dict(zip(cnames, tt[2 + len(names):]))
    if rank != 0:
        return None

    ab = algorithmic_bytes()
    peak, peak_kind = measured_peaks()
    gbs = lambda nbytes, t_ms: nbytes / (t_ms * 1e-3) / 1e9  # noqa: E731
    value = world * ab["total"] / (ms * 1e-3) / 1e9
    attn_gbs = gbs(ab["attention"], parts["attention"])
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 streams: K ~ N(0,1) x per-channel logN(0,1.5), V ~ Student-t5)",
        "config": {
            "workload": "prefill append+fetch (4x8192 tokens x 8 kv-heads x d128, k8v3) + decode step "
                        "(32 seq x 64 q-heads / 8 kv-heads, 32768 cached tokens + 1 appended, d128, k8v3)",
            "l2": "inputs larger than L2; the fetch reads the cache appended a step earlier (two caches alternate)",
            "parallelism": "single GPU" if world == 1 else
                           f"data parallel x{world}: rank r owns sequences [r*B, (r+1)*B) of the global batches "
                           "(weak scaling, no data-path collective)",
            "algorithmic_bytes_per_step": ab["total"],
        },
        "parts": {
            "encode": rate(ab["encode"], parts["encode"] * 1e3, peak),
            "decode": rate(ab["decode"], parts["decode"] * 1e3, peak),
            "append_1_token": rate(ab["append"], parts["append"] * 1e3, peak),
            "attention": {**rate(ab["attention"], parts["attention"] * 1e3, peak),
                          "us_per_step": round(parts["attention"] * 1e3, 2)},
            "decode_step_us": round((parts["append"] + parts["attention"]) * 1e3, 2),
            **config_parts(ctimes, cbytes, peak),
        },
        "roofline": {
            "kernel": "attn_split_kernel + attn_combine_kernel (timed together through tq_decode_attention)",
            "bound": "hbm",
            "achieved": round(attn_gbs, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(attn_gbs / peak, 4),
            "frac_8tbs": round(attn_gbs / NOMINAL_HBM_GBS, 4),
            "traffic": attention_traffic(kernel_source_hash()),
            "algorithmic_bytes_per_launch": ab["attention"],
        },
        "e2e": {"value": round(world * ab["total"] / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "pipelined": "copy-in, compute and copy-out streams overlap neighbouring steps (2 buffer sets; one copy in and one copy out per step)"},
        # per step: prefill append (key and value kernels), fetch (one kernel for keys
        # and values), single-token append (one kernel), attention (split + combine)
        "gpu_launches": 6 * K,
        "clocks": clocks.summary(),
    }
    return line


# ------------------------------------------------------------------ the other configurations
def flushing_timer(torch, dev):
    """fn's median device time in µs over `reps` calls, each call preceded by a
    read of a buffer twice the size of L2 (so its inputs come from HBM, and the
    previous call's dirty lines are written back before the marks, not inside
    them) and bracketed by CUDA events on the launching stream; a device spin
    queued first keeps host launch time out of the marks."""
    st = torch.cuda.current_stream()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    flush = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def timed(fn, reps=10, warmup=3):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda._sleep(PRIME_CYCLES)
        for a, b in evs:
            torch.sum(flush, dim=0, out=sink)  # reads the whole buffer
            a.record(st)
            fn()
            b.record(st)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)

    return timed


def decode_steps(tq, torch, dev, cache, knew, vnew, q, seq_len, nb, groups, steps):
    """Decode steps of nb sequences: append each sequence's new token at row
    seq_len - 1, then attention over seq_len rows.  `groups` disjoint batch
    slices of the cache take turns, so a slice's rows have left L2 before its
    next turn (each slice alone may fit in L2).  Returns µs of the append and
    of the attention (median over calls, CUDA events around each call) and of
    the whole step replayed from a CUDA graph per slice (mean over steps)."""
    st = torch.cuda.current_stream()
    QH, d = q.shape[1], q.shape[2]
    ws_bytes = tq.tq_attention_workspace_bytes(cache.batch_slice(0, nb), QH, seq_len)
    sl = []
    for i in range(groups):
        b0 = i * nb
        sl.append(dict(c=cache.batch_slice(b0, nb), kn=knew[b0:b0 + nb], vn=vnew[b0:b0 + nb], q=q[b0:b0 + nb],
                       out=torch.empty((nb, QH, d), dtype=torch.float32, device=dev),
                       ws=torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)))

    def append(x):
        tq.tq_encode_append(x["c"], x["kn"], x["vn"], seq_len - 1)

    def attend(x):
        tq.tq_decode_attention(x["c"], x["q"], seq_len, out=x["out"], workspace=x["ws"])

    for _ in range(3):
        for x in sl:
            append(x)
            attend(x)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda._sleep(PRIME_CYCLES)
    for s_, e in enumerate(ev):
        x = sl[s_ % groups]
        e[0].record(st)
        append(x)
        e[1].record(st)
        attend(x)
        e[2].record(st)
    torch.cuda.synchronize()
    app_us = statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in ev)
    att_us = statistics.median(e[1].elapsed_time(e[2]) * 1e3 for e in ev)
    graphs = []
    for x in sl:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            append(x)
            attend(x)
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(PRIME_CYCLES)
    a.record(st)
    for s_ in range(steps):
        graphs[s_ % groups].replay()
    b.record(st)
    torch.cuda.synchronize()
    step_us = a.elapsed_time(b) * 1e3 / steps
    del graphs
    return app_us, att_us, step_us


def decode_step_bytes(nb, H, QH, d, rows, bpt):
    """(append, attention) algorithmic bytes of one decode step: the new token's
    bf16 K, V in and its packed row out; every cached row plus q (bf16) and the
    output (fp32)."""
    return nb * H * (4 * d + bpt), nb * H * rows * bpt + nb * QH * d * 6


def measure_configs(tq, tq_synth, torch, dev, dcache, knew, vnew, q, T, rank, steps=20):
    """Device times (µs) of the configurations beside the headline step:
      decode attention at batch 1 and 8 (slices of the headline decode cache),
      the long-context step (32 x 8 x 131073 rows, k4v3, 4.56 GB packed),
      and encode / fetch of every cell of the width and head_dim sweep
      (8 kv-heads x 16384 tokens; d 64/256/512 x k 2/4/5/8 x v 2/3/4).
    Returns a flat {name: µs} and {name: algorithmic bytes}."""
    times, nbytes = {}, {}
    D = DECODE
    bpt = tq.tq_bytes_per_token_head(D["d"], D["kb"], D["vb"])
    for nb in (1, 8):
        groups = min(4, dcache.batch // nb)
        if groups < 1:
            continue
        app, att, step = decode_steps(tq, torch, dev, dcache, knew, vnew, q, T + 1, nb, groups, steps)
        ab, tb = decode_step_bytes(nb, D["H"], D["QH"], D["d"], T + 1, bpt)
        for k_, us, by in (("append", app, ab), ("attention", att, tb), ("step_graph", step, ab + tb)):
            times[f"decode_b{nb}_{k_}"], nbytes[f"decode_b{nb}_{k_}"] = us, by

    L = LONGCTX
    wl = tq_synth.WORKLOADS["longctx"]
    off, _ = rank_shard(rank, int(os.environ.get("WORLD_SIZE", "1")), L["B"])
    lc = tq.Cache(L["B"], L["H"], L["d"], L["T"] + 1, L["kb"], L["vb"], device=dev)
    for b0 in range(L["B"]):  # the bf16 source (17 GB in all) is generated one sequence at a time
        kc = torch.empty((1, L["H"], L["T"] + 1, L["d"]), dtype=torch.int16, device=dev)
        vc = torch.empty_like(kc)
        tq_synth.device_kv(wl, kc, vc, B=1, H=L["H"], d=L["d"], n=L["T"] + 1, b_offset=off + b0)
        tq.tq_encode_append(lc.batch_slice(b0, 1), kc.view(torch.bfloat16)[:, :, :L["T"]],
                            vc.view(torch.bfloat16)[:, :, :L["T"]], 0)
        if b0 == 0:
            kn = torch.empty((L["B"], L["H"], 1, L["d"]), dtype=torch.int16, device=dev)
            vn = torch.empty_like(kn)
        kn[b0:b0 + 1].copy_(kc[:, :, L["T"]:])
        vn[b0:b0 + 1].copy_(vc[:, :, L["T"]:])
        del kc, vc
    ql = torch.empty((L["B"], L["QH"], L["d"]), dtype=torch.int16, device=dev)
    tq_synth.device_q(wl, rank, ql, B=L["B"], QH=L["QH"], d=L["d"])
    app, att, step = decode_steps(tq, torch, dev, lc, kn.view(torch.bfloat16), vn.view(torch.bfloat16),
                                  ql.view(torch.bfloat16), L["T"] + 1, L["B"], 1, steps)
    lbpt = tq.tq_bytes_per_token_head(L["d"], L["kb"], L["vb"])
    ab, tb = decode_step_bytes(L["B"], L["H"], L["QH"], L["d"], L["T"] + 1, lbpt)
    for k_, us, by in (("append", app, ab), ("attention", att, tb), ("step_graph", step, ab + tb)):
        times[f"long_context_{k_}"], nbytes[f"long_context_{k_}"] = us, by
    del lc, kn, vn, ql
    torch.cuda.empty_cache()

    timed = flushing_timer(torch, dev)
    w = tq_synth.WORKLOADS["sweep"]
    H, Ts = SWEEP["H"], SWEEP["T"]
    for d in SWEEP["ds"]:
        k = torch.empty((1, H, Ts, d), dtype=torch.int16, device=dev)
        v = torch.empty_like(k)
        tq_synth.device_kv(w, k, v, B=1, H=H, d=d, n=Ts)
        k16, v16 = k.view(torch.bfloat16), v.view(torch.bfloat16)
        ko, vo = torch.empty_like(k16), torch.empty_like(v16)
        for kb in SWEEP["kbs"]:
            for vb in SWEEP["vbs"]:
                c = tq.Cache(1, H, d, Ts, kb, vb, device=dev)
                cb = tq.tq_bytes_per_token_head(d, kb, vb)
                name = f"sweep_d{d}_k{kb}v{vb}"
                times[name + "_encode"] = timed(lambda: tq.tq_encode_append(c, k16, v16, 0))
                times[name + "_decode"] = timed(
                    lambda: tq.tq_decode(c, 0, Ts, dtype=torch.bfloat16, k_out=ko, v_out=vo))
                nbytes[name + "_encode"] = nbytes[name + "_decode"] = H * Ts * (4 * d + cb)
                del c
        del k, v, k16, v16, ko, vo

    # decode attention at other head_dims (the specialised kernel) and widths
    # (the generic kernel): ~0.4 GB caches of 32769 rows per sequence and kv-head
    wd = tq_synth.WORKLOADS["decode"]
    Tg = T + 1
    for d, kb, vb, nbg in OTHER_ATTN:
        goff, _ = rank_shard(rank, int(os.environ.get("WORLD_SIZE", "1")), nbg)
        gc = tq.Cache(nbg, D["H"], d, Tg + (16 - Tg % 16) % 16, kb, vb, device=dev)
        for b0 in range(nbg):
            kc = torch.empty((1, D["H"], Tg, d), dtype=torch.int16, device=dev)
            vc = torch.empty_like(kc)
            tq_synth.device_kv(wd, kc, vc, B=1, H=D["H"], d=d, n=Tg, b_offset=goff + b0)
            tq.tq_encode_append(gc.batch_slice(b0, 1), kc.view(torch.bfloat16), vc.view(torch.bfloat16), 0)
            del kc, vc
        qg = torch.empty((nbg, D["QH"], d), dtype=torch.int16, device=dev)
        tq_synth.device_q(wd, 0, qg, B=nbg, QH=D["QH"], d=d)
        qgb = qg.view(torch.bfloat16)
        og = torch.empty((nbg, D["QH"], d), dtype=torch.float32, device=dev)
        wsg = torch.empty(tq.tq_attention_workspace_bytes(gc, D["QH"], Tg), dtype=torch.uint8, device=dev)
        name = f"attention_d{d}_k{kb}v{vb}"
        times[name] = timed(lambda: tq.tq_decode_attention(gc, qgb, Tg, out=og, workspace=wsg))
        nbytes[name] = nbg * D["H"] * Tg * tq.tq_bytes_per_token_head(d, kb, vb) + nbg * D["QH"] * d * 6
        del gc, qg, qgb, og, wsg
    torch.cuda.empty_cache()

    # the follow-up paths: multi-token attention (chunks of M = 4 and 128 query
    # rows over 8 sequences of the decode cache), the deferred fetch and its
    # un-rotation, row copy and clear (a prefill-shaped cache)
    nb8 = min(8, dcache.batch)
    c8 = dcache.batch_slice(0, nb8)
    for M in (4, 128):
        qm = torch.empty((nb8, M * D["QH"], D["d"]), dtype=torch.int16, device=dev)
        tq_synth.device_q(wd, 0, qm, B=nb8, QH=M * D["QH"], d=D["d"])
        qmb = qm.view(torch.bfloat16).view(nb8, M, D["QH"], D["d"])
        om = torch.empty((nb8, M, D["QH"], D["d"]), dtype=torch.float32, device=dev)
        wsm = torch.empty(tq.tq_multi_token_workspace_bytes(c8, D["QH"], M, T + 1), dtype=torch.uint8, device=dev)
        name = f"multi_token_m{M}"
        times[name] = timed(lambda: tq.tq_multi_token_attention(c8, qmb, T + 1, out=om, workspace=wsm), reps=5)
        nbytes[name] = nb8 * D["H"] * (T + 1) * bpt + nb8 * M * D["QH"] * D["d"] * 6
        nbytes[name + "_flops"] = 4.0 * D["d"] * D["QH"] * M * nb8 * (T + 1)  # MMA work of one call
        del qm, qmb, om, wsm
    P = PREFILL
    pc = tq.Cache(P["B"], P["H"], P["d"], P["T"], P["kb"], P["vb"], device=dev)
    kc = torch.empty((P["B"], P["H"], P["T"], P["d"]), dtype=torch.int16, device=dev)
    vc = torch.empty_like(kc)
    tq_synth.device_kv(tq_synth.WORKLOADS["prefill"], kc, vc)
    tq.tq_encode_append(pc, kc.view(torch.bfloat16), vc.view(torch.bfloat16), 0)
    rows = P["B"] * P["H"] * P["T"]
    vr = vc.view(torch.bfloat16)  # reused as the output buffers
    times["rotated_fetch"] = timed(lambda: tq.tq_decode_values_rotated(pc, 0, P["T"], dtype=torch.bfloat16, out=vr))
    nbytes["rotated_fetch"] = rows * (P["d"] * P["vb"] // 8 + 2 * P["d"] // 32 + 2 * P["d"])
    xr = kc.view(torch.float32).view(rows // 2, P["d"])  # 134 MB of rows un-rotated in place
    xr.normal_()
    times["unrotate"] = timed(lambda: tq.tq_unrotate(xr, out=xr))
    nbytes["unrotate"] = 2 * xr.numel() * 4
    snap = tq.Cache(P["B"], P["H"], P["d"], P["T"], P["kb"], P["vb"], device=dev)
    fmt = rows * tq.tq_bytes_per_token_head(P["d"], P["kb"], P["vb"])
    times["copy_rows"] = timed(lambda: tq.tq_cache_copy_rows(snap, 0, pc, 0, P["T"]))
    nbytes["copy_rows"] = 2 * fmt
    times["clear_rows"] = timed(lambda: tq.tq_cache_clear_rows(snap, 0, P["T"]))
    nbytes["clear_rows"] = fmt
    del pc, snap, kc, vc, vr, xr
    assert tq.tq_device_error() == 0
    return times, nbytes


def config_parts(times, nbytes, peak):
    """The measure_configs times as bench-line entries (µs, GB/s, fractions)."""
    out = {}
    for pre, desc in (("decode_b1", "decode step, batch 1, 64 q-heads / 8 kv-heads, 32769 rows, d128 k8v3"),
                      ("decode_b8", "decode step, batch 8, 64 q-heads / 8 kv-heads, 32769 rows, d128 k8v3"),
                      ("long_context", "decode step, batch 32, 64 q-heads / 8 kv-heads, 131073 rows, d128 k4v3 "
                                       "(4.56 GB packed)")):
        if pre + "_attention" not in times:
            continue
        out[pre] = {"workload": desc,
                    "attention": rate(nbytes[pre + "_attention"], times[pre + "_attention"], peak),
                    "append_1_token": rate(nbytes[pre + "_append"], times[pre + "_append"], peak),
                    "step_graph": rate(nbytes[pre + "_step_graph"], times[pre + "_step_graph"], peak)}
    for name, desc in (("multi_token_m4", "causal attention of chunks of 4 query rows, 8 sequences x 8 kv-heads x "
                                          "32769 rows, 64 q-heads, d128 k8v3 (mma.sync kernel)"),
                       ("multi_token_m128", "causal attention of chunks of 128 query rows, same cache (tcgen05 kernel)")):
        if name in times:
            r = rate(nbytes[name], times[name], peak)
            tf = nbytes[name + "_flops"] / (times[name] * 1e-6) / 1e12
            tpeak, tkind = measured_bf16_tflops()
            out[name] = {"workload": desc, **r, "TFLOP/s": round(tf, 1), "tensor_frac": round(tf / tpeak, 4),
                         "tensor_peak": tpeak, "tensor_peak_kind": tkind}
    for d, kb, vb, nbg in OTHER_ATTN:
        name = f"attention_d{d}_k{kb}v{vb}"
        kern = "specialised" if vb in (2, 3, 4) and kb in (8, 4) and d in (64, 128, 256) else "generic"
        if name in times:
            out[name] = {"workload": f"decode attention ({kern} kernel), {nbg} sequences x 8 kv-heads x 32769 rows, "
                                     f"64 q-heads, d{d} k{kb}v{vb}",
                         **rate(nbytes[name], times[name], peak)}
    for name, desc in (("rotated_fetch", "values in the rotated domain, 4 x 8 x 8192 rows, d128 v3, bf16 out"),
                       ("unrotate", "un-rotation of 131072 rows of d128, fp32 in place"),
                       ("copy_rows", "row copy between caches, 4 x 8 x 8192 rows, d128 k8v3"),
                       ("clear_rows", "row clear, 4 x 8 x 8192 rows, d128 k8v3")):
        if name in times:
            out[name] = {"workload": desc, **rate(nbytes[name], times[name], peak)}
    cells = {}
    for k_ in sorted(times):
        if k_.startswith("sweep_") and k_.endswith("_encode"):
            cell = k_[len("sweep_"):-len("_encode")]
            cells[cell] = {op: rate(nbytes[f"sweep_{cell}_{op}"], times[f"sweep_{cell}_{op}"], peak)
                           for op in ("encode", "decode")}
    if cells:
        out["sweep_codec"] = {"workload": "8 kv-heads x 16384 tokens, K ~ N(0,1) x logN(0,1), V ~ N(0,1); "
                                          "encode bf16 -> packed, fetch packed -> bf16; L2 flushed (a read of twice its size) before each call",
                              "cells": cells}
    return out


# ------------------------------------------------------------------ CPU oracle (baseline and reference arm)
class OracleSample:
    """A bounded slice of the same workload for the CPU oracle: append + fetch of
    `pre_rows` prefill tokens (all 4 x 8 sequence-heads), and the decode step's
    attention for `seqs` sequences x `heads` kv-heads (8 q-heads each) over the
    full 32769-row context.  Inputs are generated one sequence at a time."""

    def __init__(self, pre_rows: int, seqs: int, heads: int = 8):
        import numpy as np

        import oracle
        import tq_synth

        self.oracle = oracle
        P, D = PREFILL, DECODE
        wp, wd = tq_synth.WORKLOADS["prefill"], tq_synth.WORKLOADS["decode"]
        self.kp, self.vp = tq_synth.host_kv(wp, n=pre_rows)
        self.planes = oracle.Planes(P["B"], P["H"], P["d"], P["kb"], P["vb"], (pre_rows + 15) // 16 * 16)
        oracle.encode(self.planes, self.kp, self.vp)
        self.pre_rows = pre_rows
        T = D["T"]
        self.att = []
        qall = tq_synth.host_q(wd, 0, B=D["B"], QH=D["QH"])
        for b in range(seqs):
            k, v = tq_synth.host_kv(wd, B=1, H=D["H"], n=T + 1, b_offset=b)
            pl = oracle.Planes(1, heads, D["d"], D["kb"], D["vb"], T + 16)
            oracle.encode(pl, np.ascontiguousarray(k[:, :heads]), np.ascontiguousarray(v[:, :heads]))
            self.att.append((pl, np.ascontiguousarray(qall[b:b + 1, :8 * heads])))
            del k, v
        th = P["B"] * P["H"] * pre_rows
        pairs = seqs * heads
        self.bytes = th * (512 + 200) * 2 + pairs * ((T + 1) * BYTES_PER_TH + 8 * D["d"] * 6)
        self.desc = (f"append+fetch of {pre_rows} tokens x 32 sequence-heads of the prefill batch, and the "
                     f"decode-step attention of {seqs} sequences x {heads} kv-heads x 8 q-heads over 32769 rows")

    def run_once(self):
        o = self.oracle
        o.encode(self.planes, self.kp, self.vp)
        o.decode(self.planes, 0, self.pre_rows)
        for pl, q in self.att:
            o.attention(pl, q, DECODE["T"] + 1)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    cores = cpu_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    sample = OracleSample(pre_rows=256, seqs=1, heads=2)
    for _ in range(args.warmup):
        sample.run_once()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        sample.run_once()
        times.append(time.perf_counter() - t)
    per = sum(times) / len(times)
    value = sample.bytes / per / 1e9
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (same seeded streams)",
        "config": {"workload": "same as the CUDA arm, bounded sample per step", "sample": sample.desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample.desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def omp_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP regions from here on."""
    import ctypes

    import oracle

    oracle.lib()  # loads the OpenMP runtime the oracle links
    ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))


class LongContextOracleSample:
    """The long-context decode step's attention in the oracle for `seqs`
    sequences x 1 kv-head (8 q-heads each) over all 131073 rows (k4v3)."""

    def __init__(self, seqs: int):
        import oracle
        import tq_synth

        L = LONGCTX
        wl = tq_synth.WORKLOADS["longctx"]
        self.oracle = oracle
        self.items = []
        for b in range(seqs):
            k, v = tq_synth.host_kv(wl, B=1, H=1, n=L["T"] + 1, b_offset=b)
            pl = oracle.Planes(1, 1, L["d"], L["kb"], L["vb"], L["T"] + 16)
            oracle.encode(pl, k, v)
            q = tq_synth.host_q(wl, 0, B=1, QH=L["QH"] // L["H"], d=L["d"])
            self.items.append((pl, q))
            del k, v
        bpt = oracle.bytes_per_token_head(L["d"], L["kb"], L["vb"])
        self.bytes = seqs * ((L["T"] + 1) * bpt + (L["QH"] // L["H"]) * L["d"] * 6)
        self.desc = (f"long-context decode attention of {seqs} sequences x 1 kv-head x 8 q-heads over "
                     f"{L['T'] + 1} rows, k4v3")

    def run_once(self):
        for pl, q in self.items:
            self.oracle.attention(pl, q, LONGCTX["T"] + 1)


def _time_sample(sample, runs):
    t = time.perf_counter()
    for _ in range(runs):
        sample.run_once()
    dt = time.perf_counter() - t
    return runs * sample.bytes / dt / 1e9, dt


def cpu_baseline():
    cores = cpu_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    omp_threads(cores)
    # the whole step (all 8192 prefill rows, all 32 decode sequences), run twice:
    # ~12 s of oracle work on 16 cores (the oracle has nothing to warm up)
    sample = OracleSample(pre_rows=PREFILL["T"], seqs=DECODE["B"])
    runs = 2
    value, dt = _time_sample(sample, runs)
    line = {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{runs} passes of {sample.desc}", "seconds": round(dt, 2)}
    # one thread: a smaller slice of the same step
    small = OracleSample(pre_rows=512, seqs=1, heads=2)
    omp_threads(1)
    v1, dt1 = _time_sample(small, 1)
    line["single_thread"] = {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "sample": small.desc,
                             "seconds": round(dt1, 2)}
    # the long-context step's attention on all cores (16 q-head tasks)
    omp_threads(cores)
    lc = LongContextOracleSample(seqs=2)
    vl, dtl = _time_sample(lc, 1)
    line["long_context_attention"] = {"value": round(vl, 4), "unit": "GB/s", "cores": cores, "sample": lc.desc,
                                      "seconds": round(dtl, 2),
                                      "us_per_full_step": round(
                                          LONGCTX["B"] * LONGCTX["H"] / 2 * dtl * 1e6, 0)}
    return line


# ------------------------------------------------------------------ main
# ------------------------------------------------------------------ sweep of the other paths
def run_sweep(only=None):
    """Device-timed throughput of the paths beyond the headline step, each on
    inputs larger than L2: CUDA events on the launching stream around 20 calls
    after 3 warm-up calls, median.  GB/s counts the format bytes each call must
    move (cache rows read, outputs written)."""
    import torch

    import rotated_kv_cache_gb300 as tq
    import tq_synth

    torch.cuda.set_device(0)
    peak, kind = measured_peaks()
    st = torch.cuda.current_stream()

    def timed(fn, reps=20, rounds=3):
        # reps calls back to back between two events (a device spin queued
        # first and the full queue hide host launch time), median over rounds
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(PRIME_CYCLES)
            a.record(st)
            for _ in range(reps):
                fn()
            b.record(st)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / reps)
        return statistics.median(ts)

    tpeak, tkind = measured_bf16_tflops()

    def emit(kind_, config, us, nbytes, flops=None):
        gbs = nbytes / (us * 1e-6) / 1e9
        line = {"sweep": kind_, "config": config, "us": round(us, 2), "GB/s": round(gbs, 1),
                "frac": round(gbs / peak, 4), "peak": peak, "peak_kind": kind}
        if flops is not None:  # a contraction: its roofline is the tensor peak
            tf = flops / (us * 1e-6) / 1e12
            line.update({"TFLOP/s": round(tf, 1), "tensor_frac": round(tf / tpeak, 4), "tensor_peak": tpeak,
                         "tensor_peak_kind": tkind})
        print(json.dumps(line), flush=True)

    def filled_cache(B, H, d, T, kb, vb, w):
        cache = tq.Cache(B, H, d, T + (16 - T % 16) % 16, k_bits=kb, v_bits=vb)
        for b0 in range(B):
            k = torch.empty((1, H, T, d), dtype=torch.int16, device="cuda")
            v = torch.empty_like(k)
            tq_synth.device_kv(w, k, v, B=1, H=H, d=d, n=T, b_offset=b0)
            tq.tq_encode_append(cache.batch_slice(b0, 1), k.view(torch.bfloat16), v.view(torch.bfloat16), 0)
            del k, v
        return cache

    want = (lambda kind_: True) if not only else (lambda kind_: kind_ in only)
    w = tq_synth.WORKLOADS["decode"]
    H, T = 8, 32769
    for d, kb, vb, G in [] if not want("attention") else [(128, 8, 3, 8), (128, 4, 3, 8), (128, 4, 2, 8), (128, 8, 4, 8), (128, 5, 2, 8),
                         (128, 8, 3, 4), (128, 8, 3, 16), (64, 8, 3, 16), (64, 8, 3, 8), (256, 8, 3, 8), (64, 4, 3, 8),
                         (256, 4, 3, 8), (512, 4, 3, 4)]:
        bpt = tq.tq_bytes_per_token_head(d, kb, vb)
        B = max(1, round(4e8 / (H * T * bpt)))
        cache = filled_cache(B, H, d, T, kb, vb, w)
        q = torch.empty((B, G * H, d), dtype=torch.int16, device="cuda")
        tq_synth.device_q(w, 0, q, B=B, QH=G * H, d=d)
        qb = q.view(torch.bfloat16)
        out = torch.empty((B, G * H, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(tq.tq_attention_workspace_bytes(cache, G * H, T), dtype=torch.uint8, device="cuda")
        us = timed(lambda: tq.tq_decode_attention(cache, qb, T, out=out, workspace=ws))
        path = "specialised" if vb in (2, 3, 4) and kb in (8, 4) and d in (64, 128, 256) else "generic"
        emit("attention", {"B": B, "kv_heads": H, "rows": T, "d": d, "kb": kb, "vb": vb, "group": G, "kernel": path},
             us, B * H * T * bpt + B * G * H * d * 6)
        del cache, ws, out, q
    # long-context serving scale: 32 sequences x 8 kv-heads x 131072 cached rows
    # plus the appended one, k4v3 (4.56 GB packed), one decode step
    if want("long_context_attention"):
        wl = tq_synth.WORKLOADS["longctx"]
        B, Tl, G = wl.B, wl.T + 1, wl.QH // wl.H
        cache = filled_cache(B, wl.H, wl.d, Tl, wl.kb, wl.vb, wl)
        q = torch.empty((B, wl.QH, wl.d), dtype=torch.int16, device="cuda")
        tq_synth.device_q(wl, 0, q, B=B, QH=wl.QH, d=wl.d)
        qb = q.view(torch.bfloat16)
        out = torch.empty((B, wl.QH, wl.d), dtype=torch.float32, device="cuda")
        ws = torch.empty(tq.tq_attention_workspace_bytes(cache, wl.QH, Tl), dtype=torch.uint8, device="cuda")
        us = timed(lambda: tq.tq_decode_attention(cache, qb, Tl, out=out, workspace=ws))
        bpt = tq.tq_bytes_per_token_head(wl.d, wl.kb, wl.vb)
        emit("long_context_attention", {"B": B, "kv_heads": wl.H, "rows": Tl, "d": wl.d, "kb": wl.kb, "vb": wl.vb,
                                        "group": G, "kernel": "specialised"},
             us, B * wl.H * Tl * bpt + B * wl.QH * wl.d * 6)
        del cache, ws, out, q, qb
    # multi-token attention: chunks of M = 4 and 128 query rows (the page's
    # forward shapes) over a 32769-row cache.  The MMA work is 4 d flops per
    # (column, cache row), a column being one (query row, q-head).
    d, kb, vb, G, B = 128, 8, 3, 8, 8
    cache = filled_cache(B, H, d, T, kb, vb, w) if want("multi_token_attention") else None
    bpt = tq.tq_bytes_per_token_head(d, kb, vb)
    for M in (4, 128) if cache is not None else ():
        q = torch.empty((B, M * G * H, d), dtype=torch.int16, device="cuda")
        tq_synth.device_q(w, 0, q, B=B, QH=M * G * H, d=d)
        qb = q.view(torch.bfloat16).view(B, M, G * H, d)
        out = torch.empty((B, M, G * H, d), dtype=torch.float32, device="cuda")
        ws = torch.empty(tq.tq_multi_token_workspace_bytes(cache, G * H, M, T), dtype=torch.uint8, device="cuda")
        us = timed(lambda: tq.tq_multi_token_attention(cache, qb, T, out=out, workspace=ws))
        emit("multi_token_attention", {"B": B, "kv_heads": H, "rows": T, "d": d, "kb": kb, "vb": vb, "group": G,
                                       "m_queries": M}, us, B * H * T * bpt + B * M * G * H * d * 6,
             flops=4.0 * d * G * M * B * H * T)
        del q, qb, out, ws
    del cache
    # deferred fetch and un-rotation, row copies: prefill-shaped cache of 32768 rows
    if not any(want(k_) for k_ in ("rotated_fetch", "unrotate", "copy_rows", "clear_rows")):
        return
    pw = tq_synth.WORKLOADS["prefill"]
    B, H, T, d = 4, 8, 32768, 128
    cache = filled_cache(B, H, d, T, 8, 3, pw)
    vr = torch.empty((B, H, T, d), dtype=torch.bfloat16, device="cuda")
    us = timed(lambda: tq.tq_decode_values_rotated(cache, 0, T, dtype=torch.bfloat16, out=vr))
    if want("rotated_fetch"):
        emit("rotated_fetch", {"B": B, "kv_heads": H, "rows": T, "d": d, "vb": 3, "out": "bf16"}, us,
             B * H * T * (48 + 8 + d * 2))
    x = torch.randn((B * H * T // 4, d), dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    us = timed(lambda: tq.tq_unrotate(x, out=y))
    if want("unrotate"):
        emit("unrotate", {"rows": x.shape[0], "d": d, "in": "fp32", "out": "fp32"}, us, 2 * x.numel() * 4)
    del x, y, vr
    snap = tq.Cache(B, H, d, T)
    us = timed(lambda: tq.tq_cache_copy_rows(snap, 0, cache, 0, T))
    if want("copy_rows"):
        emit("copy_rows", {"B": B, "kv_heads": H, "rows": T, "d": d, "kb": 8, "vb": 3}, us, 2 * B * H * T * 200)
    us = timed(lambda: tq.tq_cache_clear_rows(snap, 0, T))
    if want("clear_rows"):
        emit("clear_rows", {"B": B, "kv_heads": H, "rows": T, "d": d, "kb": 8, "vb": 3}, us, B * H * T * 200)


PROFILE_CASES = {
    # name: (operation, head_dim, k_bits, v_bits, batch, kv-heads, rows, q-heads per kv-head)
    "prefill_codec": ("codec", 128, 8, 3, 4, 8, 8192, 0),
    "decode_attention_b1": ("attention", 128, 8, 3, 1, 8, 32769, 8),
    "decode_attention_b2": ("attention", 128, 8, 3, 2, 8, 32769, 8),
    "long_context_attention_b2": ("attention", 128, 4, 3, 2, 8, 131073, 8),
    "sweep_codec_d64_k8v3": ("codec", 64, 8, 3, 1, 8, 16384, 0),
    "sweep_codec_d512_k4v3": ("codec", 512, 4, 3, 1, 8, 16384, 0),
    "attention_d256_k8v3_b4": ("attention", 256, 8, 3, 4, 8, 32769, 8),
    "attention_d64_k8v3_b8": ("attention", 64, 8, 3, 8, 8, 32769, 8),
    "attention_d128_k8v4_b4": ("attention", 128, 8, 4, 4, 8, 32769, 8),
    "attention_group16_b2": ("attention", 128, 8, 3, 2, 8, 32769, 16),
    "generic_attention_d512_k4v3_b3": ("attention", 512, 4, 3, 3, 8, 32769, 4),
    # multi-token attention: M = 128 query rows per sequence (the tcgen05 kernel)
    "multi_token_m128_b2": ("multi128", 128, 8, 3, 2, 8, 32769, 8),
}


def run_profile_case(name: str, reps: int) -> None:
    """One small workload for a profiler capture: the cache (and inputs) are
    built, then the operation runs `reps` times (codec: encode then fetch to
    bf16; attention: one decode step's attention).  Prints nothing timed."""
    import torch

    from rotated_kv_cache_gb300 import build as libbuild

    libbuild.build()
    import rotated_kv_cache_gb300 as tq
    import tq_synth

    op, d, kb, vb, B, H, T, G = PROFILE_CASES[name]
    w = tq_synth.WORKLOADS["prefill" if op == "codec" and d == 128 else "sweep" if op == "codec" else "decode"]
    dev = torch.device("cuda", 0)
    cache = tq.Cache(B, H, d, T, kb, vb, device=dev)
    k = torch.empty((B, H, T, d), dtype=torch.int16, device=dev)
    v = torch.empty_like(k)
    tq_synth.device_kv(w, k, v, B=B, H=H, d=d, n=T)
    k16, v16 = k.view(torch.bfloat16), v.view(torch.bfloat16)
    tq.tq_encode_append(cache, k16, v16, 0)
    if op == "codec":
        ko, vo = torch.empty_like(k16), torch.empty_like(v16)
        for _ in range(reps):
            tq.tq_encode_append(cache, k16, v16, 0)
            tq.tq_decode(cache, 0, T, dtype=torch.bfloat16, k_out=ko, v_out=vo)
    elif op == "multi128":
        del k, v, k16, v16
        M = 128
        q = torch.empty((B, M * G * H, d), dtype=torch.int16, device=dev)
        tq_synth.device_q(w, 0, q, B=B, QH=M * G * H, d=d)
        qm = q.view(torch.bfloat16).view(B, M, G * H, d)
        out = torch.empty((B, M, G * H, d), dtype=torch.float32, device=dev)
        ws = torch.empty(tq.tq_multi_token_workspace_bytes(cache, G * H, M, T), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            tq.tq_multi_token_attention(cache, qm, T, out=out, workspace=ws)
    else:
        del k, v, k16, v16
        q = torch.empty((B, G * H, d), dtype=torch.int16, device=dev)
        tq_synth.device_q(w, 0, q, B=B, QH=G * H, d=d)
        out = torch.empty((B, G * H, d), dtype=torch.float32, device=dev)
        ws = torch.empty(tq.tq_attention_workspace_bytes(cache, G * H, T), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            tq.tq_decode_attention(cache, q.view(torch.bfloat16), T, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    print(json.dumps({"profile_case": name, "reps": reps, "ok": True}), flush=True)


def free_port() -> int:
    import socket

    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launcher_command(n: int, argv) -> list:
    """torch.distributed.run with one rank per GPU on this node, rendezvous on
    127.0.0.1, re-running this script with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the configurations beside the headline step (batch 1 and 8 decode, long context, "
                         "the codec sweep)")
    ap.add_argument("--decode-batch", type=int, default=DECODE["B"],
                    help="sequences of the decode step (smaller values for profiling captures)")
    ap.add_argument("--sweep", action="store_true",
                    help="measure the paths beyond the headline step instead (one JSON line each)")
    ap.add_argument("--only", default="",
                    help="with --sweep: comma-separated kinds to run (attention, long_context_attention, "
                         "multi_token_attention, rotated_fetch, unrotate, copy_rows, clear_rows)")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                    help="run one small workload `--reps` times for a profiler capture (no timing)")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.reps)
        return
    if args.sweep:
        run_sweep(set(filter(None, args.only.split(","))))
        return
    if args.warmup < 3:
        args.warmup = 3
    DECODE["B"] = args.decode_batch
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks under torch.distributed.run
        sys.exit(subprocess.call(launcher_command(args.gpus, sys.argv[1:])))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE is {world}: launch one rank per GPU")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    baseline = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        baseline = cpu_baseline()
    if rank == 0:
        line["cpu_baseline"] = baseline
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
