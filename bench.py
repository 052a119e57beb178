#!/usr/bin/env python3
"""Benchmark of the ragged GQA fused attention forward on GB300.

One step = one trt_attention / trt_quantized_attention call over one batch of
the workload (device-side scheduler + the attention kernel).  The headline is
the ragged packed GQA prefill workload (8 sequences of 128-2048 tokens,
Hq=32, Hkv=8, D=128, bf16, upper_left causal) in TFLOP/s, with FLOPs = 4 * D
* attendable pairs counted exactly.  The other workloads (chunked context,
decode in KV GB/s over a 16-bit and an fp8 KV cache, tree decoding,
quantized P, the KV cache update) are reported under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Inputs are synthetic (seeded) and resident
in HBM for ``value``; ``e2e`` times the same call from pinned host buffers
with the host<->device copies inside the timed region.  L2 is flushed
between timed iterations (a 256 MiB write, then a 256 MiB read that leaves
no dirty lines behind).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ragged_gqa_attention_gb300 import binding, metrics  # noqa: E402
from ragged_gqa_attention_gb300 import workloads as W  # noqa: E402

HEADLINE = 2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


PROFILES = {   # headline kernel source and the ncu summary of it
    "prefill": ("ragged_gqa_attention_gb300/csrc/prefill.cuh",
                "profiles/prefill_kernel_packed_ragged_prefill_gqa32x8_d128_bf16.md"),
    "decode": ("ragged_gqa_attention_gb300/csrc/decode.cuh",
               "profiles/decode_kernel_decode_b64_gqa64x8_kv4096_d128_bf16.md"),
}


def profile_traffic(kind):
    """DRAM bytes per launch (read + write) from the committed ncu summary, or
    None when the kernel source has changed since that capture."""
    import hashlib
    import re
    src, md = (os.path.join(ROOT, x) for x in PROFILES[kind])
    try:
        text = open(md).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    m_sha = re.search(r"sha256 ([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic \(read \+ write\) \| ([0-9.]+) MB", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1)) * 1e6


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class Runner:
    """One prepared call on device-resident inputs (arguments built once)."""

    def __init__(self, dc: W.Case, stream):
        import ctypes
        self.ctypes = ctypes
        self.lib = binding.load()
        self.dc = dc
        self.stream = stream
        self.y = torch.empty_like(dc.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dc.q.device)
        paged = dc.kv_form == W.PAGED
        a = binding.make_args(dc.q, dc.k, dc.v, self.y, q_form=dc.q_form,
                              kv_form="padded" if paged else dc.kv_form,
                              query_lengths=dc.query_lengths, kv_lengths=dc.kv_lengths,
                              mask=dc.mask, scale=dc.scale, causal=dc.causal, norm=dc.norm,
                              status=self.status, batch=dc.batch)
        self.pk = None
        if paged:
            ks, vs = dc.kv_scales if dc.kv_scales is not None else (None, None)
            self.pk = binding.make_paged(dc.k, dc.v, dc.page_table, k_scale=ks, v_scale=vs)
            a.kv_seq = self.pk.max_pages_per_seq * self.pk.page_size
        n = self.lib.rga_attention_workspace_size(ctypes.byref(a))
        self.ws = torch.empty(n, dtype=torch.uint8, device=dc.q.device)
        a.workspace, a.workspace_bytes = self.ws.data_ptr(), n
        self.args = a
        self.h = ctypes.c_void_p(stream.cuda_stream)
        if dc.quant is not None:
            self.qt = binding.QUANT[dc.quant]
            self.qs = ctypes.c_void_p(dc.quant_scale.data_ptr())
            self.qsd = binding.DTYPES[dc.quant_scale.dtype]
        if dc.kv_scales is not None:
            self.ks = ctypes.c_void_p(dc.kv_scales[0].data_ptr())
            self.vs = ctypes.c_void_p(dc.kv_scales[1].data_ptr())

    def __call__(self):
        b = self.ctypes.byref(self.args)
        if self.pk is not None:
            rc = self.lib.trt_attention_paged_kv(b, self.ctypes.byref(self.pk), self.h)
        elif self.dc.kv_scales is not None:
            rc = self.lib.trt_attention_fp8_kv(b, self.ks, self.vs, self.h)
        elif self.dc.quant is None:
            rc = self.lib.trt_attention(b, self.h)
        else:
            rc = self.lib.trt_quantized_attention(b, self.qt, self.qs, self.qsd, self.h)
        if rc != 0:
            raise binding.RgaError(rc, "bench call")

    def check_status(self):
        torch.cuda.synchronize()
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError(f"device status {binding.STATUS_NAMES.get(st, st)}")


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x, dist_on):
    """Largest x over the ranks (a time: the slowest rank sets the step)."""
    if not dist_on:
        return x
    nccl = torch.distributed.get_backend() == "nccl"   # NCCL reduces device tensors only
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if nccl else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def device_timed(run, stream, steps, warmup, dist_on, sampler_index=None):
    """Per-step CUDA-event durations (ms) with an L2 flush between steps.

    The flush writes a 256 MiB buffer (twice L2) and then reads another one,
    so that each timed call starts with none of its inputs in L2 and without
    the flush's dirty lines, whose write-back would otherwise be charged to
    the call."""
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")   # 256 MiB
    clean = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device="cuda")   # 256 MiB
    sink = torch.empty((), dtype=torch.float32, device="cuda")   # 0-d: the sum's shape

    def l2_flush():
        flush.zero_()
        torch.sum(clean, dim=0, out=sink)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            l2_flush()
            run()
    barrier(dist_on)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    if sampler:
        sampler.__enter__()
    with torch.cuda.stream(stream):
        for s, e in ev:
            l2_flush()
            s.record(stream)
            run()
            e.record(stream)
    barrier(dist_on)
    if sampler:
        sampler.__exit__(None, None, None)
    times = [s.elapsed_time(e) for s, e in ev]
    return times, (sampler.summary() if sampler else None)


UPLOAD_STREAMS = 1


def h2d_peak_gbs(nbytes=512 << 20, streams=(1, UPLOAD_STREAMS), reps=3):
    """Best pinned copy rates of this machine (GB/s): host->device with one large
    buffer split evenly over 1 or several copy streams, device->host, and
    both directions at once: the link the e2e number is judged against."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = {}
    for ns in streams:
        ss = [torch.cuda.Stream() for _ in range(ns)]
        chunk = nbytes // ns
        best = 0.0
        for _ in range(reps):
            start = torch.cuda.Event(enable_timing=True)
            ends = [torch.cuda.Event(enable_timing=True) for _ in ss]
            torch.cuda.synchronize()
            start.record(ss[0])
            for i, st in enumerate(ss):
                st.wait_event(start)
                with torch.cuda.stream(st):
                    dst[i * chunk:(i + 1) * chunk].copy_(src[i * chunk:(i + 1) * chunk],
                                                         non_blocking=True)
                ends[i].record(st)
            torch.cuda.synchronize()
            ms = max(start.elapsed_time(e) for e in ends)
            best = max(best, nbytes / (ms * 1e-3) / 1e9)
        out[f"{ns}_stream" + ("s" if ns > 1 else "")] = round(best, 1)
    # device->host alone, and both directions at once (as in the e2e loop,
    # whose uploads and downloads overlap): host->device into one half of
    # the device buffer while the other half goes back, bytes of both over
    # the time of both
    back = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    half = nbytes // 2
    best_d2h = best_both = 0.0
    for _ in range(reps):
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(down)
        with torch.cuda.stream(down):
            back.copy_(dst, non_blocking=True)
        end.record(down)
        torch.cuda.synchronize()
        best_d2h = max(best_d2h, nbytes / (start.elapsed_time(end) * 1e-3) / 1e9)
        start = torch.cuda.Event(enable_timing=True)
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        start.record(up)
        down.wait_event(start)
        with torch.cuda.stream(up):
            dst[:half].copy_(src[:half], non_blocking=True)
        ends[0].record(up)
        with torch.cuda.stream(down):
            back[half:].copy_(dst[half:], non_blocking=True)
        ends[1].record(down)
        torch.cuda.synchronize()
        ms = max(start.elapsed_time(e) for e in ends)
        best_both = max(best_both, 2 * half / (ms * 1e-3) / 1e9)
    out["d2h_1_stream"] = round(best_d2h, 1)
    out["both_directions"] = round(best_both, 1)
    del src, dst, back
    return out


def e2e_timed(case: W.Case, stream, steps, warmup, dist_on):
    """The public call from pinned host buffers, every step: H2D of all its
    inputs, the attention call, D2H of Y.  Steps are pipelined over two sets
    of device buffers and streams for uploads (each input split evenly over
    UPLOAD_STREAMS copy streams), calls and downloads, so that step i+1's
    upload and step i-1's download overlap step i's call, as a serving loop
    would run them; each step still moves all its own bytes.
    Returns (ms per step over the timed steps, bytes in, bytes out)."""
    host = {}
    for name in ("q", "k", "v", "query_lengths", "kv_lengths", "mask", "quant_scale",
                 "page_table"):
        t = getattr(case, name)
        host[name] = None if t is None else t.pin_memory()
    if case.kv_scales is not None:   # fp8 KV cache: the two dequantisation scales
        for i, t in enumerate(case.kv_scales):
            host[f"kv_scale{i}"] = t.pin_memory()
    sets = []
    for _ in range(2):
        dev = {n: (None if t is None else torch.empty_like(t, device="cuda"))
               for n, t in host.items()}
        fields = {n: t for n, t in dev.items() if not n.startswith("kv_scale")}
        if case.kv_scales is not None:
            fields["kv_scales"] = (dev["kv_scale0"], dev["kv_scale1"])
        run = Runner(W.Case(**{**case.__dict__, **fields}), stream)
        y_host = torch.empty(case.q.shape, dtype=case.q.dtype).pin_memory()
        sets.append((dev, run, y_host))
    ups = [torch.cuda.Stream() for _ in range(UPLOAD_STREAMS)]
    up = ups[0]
    down = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    uploaded = [[ev() for _ in ups], [ev() for _ in ups]]
    computed, downloaded = [ev(), ev()], [ev(), ev()]
    used = [False, False]
    # each input in UPLOAD_STREAMS contiguous byte ranges, one per copy stream
    parts = {}
    for n, t in host.items():
        if t is None:
            continue
        nb = t.numel() * t.element_size()
        cut = [(nb * k // UPLOAD_STREAMS) // 16 * 16 for k in range(UPLOAD_STREAMS)] + [nb]
        parts[n] = cut

    def step(i):
        b = i % 2
        dev, run, y_host = sets[b]
        if used[b]:   # buffers b were last used by step i-2
            for u in ups:
                u.wait_event(computed[b])
            stream.wait_event(downloaded[b])
        for k, u in enumerate(ups):
            with torch.cuda.stream(u):
                for n, t in host.items():
                    if t is None:
                        continue
                    lo, hi = parts[n][k], parts[n][k + 1]
                    if hi > lo:
                        dst = dev[n].view(-1).view(torch.uint8)
                        src = t.view(-1).view(torch.uint8)
                        dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                uploaded[b][k].record(u)
        for k in range(len(ups)):
            stream.wait_event(uploaded[b][k])
        with torch.cuda.stream(stream):
            run()
            computed[b].record(stream)
        down.wait_event(computed[b])
        with torch.cuda.stream(down):
            y_host.copy_(run.y, non_blocking=True)
            downloaded[b].record(down)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(dist_on)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for u in ups[1:]:
        u.wait_event(t0)
    for i in range(warmup, warmup + steps):
        step(i)
    last = (warmup + steps - 1) % 2
    down.wait_event(downloaded[last])
    t1.record(down)
    torch.cuda.synchronize()
    barrier(dist_on)
    for _, run, _ in sets:
        run.check_status()
    bi = metrics.input_bytes(case)
    bo = case.q.numel() * case.q.element_size()
    return t0.elapsed_time(t1) / steps, bi, bo


def oracle_sample(case: W.Case, budget_s: float, max_units=None, threads=None):
    """Time the CPU oracle, as it stands, on whole sequences of the workload
    (all heads), shortest first, until ``budget_s`` seconds have been spent,
    with ``threads`` worker threads (default: one per host core).  Returns
    (work done, seconds, threads, description); work is FLOPs, or decode
    bytes for a decode workload."""
    import oracle   # the CPU baseline leg is one of the oracle's permitted users
    if case.kv_form == W.PAGED:   # the oracle reads the gathered (linear) cache
        case = W.Case(**{**case.__dict__, "kv_form": W.PADDED, "page_table": None,
                         "k": oracle.gather_pages(case.k, case.page_table, 0, case.kv_lens),
                         "v": oracle.gather_pages(case.v, case.page_table, 1, case.kv_lens)})
    order = sorted(range(case.batch), key=lambda b: (case.q_lens[b] * case.kv_lens[b], b))
    threads = threads or os.cpu_count() or 1
    done_flops, spent, seqs = 0.0, 0.0, []
    for b in order:
        sub = single_sequence(case, b)
        if metrics.flops(sub) == 0:
            continue
        f = metrics.decode_bytes(sub) if metrics.is_decode(case) else metrics.flops(sub)
        t0 = time.perf_counter()
        oracle.attention(sub.q, sub.k, sub.v, q_form=sub.q_form, kv_form=sub.kv_form,
                         query_lengths=sub.query_lengths, kv_lengths=sub.kv_lengths,
                         mask=sub.mask, scale=sub.scale, causal=sub.causal, norm=sub.norm,
                         quant=sub.quant, quant_scale=sub.quant_scale, nthreads=threads,
                         kv_fp8_scales=sub.kv_scales)
        spent += time.perf_counter() - t0
        done_flops += f
        seqs.append(b)
        if spent >= budget_s or (max_units and len(seqs) >= max_units):
            break
    desc = (f"sequences {seqs} of {case.name} (all {case.q_heads} query heads each), "
            f"oracle fp64 C with {threads} threads")
    return done_flops, spent, threads, desc


def single_sequence(case: W.Case, b: int) -> W.Case:
    """Sequence b of a case as a batch of one (layout slicing only)."""
    ql, kl = case.q_lens[b], case.kv_lens[b]
    if case.q_form == W.PACKED:
        o = int(case.query_lengths[b])
        q, qlen = case.q[o:o + ql], torch.tensor([0, ql], dtype=torch.int32)
    else:
        q = case.q[b:b + 1]
        qlen = None if case.query_lengths is None else torch.tensor([0, ql], dtype=torch.int32)
    if case.kv_form == W.PACKED:
        o = int(case.kv_lengths[b])
        k, v, klen = case.k[o:o + kl], case.v[o:o + kl], torch.tensor([0, kl], dtype=torch.int32)
    else:
        k, v = case.k[b:b + 1], case.v[b:b + 1]
        klen = None if case.kv_lengths is None else torch.tensor([kl], dtype=torch.int32)
    mask = case.mask
    if mask is not None:
        m = mask.reshape((1,) * (4 - mask.dim()) + tuple(mask.shape))
        mask = m[b:b + 1] if m.shape[0] > 1 else m
    return W.Case(**{**case.__dict__, "q": q, "k": k, "v": v, "batch": 1,
                     "query_lengths": qlen, "kv_lengths": klen, "q_lens": [ql],
                     "kv_lens": [kl], "mask": mask})


def measure(index, quant, stream, steps, warmup, dist_on, peaks, rank, clocks=False):
    """Device-timed throughput of one workload (inputs resident in HBM)."""
    case = W.workload(index, quant=quant, kv_pad=0.0)
    dc = W.to_device(case, "cuda")
    run = Runner(dc, stream)
    times, clk = device_timed(run, stream, steps, warmup, dist_on,
                              sampler_index=(torch.cuda.current_device() if clocks else None))
    run.check_status()
    ms = max_over_ranks(statistics.mean(times), dist_on)
    dec = metrics.is_decode(case)
    if dec:
        work, unit, bound = metrics.decode_bytes(case), "GB/s", "hbm"
        value = work / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
    else:
        work, unit, bound = metrics.flops(case), "TFLOP/s", "tensor"
        value = work / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
    return dict(case=case, ms=ms, value=value, unit=unit, bound=bound, peak=peak, work=work,
                clocks=clk, launches_per_step=2, times=times)


def measure_kv_update(stream, steps, warmup, dist_on, peaks):
    """TRT_KVCacheUpdate in place: the chunked-prefill workload's new K rows
    (packed, one chunk per sequence) written into its padded 8192-key cache
    at the chunk's positions.  GB/s of the update rows read and written."""
    import ctypes
    c = W.workload(3, kv_pad=0.0)
    g = torch.Generator().manual_seed(3)
    cache = c.k.to("cuda")                                   # [16, 8, 8192, 128]
    upd = torch.randn(sum(c.q_lens), c.kv_heads, c.head_dim, generator=g).to(c.k.dtype).cuda()
    cu = torch.zeros(c.batch + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(c.q_lens), 0)
    wi = torch.tensor([kl - ql for ql, kl in zip(c.q_lens, c.kv_lens)], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = binding.load()
    wi_d, cu_d = wi.cuda(), cu.cuda()      # referenced for as long as `a` is used
    a = binding.make_kv_args(cache, upd, cache, update_form="packed", write_indices=wi_d,
                             update_lengths=cu_d, status=status)
    h = ctypes.c_void_p(stream.cuda_stream)

    def run():
        rc = lib.trt_kv_cache_update(ctypes.byref(a), h)
        if rc != 0:
            raise binding.RgaError(rc, "bench kv update")

    times, _ = device_timed(run, stream, steps, warmup, dist_on)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"kv update device status {int(status.item())}")
    ms = max_over_ranks(statistics.mean(times), dist_on)
    work = 2 * upd.numel() * upd.element_size()
    value = work / (ms * 1e-3) / 1e9
    name = f"kv_cache_update_packed{upd.shape[0]}_into_b16_h8_n8192_d128_bf16"
    return name, dict(value=value, unit="GB/s", ms=ms, bound="hbm", peak=peaks["hbm_gbs"],
                      work=work)


def measure_rope_kv_update(stream, steps, warmup, dist_on, peaks):
    """RoPE fused with the KV cache update: the chunked-prefill workload's new
    K rows (packed, one chunk per sequence) rotated into its padded 8192-key
    cache at the chunk's positions, and its 4430 x 32-head Q rotated in
    place, in one launch.  GB/s of the rows read and written (Q twice, the
    new keys read and written, the cos/sin table read)."""
    import ctypes
    c = W.workload(3, kv_pad=0.0)
    g = torch.Generator().manual_seed(3)
    cache = c.k.to("cuda")
    T = sum(c.q_lens)
    upd = torch.randn(T, c.kv_heads, c.head_dim, generator=g).to(c.k.dtype).cuda()
    q = c.q.to("cuda")
    cu = torch.zeros(c.batch + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(c.q_lens), 0)
    wi = torch.tensor([kl - ql for ql, kl in zip(c.q_lens, c.kv_lens)], dtype=torch.int32)
    pos = torch.cat([torch.arange(w, w + ql) for w, ql in zip(wi.tolist(), c.q_lens)]).to(torch.int32)
    cs = W.rope_cos_sin(pos, c.head_dim).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = binding.load()
    wi_d, cu_d, pos_d = wi.cuda(), cu.cuda(), pos.cuda()   # referenced while `a`, `r` are used
    a = binding.make_kv_args(cache, upd, cache, update_form="packed", write_indices=wi_d,
                             update_lengths=cu_d, status=status)
    r = binding.make_rope_args(q, None, cs, pos_d, kv_heads=c.kv_heads)
    r.dtype, r.head_dim = a.dtype, c.head_dim
    h = ctypes.c_void_p(stream.cuda_stream)

    def run():
        rc = lib.trt_kv_cache_update_rope(ctypes.byref(a), ctypes.byref(r), h)
        if rc != 0:
            raise binding.RgaError(rc, "bench rope kv update")

    times, _ = device_timed(run, stream, steps, warmup, dist_on)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"rope kv update device status {int(status.item())}")
    ms = max_over_ranks(statistics.mean(times), dist_on)
    work = 2 * (q.numel() + upd.numel()) * q.element_size() + cs.numel() * 4
    value = work / (ms * 1e-3) / 1e9
    name = f"rope_kv_cache_update_packed{T}_q32_into_b16_h8_n8192_d128_bf16"
    return name, dict(value=value, unit="GB/s", ms=ms, bound="hbm", peak=peaks["hbm_gbs"],
                      work=work)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=HEADLINE)
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads (headline only)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle CPU work for cpu_baseline")
    ap.add_argument("--quant", choices=["fp8", "int8"], default="fp8",
                    help="P's quantisation when --workload is the quantized workload (5)")
    ap.add_argument("--aux", choices=["kv_update", "rope_kv_update"],
                    help="time only this cache-update kernel and print its line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    torch.cuda.set_device(local)
    if dist_on:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    binding.load(build_if_missing=(rank == 0))
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()

    if args.aux:
        fn = measure_kv_update if args.aux == "kv_update" else measure_rope_kv_update
        name, r = fn(stream, args.steps, args.warmup, dist_on, peaks)
        if rank == 0:
            print(json.dumps({"metric": f"{args.aux} GB/s", "value": round(r["value"] * world, 3),
                              "unit": r["unit"], "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": round(r["ms"], 4),
                              "config": {"workload": name},
                              "frac_of_peak": round(r["value"] / r["peak"], 4),
                              "peak": r["peak"], "peak_source": peak_src}), flush=True)
        if dist_on:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return

    head = measure(args.workload, args.quant, stream, args.steps, args.warmup, dist_on, peaks, rank,
                   clocks=True)
    case = head["case"]
    e2e_step_ms, bi, bo = e2e_timed(case, stream, max(3, args.steps // 2), 3, dist_on)
    h2d_peak = h2d_peak_gbs()
    e2e_ms = max_over_ranks(e2e_step_ms, dist_on)
    scale = 1e12 if head["unit"] == "TFLOP/s" else 1e9
    e2e_val = head["work"] / (e2e_ms * 1e-3) / scale

    secondary = {}
    if not args.no_secondary:
        for idx, q in ((3, "fp8"), (4, "fp8"), (5, "fp8"), (5, "int8"), (6, "fp8"), (7, "fp8"),
                       (8, "fp8"), (9, "fp8"), (10, "fp8")):
            if idx == args.workload:
                continue
            torch.cuda.empty_cache()
            r = measure(idx, q, stream, max(5, args.steps // 2), 3, dist_on, peaks, rank)
            secondary[r["case"].name] = {
                "value": round(r["value"] * world, 3), "unit": r["unit"],
                "ms_per_step": round(r["ms"], 4), "bound": r["bound"],
                "frac_of_peak": round(r["value"] / r["peak"], 4),
                "peak": r["peak"], "peak_source": peak_src}
            del r
        torch.cuda.empty_cache()
        for fn in (measure_kv_update, measure_rope_kv_update):
            torch.cuda.empty_cache()
            name, r = fn(stream, max(5, args.steps // 2), 3, dist_on, peaks)
            secondary[name] = {
                "value": round(r["value"] * world, 3), "unit": r["unit"],
                "ms_per_step": round(r["ms"], 4), "bound": r["bound"],
                "frac_of_peak": round(r["value"] / r["peak"], 4),
                "peak": r["peak"], "peak_source": peak_src}

    cpu = None
    if rank == 0:
        # the oracle with one thread per host core, then single-threaded
        f, s, thr, desc = oracle_sample(case, args.cpu_budget)
        f1, s1, _, desc1 = oracle_sample(case, args.cpu_budget / 2, threads=1)
        cpu = {"value": (f / s / scale) if s > 0 else None, "unit": head["unit"],
               "cores": thr, "kind": "oracle", "sample": desc, "seconds": round(s, 2),
               "single_thread": {"value": (f1 / s1 / scale) if s1 > 0 else None,
                                 "unit": head["unit"], "cores": 1, "sample": desc1,
                                 "seconds": round(s1, 2)}}

    if rank == 0:
        value = head["value"] * world
        line = {
            "metric": "attention TFLOP/s (prefill) / KV-read GB/s (decode) and % of roofline, 1 GB300",
            "value": round(value, 3), "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(head["ms"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": str(case.q.dtype).replace("torch.", ""),
            "data": "synthetic (seeded N(0,1) inputs, seeded lengths)",
            "config": {"workload": case.name, "batch": case.batch, "q_heads": case.q_heads,
                       "kv_heads": case.kv_heads, "head_dim": case.head_dim,
                       "q_tokens": sum(case.q_lens), "kv_tokens": sum(case.kv_lens),
                       "causal": case.causal, "l2": "flushed between steps (256 MiB written, then 256 MiB read)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": head["bound"], "achieved": round(head["value"], 3),
                         "peak": head["peak"], "unit": head["unit"],
                         "frac": round(head["value"] / head["peak"], 4),
                         "traffic": profile_traffic("decode" if metrics.is_decode(case)
                                                    else "prefill"),
                         "peak_source": peak_src,
                         "note": "achieved = algorithmic work / CUDA-event time of the whole "
                                 "call (scheduler + attention kernel)"},
            "e2e": {"value": round(e2e_val * world, 3), "unit": head["unit"],
                    "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                    "ms_per_step": round(e2e_ms, 4),
                    "h2d_gbs_achieved": round(bi / (e2e_ms * 1e-3) / 1e9, 1),
                    "h2d_peak_gbs": h2d_peak, "upload_streams": UPLOAD_STREAMS},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": head["clocks"],
            "cpu_baseline": cpu,
            "workloads": secondary,
        }
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample (whole sequences of the workload) timed on the CPU."""
    if rank != 0:
        return
    case = W.workload(args.workload, kv_pad=0.0)
    for _ in range(args.warmup):
        oracle_sample(case, 0.0, max_units=1)
    flops = secs = 0.0
    thr, desc = 1, ""
    for _ in range(args.steps):
        f, s, thr, desc = oracle_sample(case, 0.0, max_units=1)
        flops += f
        secs += s
    unit, div = ("GB/s", 1e9) if metrics.is_decode(case) else ("TFLOP/s", 1e12)
    val = flops / secs / div if secs > 0 else None
    line = {"impl": "reference", "metric": "attention TFLOP/s (prefill) / KV-read GB/s (decode) "
            "and % of roofline, 1 GB300", "value": val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / max(args.steps, 1) * 1e3, "higher_is_better": True,
            "config": {"workload": case.name}, "dtype": "f64",
            "cpu_baseline": {"value": val, "unit": unit, "cores": thr, "kind": "oracle",
                             "sample": desc + " per step"},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
