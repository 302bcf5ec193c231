#!/usr/bin/env python3
"""Benchmark of the attention forward on GB300.

One step = one fused prefill call (attn_fwd_prefill) on the headline workload, the
long-context GQA causal prefill (batch 1, 32 query heads over 8 kv heads, 32768 x 32768,
head_dim 128, bf16, 1% of Q elements scaled x8), with inputs resident in HBM.  The final
line also carries, end to end, the same call with host buffers (copies inside the timed
region), and a summary of the other hot-path workloads, each timed the same way and printed
in full on a line of its own before it: the tiny and the 2K prefills, the 8K head_dim-256
sliding-window prefill, the paged decode (split-KV + log-sum-exp combine) with 1 and 4 new
tokens, packed sequences, the attention sink, the FP8-e4m3 cache, and a windowed decode
with RoPE.  Each line carries the fp64 CPU oracle timed on the host cores beside it.

Timing: W untimed warm-up steps, then exactly K timed steps; every step is bracketed
by CUDA events on the launching stream, and between steps a 256 MiB buffer is written
(flushing the 129 MB L2) and another 256 MiB read (so the flush leaves no dirty line to be
written back inside the next step).  A barrier plus torch.cuda.synchronize() bracket the timed
region; with N > 1 ranks each rank runs its own replica and the max over ranks is used.
SM clocks are sampled with nvidia-smi while the timed regions run.

``--impl reference`` times the fp64 CPU oracle (the only reference that exists for this
path) on bounded samples of the headline workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
METRIC = "prefill attn TFLOPS & decode KV GB/s on 1\u00d7GB300 (fraction of roofline)"


# --------------------------------------------------------------------------- ranks
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(
        os.environ.get("LOCAL_RANK", 0))


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar across the job (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, seconds_per_rank: float, world: int, device=None):
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    slowest = max_over_ranks(seconds_per_rank, world, device)
    return units_per_rank * world / slowest, slowest


# --------------------------------------------------------------------------- peaks, clocks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"attn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        load = [x for x in sm if smax is None or x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- traffic record
def source_sha(*rel_paths) -> str:
    h = hashlib.sha256()
    for rel in rel_paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "prefill": ("flash_attention_forward_attn_gb300/csrc/prefill_sm103.cu",
                "flash_attention_forward_attn_gb300/csrc/attn_ptx.cuh"),
    # the decode launch shape (split length) is chosen in the API layer
    "decode": ("flash_attention_forward_attn_gb300/csrc/decode_sm103.cu",
               "flash_attention_forward_attn_gb300/csrc/attn_ptx.cuh",
               "flash_attention_forward_attn_gb300/csrc/api.cu",
               "flash_attention_forward_attn_gb300/csrc/attn_internal.h"),
}


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("source_sha") != source_sha(*KERNEL_SOURCES[kind]):
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- GPU timing
def check_device(stream, what):
    """Raise with the library's status if a kernel reported a device-side error."""
    import flash_attention_forward_attn_gb300 as A

    err = A.attn_get_device_error(stream)
    if err != 0:
        raise RuntimeError(f"{what}: device error {A.attn_status_string(err)}")


class L2Flush:
    """The L2 flush between timed steps: a write of L2_FLUSH_BYTES evicts every line the step
    read, then a read of another L2_FLUSH_BYTES writes the first buffer's dirty lines back.
    Without the read the L2 would start the timed step holding about its size in dirty lines
    of the flush buffer, whose write-back would fall inside the timed region (measured: 8 %
    of the 0.2 ms windowed decode)."""

    def __init__(self, dev):
        import torch

        self.write_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.read_buf = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self, i):
        self.write_buf.fill_(i & 0xFF)
        self.read_buf.sum()


L2_NOTE = (f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB written, then another "
           f"{L2_FLUSH_BYTES >> 20} MiB read so no dirty line is left)")


def time_steps(fn, steps, warmup, flush, stream):
    """Per-step device time (ms) with CUDA events on `stream`; L2 flushed before each step."""
    import torch

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush(i)
            fn()
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush(i)  # on the timing stream, outside the events
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def prefill_entry(w, dev, steps, warmup, flush, stream, peaks, world, e2e=False, sink=False,
                  cpu_threads=0):
    """Time attn_fwd_prefill on workload w (with sink=True: attn_fwd_prefill_ex with the
    per-head sink logits of workloads.configs.sink_logits).  cpu_threads > 0 also times the
    fp64 oracle on a bounded sample of the same inputs (after the GPU timing)."""
    import torch

    import flash_attention_forward_attn_gb300 as A
    from workloads import configs as C

    q, k, v = C.prefill_inputs_torch(w, dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16 if w.o_dtype == "bf16" else torch.float32,
                    device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    sk = torch.from_numpy(C.sink_logits(w.hq)).to(dev) if sink else None

    def step():
        if sink:
            A.attn_fwd_prefill_ex(q, k, v, causal=w.causal, window=w.window, scale=w.scale, o=o,
                                  lse=lse, sink=sk, stream=stream)
        else:
            A.attn_fwd_prefill(q, k, v, causal=w.causal, window=w.window, scale=w.scale, o=o,
                               lse=lse, stream=stream)

    ms = time_steps(step, steps, warmup, flush, stream)
    check_device(stream, w.name)
    mean_ms = sum(ms) / len(ms)
    flops = w.flops()
    value, slowest_s = aggregate_throughput(flops * steps, sum(ms) / 1e3, world, dev)
    tflops = value / 1e12
    achieved = flops / (mean_ms / 1e3) / 1e12
    traffic = None if sink else recorded_traffic("prefill", w.name)
    ent = {
        "workload": w.name + ("+sink" if sink else ""), "value": tflops, "unit": "TFLOP/s", "ms_per_step": mean_ms,
        "ms_min": min(ms), "flops_per_step": flops, "steps": steps, "gpu_launches": steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "traffic": traffic, "algorithmic_bytes": w.io_bytes(),
                     "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"},
        "slowest_rank_s": slowest_s,
    }
    if e2e:
        ent["e2e"] = prefill_e2e(w, q, k, v, o, lse, steps, warmup, stream, world, dev)
        check_device(stream, w.name + " (end to end)")
    if cpu_threads:
        ent["cpu_baseline"] = cpu_prefill(w, q, k, v, cpu_threads,
                                          C.sink_logits(w.hq) if sink else None)
    del q, k, v, o, lse
    torch.cuda.empty_cache()
    return ent


def packed_prefill_entry(pw, dev, steps, warmup, flush, stream, peaks, world, cpu_threads=0):
    """Time attn_fwd_prefill_ex on packed sequences (attn_opts.cu_seqlens)."""
    import torch

    import flash_attention_forward_attn_gb300 as A
    from workloads import configs as C

    w = pw.as_prefill()
    q, k, v = C.prefill_inputs_torch(w, dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    cu_q, cu_k = (torch.from_numpy(x).to(dev) for x in pw.offsets())

    def step():
        A.attn_fwd_prefill_ex(q, k, v, causal=True, scale=pw.scale, o=o, lse=lse,
                              cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, stream=stream)

    ms = time_steps(step, steps, warmup, flush, stream)
    check_device(stream, pw.name)
    mean_ms = sum(ms) / len(ms)
    flops = pw.flops()
    value, slowest_s = aggregate_throughput(flops * steps, sum(ms) / 1e3, world, dev)
    achieved = flops / (mean_ms / 1e3) / 1e12
    ent = {
        "workload": pw.name, "value": value / 1e12, "unit": "TFLOP/s", "ms_per_step": mean_ms,
        "ms_min": min(ms), "flops_per_step": flops, "steps": steps,
        "gpu_launches": 2 * steps,  # the work-order pass and the prefill kernel
        "packing": {"nseq": pw.nseq, "sq": w.sq, "skv": w.skv},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "traffic": recorded_traffic("prefill", pw.name),
                     "algorithmic_bytes": pw.io_bytes(),
                     "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"},
        "slowest_rank_s": slowest_s,
    }
    if cpu_threads:
        ent["cpu_baseline"] = cpu_packed(pw, q, k, v, cpu_threads)
    del q, k, v, o, lse
    torch.cuda.empty_cache()
    return ent


def prefill_e2e(w, q, k, v, o, lse, steps, warmup, stream, world, dev):
    """Same metric through the public API with host buffers: every step copies Q, K, V from
    pinned host memory, calls attn_fwd_prefill, and copies O and LSE back, all inside the
    timed region.  Steps are pipelined the way a serving loop would run them: two sets of
    device buffers, each input copied on its own stream (several copy engines), the call on
    `stream`, the results copied back on another stream, so step i+1's uploads overlap step
    i's call and download.  Events order each step's copies, call and download."""
    import torch

    import flash_attention_forward_attn_gb300 as A

    hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (q, k, v))
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in (hq_, hk_, hv_))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    dev_in = [(q, k, v)] + [tuple(torch.empty_like(x) for x in (q, k, v))]
    dev_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
    up = [torch.cuda.Stream(device=dev) for _ in range(3)]
    down = torch.cuda.Stream(device=dev)
    ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
    ev_call = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]  # a buffer set's download is done
    used = [False, False]

    def step(i):
        bset = i & 1
        din, (do_, dl) = dev_in[bset], dev_out[bset]
        for j, (dst, src) in enumerate(zip(din, (hq_, hk_, hv_))):
            if used[bset]:
                up[j].wait_event(ev_free[bset])  # the set's previous step is fully done
            with torch.cuda.stream(up[j]):
                dst.copy_(src, non_blocking=True)
            ev_in[bset][j].record(up[j])
        for j in range(3):
            stream.wait_event(ev_in[bset][j])
        A.attn_fwd_prefill(din[0], din[1], din[2], causal=w.causal, window=w.window,
                           scale=w.scale, o=do_, lse=dl, stream=stream)
        ev_call[bset].record(stream)
        down.wait_event(ev_call[bset])
        with torch.cuda.stream(down):
            ho[bset].copy_(do_, non_blocking=True)
            hl[bset].copy_(dl, non_blocking=True)
        ev_free[bset].record(down)
        used[bset] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(up[0])
    for j in (1, 2):
        up[j].wait_event(s)
    for i in range(steps):
        step(warmup + i)
    e.record(down)
    torch.cuda.synchronize()
    barrier(world)
    value, _ = aggregate_throughput(w.flops() * steps, s.elapsed_time(e) / 1e3, world, dev)
    return {"value": value / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": s.elapsed_time(e) / steps,
            "pipelining": "2 buffer sets; per-input upload streams; download stream"}


def rope_inv_freq(d):
    """RoPE inverse frequencies 10000^(-2i/d), i < d/2 (fp32)."""
    import numpy as np

    return np.array([10000.0 ** (-2.0 * i / d) for i in range(d // 2)], dtype=np.float32)


def decode_entry(w, dev, steps, warmup, flush, stream, peaks, world, sink=False, e4m3=False,
                 window=0, rope=False, kv_chunk=0, cpu_threads=0):
    """Time attn_fwd_decode on workload w (with sink=True: attn_fwd_decode_ex with the
    per-head sink logits of workloads.configs.sink_logits; with e4m3=True: attn_fwd_decode_ex
    over the same caches rounded to FP8-e4m3, k_scale = v_scale = 1; window > 0 and rope:
    attn_fwd_decode_ex with that window and RoPE of the queries, inverse frequencies
    10000^(-2i/d)).  cpu_threads > 0 also times the fp64 oracle on a sample of sequences."""
    import torch

    import flash_attention_forward_attn_gb300 as A
    from workloads import configs as C

    t = C.decode_inputs_e4m3_torch(w, dev) if e4m3 else C.decode_inputs_torch(w, dev)
    ws = torch.empty(A.attn_decode_workspace_bytes(w.b, w.hq, w.s_active, w.d, t["max_cache_len"],
                                                   kv_chunk), dtype=torch.uint8, device=dev)
    o = torch.empty(t["q"].shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=dev)
    sk = torch.from_numpy(C.sink_logits(w.hq)).to(dev) if sink else None
    args = (t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["cache_len"])
    inv = torch.from_numpy(rope_inv_freq(w.d)).to(dev) if rope else None

    def step():
        if sink or e4m3 or window or rope:
            A.attn_fwd_decode_ex(*args, max_cache_len=t["max_cache_len"], scale=w.scale, o=o,
                                 lse=lse, sink=sk, window=window, rope_inv_freq=inv,
                                 kv_chunk=kv_chunk, workspace=ws, stream=stream)
        else:
            A.attn_fwd_decode(*args, max_cache_len=t["max_cache_len"], scale=w.scale, o=o,
                              lse=lse, kv_chunk=kv_chunk, workspace=ws, stream=stream)

    ms = time_steps(step, steps, warmup, flush, stream)
    check_device(stream, w.name)
    mean_ms = sum(ms) / len(ms)
    nbytes = C.decode_io_bytes(w, t["lens"], kv_bytes=1 if e4m3 else 2, window=window) + (
        w.d // 2 * 4 if rope else 0)
    value, slowest_s = aggregate_throughput(nbytes * steps, sum(ms) / 1e3, world, dev)
    achieved = nbytes / (mean_ms / 1e3) / 1e9
    label = (w.name + ("+sink" if sink else "") + ("+e4m3" if e4m3 else "") +
             (f"+w{window}" if window else "") + ("+rope" if rope else ""))
    ent = {
        "workload": label, "value": value / 1e9, "unit": "GB/s", "ms_per_step": mean_ms,
        "ms_min": min(ms), "bytes_per_step": nbytes, "mean_cache_len": float(t["lens"].mean()),
        "steps": steps, "gpu_launches": 2 * steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("decode", label),
                     "timed": "whole call (split-KV kernel + combine kernel)",
                     "peak_source": f"{peaks['source']} HBM copy (MEASURED_PEAKS.json)"},
        "slowest_rank_s": slowest_s,
    }
    if cpu_threads:
        ent["cpu_baseline"] = cpu_decode(w, t, cpu_threads, C.sink_logits(w.hq) if sink else None,
                                         e4m3, window, rope_inv_freq(w.d) if rope else None)
    del t, ws, o, lse
    torch.cuda.empty_cache()
    return ent


# --------------------------------------------------------------------------- CPU oracle
# The fp64 oracle, as it stands, timed on the host cores beside each GPU line.  Its inputs
# are the seeded generator's values already made for the GPU timing, copied to the host (the
# same bits the kernels read); only the oracle calls are inside the timer.  Workloads whose
# full oracle run would take minutes are timed on a bounded sample and extrapolated at the
# measured rate (FLOPs for prefill, algorithmic bytes for decode), labelled as such.
SAMPLE_ROWS = 256     # query rows per sampled head
SAMPLE_HEADS = 8      # (batch, head) pairs sampled
FULL_PREFILL_FLOP = 5e10  # prefills up to this size are timed in full
DECODE_SAMPLE_SEQS = 2


def _bits(t):
    import numpy as np
    import torch

    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.uint8).cpu().numpy()


def _timed_pool(fn, jobs, threads):
    from concurrent.futures import ThreadPoolExecutor

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fn, jobs))
    return time.perf_counter() - t0


def _sample_rows(w, n, seed):
    """Rows 0 and sq-1, the 128-row tile boundaries around them and seeded uniform rows."""
    import numpy as np

    from workloads import rng

    if n >= w.sq:
        return np.arange(w.sq)
    rows = {0, w.sq - 1, 127, 128, 129, w.sq - 128, w.sq - 129}
    u = rng.uniform_np(rng.stream_seed(seed, "cpu_sample_rows"), 0, 4 * n)
    for x in (u * w.sq).astype(np.int64):
        if len(rows) >= n:
            break
        rows.add(int(x))
    return np.array(sorted(r for r in rows if 0 <= r < w.sq))


def cpu_prefill(w, q, k, v, threads, sink=None):
    """Oracle rows of prefill workload w: every row of every head when the workload is at
    most FULL_PREFILL_FLOP, else SAMPLE_ROWS rows of SAMPLE_HEADS heads."""
    import numpy as np

    import oracle

    full = w.flops() <= FULL_PREFILL_FLOP
    pairs = [(b, h) for b in range(w.b) for h in range(w.hq)]
    if not full:
        pick = np.linspace(0, len(pairs) - 1, SAMPLE_HEADS).round().astype(int)
        pairs = [pairs[i] for i in sorted(set(pick))]
    rows = np.arange(w.sq) if full else _sample_rows(w, SAMPLE_ROWS, w.seed)
    qp = rows + (w.skv - w.sq)
    hi = np.minimum(qp, w.skv - 1) if w.causal else np.full_like(qp, w.skv - 1)
    lo = np.maximum(0, qp - w.window + 1) if w.window > 0 else np.zeros_like(qp)
    flops = 4.0 * w.d * float(np.clip(hi - lo + 1, 0, None).sum()) * len(pairs)
    data = {}
    for (b, h) in pairs:
        g = oracle.kv_head(h, w.hq, w.hkv)
        data[(b, h)] = (_bits(q[b, h])[rows], _bits(k[b, g]), _bits(v[b, g]))
    jobs = [(p, s) for p in pairs for s in range(0, len(rows), 16)]

    def run(job):
        (b, h), s = job
        qr, kh, vh = data[(b, h)]
        oracle.attention_rows(qr[s:s + 16], kh, vh, qp[s:s + 16], w.scale, w.causal, w.window,
                              sink=None if sink is None else sink[h])

    secs = _timed_pool(run, jobs, threads)
    rate = flops / secs
    ent = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "seconds": secs}
    if full:
        ent["sample"] = f"all {w.b * w.hq} heads x {w.sq} rows (the whole workload)"
    else:
        ent["sample"] = (f"{len(pairs)} of {w.b * w.hq} heads x {len(rows)} rows (0, sq-1, tile "
                         f"boundaries, seeded uniform); rate over the sampled rows' allowed keys")
        ent["extrapolated_full_s"] = w.flops() / rate
    return ent


def cpu_packed(pw, q, k, v, threads):
    """Oracle rows of a packed prefill: SAMPLE_ROWS rows of two heads, each row against its
    own sequence's keys."""
    import numpy as np

    import oracle

    cu_q, cu_k = pw.offsets()
    w = pw.as_prefill()
    rows = _sample_rows(w, SAMPLE_ROWS, pw.seed)
    seq = np.searchsorted(cu_q, rows, side="right") - 1
    jobs, flops = [], 0.0
    for h in (0, pw.hq - 1):
        g = oracle.kv_head(h, pw.hq, pw.hkv)
        qh, kh, vh = _bits(q[0, h]), _bits(k[0, g]), _bits(v[0, g])
        for s in np.unique(seq):
            r = rows[seq == s]
            k0, k1 = int(cu_k[s]), int(cu_k[s + 1])
            qp = r - cu_q[s] + (k1 - k0) - (cu_q[s + 1] - cu_q[s])
            jobs.append((qh[r], kh[k0:k1], vh[k0:k1], qp))
            flops += 4.0 * pw.d * float(np.clip(np.minimum(qp, k1 - k0 - 1) + 1, 0, None).sum())

    def run(job):
        qr, kk, vv, qp = job
        oracle.attention_rows(qr, kk, vv, qp, pw.scale, True, 0)

    secs = _timed_pool(run, jobs, threads)
    rate = flops / secs
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": secs, "extrapolated_full_s": pw.flops() / rate,
            "sample": f"2 of {pw.hq} heads x {len(rows)} packed rows, each against its sequence"}


# Caches up to this size are copied to the host whole and the oracle decodes every
# sequence; larger ones are sampled (the first DECODE_SAMPLE_SEQS sequences).
DECODE_FULL_MAX_BYTES = 12 << 30


def cpu_decode(w, t, threads, sink=None, e4m3=False, window=0, inv_freq=None):
    """Oracle decode of the whole workload (every sequence and head, the caches copied to the
    host); for caches above DECODE_FULL_MAX_BYTES, of the first DECODE_SAMPLE_SEQS sequences
    (all heads, whole caches, gathered through their own compacted page table)."""
    import numpy as np
    import torch

    import oracle
    from workloads import configs as C

    cache_bytes = 2 * t["k_cache"].numel() * t["k_cache"].element_size()
    if cache_bytes <= DECODE_FULL_MAX_BYTES:
        n, lens, sub = w.b, t["lens"], t["table"]
        kc, vc = _bits(t["k_cache"]), _bits(t["v_cache"])
    else:
        n = min(DECODE_SAMPLE_SEQS, w.b)
        lens = t["lens"][:n]
        table = t["table"]
        npg = [-(-int(x) // w.page_size) for x in lens]
        pages = np.concatenate([table[b, :npg[b]] for b in range(n)]).astype(np.int64)
        idx = torch.from_numpy(pages).to(t["k_cache"].device)
        kc, vc = _bits(t["k_cache"][idx]), _bits(t["v_cache"][idx])
        sub = np.full((n, w.max_pages_per_seq), 0xFFFFFFFF, dtype=np.uint32)
        off = 0
        for b in range(n):
            sub[b, :npg[b]] = np.arange(off, off + npg[b], dtype=np.uint32)
            off += npg[b]
    qb = _bits(t["q"][:n])
    t0 = time.perf_counter()
    if e4m3:
        oracle.decode_e4m3(qb, kc, vc, sub, lens, w.scale, 1.0, 1.0, threads=threads, sink=sink)
    elif window or inv_freq is not None:
        oracle.decode_ext(qb, kc, vc, sub, lens, w.scale, window=window, inv_freq=inv_freq,
                          sink=sink, threads=threads)
    else:
        oracle.decode(qb, kc, vc, sub, lens, w.scale, threads=threads, sink=sink)
    secs = time.perf_counter() - t0
    nbytes = C.decode_io_bytes(w.with_(b=n), lens, kv_bytes=1 if e4m3 else 2, window=window)
    rate = nbytes / secs
    ent = {"value": rate / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "seconds": secs}
    if n == w.b:
        ent["sample"] = f"the whole workload: all {w.b} sequences and {w.hq} heads"
    else:
        full = C.decode_io_bytes(w, t["lens"], kv_bytes=1 if e4m3 else 2, window=window)
        ent["extrapolated_full_s"] = full / rate
        ent["sample"] = (f"{n} of {w.b} sequences (cache lens "
                         f"{', '.join(str(int(x)) for x in lens)}), all {w.hq} heads; rate over "
                         f"their algorithmic bytes")
    return ent


# --------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle on the host cores, rank 0 only, on bounded
    samples of the headline workload: each step is the last 16 query rows (the rows with
    the most keys) of one head."""
    import numpy as np

    import oracle
    from workloads import configs as C

    if rank != 0:
        return 0
    w = HEADLINE(C)
    threads = os.cpu_count() or 1
    rows = np.arange(w.sq - 16, w.sq)
    qp = rows + (w.skv - w.sq)
    kh = C.prefill_kv_head_np(w, "k", 0, 0)
    vh = C.prefill_kv_head_np(w, "v", 0, 0)
    qr = C.prefill_q_rows_np(w, 0, 0, int(rows[0]), len(rows))
    flops = 4.0 * w.d * float((np.minimum(qp, w.skv - 1) + 1).sum())

    def one_step():
        def run(s):
            oracle.attention_rows(qr[s:s + 1], kh, vh, qp[s:s + 1], w.scale, w.causal, w.window)

        return _timed_pool(run, range(len(rows)), threads)

    for _ in range(args.warmup):
        one_step()
    tot_s = sum(one_step() for _ in range(args.steps))
    value = flops * args.steps / tot_s / 1e12
    desc = (f"each step: head 0, the last {len(rows)} query rows of {w.name} (fp64, full "
            f"score rows, {threads} threads)")
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, 1),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def HEADLINE(C):
    """The headline workload: the largest single-GPU configuration, the 32K GQA prefill."""
    return C.GQA_PREFILL_32K


def workload_config(w, world):
    return {"workload": w.name, "b": w.b, "hq": w.hq, "hkv": w.hkv, "sq": w.sq, "skv": w.skv,
            "d": w.d, "causal": w.causal, "window": w.window, "o_dtype": w.o_dtype,
            "q_outliers": w.outlier_frac,
            "l2": L2_NOTE,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def compact(ent):
    """One workload's numbers in a few keys, for the summary at the end of the final line."""
    if "error" in ent:
        return {"error": ent["error"][:80]}
    out = {"v": round(ent["value"], 1), "u": ent["unit"], "ms": round(ent["ms_per_step"], 4),
           "frac": round(ent["roofline"]["frac"], 3)}
    cpu = ent.get("cpu_baseline")
    if cpu:
        out["cpu"] = float(f"{cpu['value']:.3g}")
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None,
                    help="time only this named workload (profiling runs); prints its entry")
    ap.add_argument("--sink", action="store_true",
                    help="with --workload: the _ex call with per-head attention-sink logits")
    ap.add_argument("--e4m3", action="store_true",
                    help="with a decode --workload: the caches rounded to FP8-e4m3")
    ap.add_argument("--window", type=int, default=0, help="with a decode --workload: a window")
    ap.add_argument("--rope", action="store_true", help="with a decode --workload: RoPE of Q")
    ap.add_argument("--kv-chunk", type=int, default=0, help="with a decode --workload: split length")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch

    import flash_attention_forward_attn_gb300 as A
    from workloads import configs as C

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    A.load_library()
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    # the oracle beside each line: rank 0 of a single-GPU run only
    cpu = (os.cpu_count() or 1) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else 0

    if args.workload is not None:
        wx = C.REGISTRY[args.workload]
        if isinstance(wx, C.PackedPrefillWorkload):
            ent = packed_prefill_entry(wx, dev, args.steps, args.warmup, flush, stream, peaks,
                                       world)
        elif isinstance(wx, C.PrefillWorkload):
            ent = prefill_entry(wx, dev, args.steps, args.warmup, flush, stream, peaks, world,
                                sink=args.sink)
        else:
            ent = decode_entry(wx, dev, args.steps, args.warmup, flush, stream, peaks, world,
                               sink=args.sink, e4m3=args.e4m3, window=args.window, rope=args.rope,
                               kv_chunk=args.kv_chunk)
        if rank == 0:
            print(json.dumps(ent), flush=True)
        return 0

    w = HEADLINE(C)
    extras = {}
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        main_ent = prefill_entry(w, dev, args.steps, args.warmup, flush, stream, peaks, world,
                                 e2e=True, cpu_threads=cpu)
        torch.cuda.synchronize()
        barrier(world)
        if not args.no_extra:
            ext_steps = max(10, min(args.steps, 30))
            dec_steps = max(ext_steps, 50)

            def pre(wx, **kw):
                return lambda: prefill_entry(wx, dev, ext_steps, args.warmup, flush, stream, peaks,
                                             world, cpu_threads=cpu, **kw)

            def dec(wx, **kw):
                return lambda: decode_entry(wx, dev, dec_steps, args.warmup, flush, stream, peaks,
                                            world, cpu_threads=cpu, **kw)

            runs = [
                # the five workloads of the problem statement
                (C.TINY_PREFILL.name, pre(C.TINY_PREFILL)),
                (C.CAUSAL_PREFILL_2K.name, pre(C.CAUSAL_PREFILL_2K)),
                (C.SWA_PREFILL_8K.name, pre(C.SWA_PREFILL_8K)),
                (C.PAGED_DECODE.name, dec(C.PAGED_DECODE)),
                (C.PAGED_DECODE_SPEC4.name, dec(C.PAGED_DECODE_SPEC4)),
                # packed sequences (attn_opts.cu_seqlens): 16 causal sequences with prefixes
                (C.PACKED_PREFILL.name, lambda: packed_prefill_entry(
                    C.PACKED_PREFILL, dev, ext_steps, args.warmup, flush, stream, peaks, world,
                    cpu_threads=cpu)),
                # the attention sink (attn_opts.sink) on the 2K prefill and the 1-token decode
                (C.CAUSAL_PREFILL_2K.name + "+sink", pre(C.CAUSAL_PREFILL_2K, sink=True)),
                (C.PAGED_DECODE.name + "+sink", dec(C.PAGED_DECODE, sink=True)),
                # the FP8-e4m3 KV cache (attn_opts.kv_dtype): half the cache bytes
                (C.PAGED_DECODE.name + "+e4m3", dec(C.PAGED_DECODE, e4m3=True)),
                (C.PAGED_DECODE_SPEC4.name + "+e4m3", dec(C.PAGED_DECODE_SPEC4, e4m3=True)),
                # a 4096-token window with RoPE of the queries (the pages' decode options)
                (C.PAGED_DECODE_SPEC4.name + "+w4096+rope",
                 dec(C.PAGED_DECODE_SPEC4, window=4096, rope=True)),
                # head_dim 256 decode
                (C.PAGED_DECODE_D256.name, dec(C.PAGED_DECODE_D256)),
            ]
            for label, run in runs:
                try:
                    ent = run()
                except RuntimeError as e:  # a device-side error report: keep the other lines
                    if world > 1:
                        raise  # ranks must stay in step for the collectives
                    torch.cuda.synchronize()
                    ent = {"workload": label, "error": str(e)}
                    print(f"bench: {label}: {e}", file=sys.stderr, flush=True)
                extras[ent["workload"]] = ent
                if rank == 0:  # each workload's full entry on a line of its own
                    print(json.dumps({"bench_workload": ent}), flush=True)
    clocks = clk.summary()

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": main_ent["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_ent["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) rounded to bf16; 1% of Q elements x8)",
            "config": workload_config(w, world),
            "roofline": main_ent["roofline"],
            "e2e": main_ent["e2e"],
            "gpu_launches": main_ent["gpu_launches"],
            "clocks": clocks,
            "cpu_baseline": main_ent.get("cpu_baseline"),
            # last, so that the end of the line carries every workload's numbers:
            # v = throughput, u = its unit, ms per call, frac = roofline fraction (of
            # measured peak), cpu = the oracle's rate on the host cores
            "workloads": {k: compact(e) for k, e in extras.items()},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
