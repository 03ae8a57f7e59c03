#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on one GB300.

One step = one decode step of a Qwen3-0.6B-shaped model over a batch of 256
sequences with contexts uniform in [1024, 8192] tokens and all 28 layers'
KV caches resident in HBM (separate per-layer pools, block size 256): for
each layer, kv_store of the step's new token then paged decode attention.
Inputs total ~139 GB, far larger than L2, so no flush is needed between steps.

Printed (one JSON line, rank 0):
  value        algorithmic HBM bytes of the whole step (store + decode, 28 layers) / step time, GB/s
  roofline     the dominant kernel (paged decode) against the measured HBM copy peak, with its
               ncu DRAM traffic per launch while the decode sources match the recorded capture
  e2e          the same metric through the public API with host buffers (H2D inputs, D2H outputs)
  clocks       nvidia-smi SM clock and throttle reasons sampled inside the timed region
  gpu_launches this library's kernel launches inside the timed region
  prefill, prefill_long_history
               the varlen prefill row (16-sequence prefix-cached chunked batch; one sequence
               with a 16k-token history), TFLOP/s against the measured bf16 peak
  decode_b32   one layer of the batch-32 decode (contexts uniform in [128, 2048]), L2 flushed
  long_context, verify, kv_store, copy_blocks, cuda_graph_decode, fp8_kv
               the other rows: long-context split decode, speculative verify (q_len 4), the
               store alone, copy-on-write block copies, the batch-8 step replayed as a CUDA
               graph, and the step over an E4M3 cache
  cpu_baseline the CPU oracle on every host core (all sequences of layer 0), with a one-thread figure

``--impl reference`` times the CPU oracle itself on bounded samples of the
same workload (there is no other reference implementation of this path).
"""

from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")  # one thread per oracle process; the parallel oracle uses one process per core

import argparse
import datetime
import hashlib
import json
import math
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s"
UNIT = "GB/s"


# ---------------------------------------------------------------- distributed plumbing

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local, backend):
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- peaks and clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons; the summary keeps
    the samples stamped inside the timed region (mark() before it, mark() after it)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.marks = []
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        sel = self._selector(device_index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"] + sel, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @staticmethod
    def _selector(device_index: int):
        try:
            props = torch.cuda.get_device_properties(device_index)
            bus = getattr(props, "pci_bus_id", None)
            dom = getattr(props, "pci_domain_id", 0)
            dev = getattr(props, "pci_device_id", 0)
            if bus is not None:
                return ["-i", f"{dom:08x}:{bus:02x}:{dev:02x}.0"]
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return ["-i", vis.split(",")[device_index]]
        return ["-i", str(device_index)]

    def mark(self) -> None:
        """Host wall-clock time of the start (first call) or end (second call) of the timed region."""
        self.marks.append(time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        text = self.file.read()
        os.unlink(self.file.name)
        window = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else None
        return self.summarise(text, window)

    @classmethod
    def summarise(cls, text: str, window) -> dict:
        """Median SM clock, max clock and active throttle reasons of the samples stamped within
        `window` (host seconds, widened by one 50 ms interval); all samples if none fall inside."""
        rows = []
        for line in text.strip().splitlines():
            r = [x.strip() for x in line.split(",")]
            if len(r) < 9:
                continue
            try:
                stamp = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                stamp = None
            try:
                rows.append((stamp, float(r[1]), float(r[2]), r[5:9]))
            except ValueError:
                continue
        inside = rows
        scope = "all samples"
        if window is not None:
            lo, hi = window[0] - 0.05, window[1] + 0.05
            sel = [r for r in rows if r[0] is not None and lo <= r[0] <= hi]
            if sel:
                inside, scope = sel, "timed region"
        reasons = {name for r in inside for name, val in zip(cls.REASONS, r[3]) if val.lower() == "active"}
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "samples": len(inside), "window": scope, "reasons": sorted(reasons)}


DECODE_SOURCES = ("decode.cu", "decode_plan.cuh", "decode_simt.cuh", "decode_mma.cuh", "decode_launch.cuh",
                  "common.cuh")


def decode_sources_sha256() -> str:
    """sha256 over the decode kernel's source files, in order."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "pagedattention_kv_cache_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def decode_traffic_record():
    """ncu DRAM bytes per decode launch, valid only for the decode sources it was taken on."""
    path = os.path.join(ROOT, "profiles", "paged_decode_qwen3_b256_traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"decode sources sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram bytes per full launch:\s*([0-9]+)", text)
    if not m_sha or not m_b:
        return None
    return int(m_b.group(1)) if decode_sources_sha256() == m_sha.group(1) else None


# ---------------------------------------------------------------- algorithmic work

HBM_NOMINAL_GBS = 8000.0  # GB300 HBM3e, the ~8 TB/s nominal figure the target is stated against


def roofline_hbm(gbs: float, hbm_peak: float, **extra) -> dict:
    """An HBM roofline object: the fraction of the measured copy peak, and of the nominal ~8 TB/s."""
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4), "frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4),
            "nominal_peak": HBM_NOMINAL_GBS, **extra}


def decode_alg_bytes(w) -> int:
    elt = torch.finfo(w.dtype).bits // 8
    kv = sum(w.context_lens) * w.num_kv_heads * w.head_dim * 2 * elt
    qo = 2 * w.batch * w.num_q_heads * w.head_dim * elt
    meta = sum(-(-n // w.block_size) for n in w.context_lens) * 4 + w.batch * 4
    return kv + qo + meta


def store_alg_bytes(n_tokens: int, w) -> int:
    elt = torch.finfo(w.dtype).bits // 8
    return 2 * 2 * n_tokens * w.num_kv_heads * w.head_dim * elt + 4 * n_tokens


def prefill_flops(p) -> int:
    total = 0
    for c, n in zip(p.num_cached, p.num_new):
        total += n * c + n * (n + 1) // 2  # sum over rows r < n of (c + r + 1) keys
    return 4 * p.head_dim * p.num_q_heads * total


def prefill_alg_bytes(p) -> int:
    elt = 2
    q = sum(p.num_new) * p.num_q_heads * p.head_dim * elt
    kv = sum(c + n for c, n in zip(p.num_cached, p.num_new)) * p.num_kv_heads * p.head_dim * 2 * elt
    return 2 * q + kv


# ---------------------------------------------------------------- GPU arm

class DecodeState:
    def __init__(self, w, device):
        import pagedattention_kv_cache_gb300 as pkv
        from pagedattention_kv_cache_gb300 import metadata as md
        from pagedattention_kv_cache_gb300 import workloads as wl

        self.pkv = pkv
        self.w = w
        L = w.num_layers
        elt = torch.finfo(w.dtype).bits // 8
        need = 2 * L * w.num_blocks * w.block_size * w.num_kv_heads * w.head_dim * elt
        free, _ = torch.cuda.mem_get_info(device)
        if need + (8 << 30) > free:
            raise RuntimeError(f"workload needs {need / 1e9:.1f} GB of KV cache; {free / 1e9:.1f} GB free")
        self.k_cache, self.v_cache, self.q, self.k_new, self.v_new = [], [], [], [], []
        for layer in range(L):
            t = wl.decode_tensors(w, device, layer=layer)
            self.k_cache.append(t["k_cache"])
            self.v_cache.append(t["v_cache"])
            self.q.append(t["q"])
            self.k_new.append(t["k_new"])
            self.v_new.append(t["v_new"])
            del t
        meta = md.decode_metadata(w.block_tables, w.context_lens, w.block_size)
        self.meta_host = meta
        self.meta = md.to_device(meta, device)
        self.out = [torch.empty_like(q) for q in self.q]
        self.ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0, device=device)

    def step(self, events=None, q=None, k_new=None, v_new=None, meta=None, out=None):
        pkv = self.pkv
        q = q or self.q
        k_new = k_new or self.k_new
        v_new = v_new or self.v_new
        meta = meta or self.meta
        out = out or self.out
        for layer in range(self.w.num_layers):
            pkv.kv_store(k_new[layer], v_new[layer], self.k_cache[layer], self.v_cache[layer], meta["slot_mapping"])
            if events is not None:
                events[layer][0].record()
            pkv.paged_decode_attn(q[layer], self.k_cache[layer], self.v_cache[layer], meta["block_tables"],
                                  meta["context_lens"], self.w.scale, workspace=self.ws, out=out[layer])
            if events is not None:
                events[layer][1].record()


def bench_decode(args, device, world):
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b256_28l()
    st = DecodeState(w, device)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    L = w.num_layers
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index or 0)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark()
    torch.cuda.nvtx.range_push("timed_steps")
    start.record()
    for k in range(args.steps):
        st.step(events=ev[k])
    stop.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    sampler.mark()
    barrier(world)
    clocks = sampler.stop()
    ms_total = max_over_ranks(start.elapsed_time(stop), world, device)
    decode_ms = [a.elapsed_time(b) for per in ev for (a, b) in per]
    assert st.pkv.device_error() == 0

    step_bytes = L * (decode_alg_bytes(w) + store_alg_bytes(w.batch, w))
    ms_step = ms_total / args.steps
    value = sum_over_ranks(step_bytes * args.steps, world, device) / (ms_total * 1e-3) / 1e9
    return dict(w=w, st=st, ms_step=ms_step, value=value, decode_ms=decode_ms, clocks=clocks,
                step_bytes=step_bytes, launches=2 * L * args.steps)


def bench_e2e(args, res, device, world):
    """Same step through the public API with pinned host inputs copied in and outputs copied out."""
    st, w = res["st"], res["w"]
    L = w.num_layers
    h_q = [q.cpu().pin_memory() for q in st.q]
    h_k = [k.cpu().pin_memory() for k in st.k_new]
    h_v = [v.cpu().pin_memory() for v in st.v_new]
    h_meta = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in st.meta_host.items()}
    h_out = [torch.empty_like(o, device="cpu").pin_memory() for o in st.out]
    d_q = [torch.empty_like(q) for q in st.q]
    d_k = [torch.empty_like(k) for k in st.k_new]
    d_v = [torch.empty_like(v) for v in st.v_new]
    d_meta = {k: torch.empty_like(v, device=device) for k, v in h_meta.items()}
    h2d = sum(t.numel() * t.element_size() for t in h_q + h_k + h_v + list(h_meta.values()))
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    # Host copies overlap the kernels, as a serving loop would run them: layer l's inputs go up on
    # one copy stream while earlier layers compute, and its output comes down on another while
    # later layers compute.  Every step still moves all its inputs in and all its outputs out.
    compute = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    pkv = st.pkv

    def one():
        up.wait_stream(compute)  # the previous step no longer reads the device inputs
        ready = []
        with torch.cuda.stream(up):
            for key in h_meta:
                d_meta[key].copy_(h_meta[key], non_blocking=True)
            for layer in range(L):
                for dst, src in ((d_q[layer], h_q[layer]), (d_k[layer], h_k[layer]), (d_v[layer], h_v[layer])):
                    dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(up)
                ready.append(ev)
        for layer in range(L):
            compute.wait_event(ready[layer])
            pkv.kv_store(d_k[layer], d_v[layer], st.k_cache[layer], st.v_cache[layer], d_meta["slot_mapping"])
            pkv.paged_decode_attn(d_q[layer], st.k_cache[layer], st.v_cache[layer], d_meta["block_tables"],
                                  d_meta["context_lens"], w.scale, workspace=st.ws, out=st.out[layer])
            done = torch.cuda.Event()
            done.record(compute)
            down.wait_event(done)
            with torch.cuda.stream(down):
                h_out[layer].copy_(st.out[layer], non_blocking=True)
        compute.wait_stream(down)  # the step ends when its last output is on the host

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        one()
    stop.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    ms = max_over_ranks(max(start.elapsed_time(stop), wall * 1e3), world, device)
    value = sum_over_ranks(res["step_bytes"] * args.steps, world, device) / (ms * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / args.steps, 4)}


FP8_K_SCALE = 1.0 / 64
FP8_V_SCALE = 1.0 / 64


def decode_alg_bytes_fp8(w) -> int:
    kv = sum(w.context_lens) * w.num_kv_heads * w.head_dim * 2  # one byte per element
    qo = 2 * w.batch * w.num_q_heads * w.head_dim * 2  # bf16 q and out
    meta = sum(-(-n // w.block_size) for n in w.context_lens) * 4 + w.batch * 4
    return kv + qo + meta


def bench_fp8(args, device, world):
    """The same 28-layer decode step over an FP8 (E4M3) cache: quantizing store + decode."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b256_28l()
    L = w.num_layers
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 7)
    kc, vc, q, kn, vn = [], [], [], [], []
    for _ in range(L):
        for pool, scale in ((kc, FP8_K_SCALE), (vc, FP8_V_SCALE)):
            x = torch.randn(shape, generator=gen, device=device)
            pool.append((x / scale).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8))
            del x
        q.append(torch.randn(w.batch, w.num_q_heads, w.head_dim, generator=gen, device=device).bfloat16())
        kn.append(torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen, device=device).bfloat16())
        vn.append(torch.randn(w.batch, w.num_kv_heads, w.head_dim, generator=gen, device=device).bfloat16())
    meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
    out = [torch.empty_like(x) for x in q]
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0, device=device)

    def step(events=None):
        for layer in range(L):
            pkv.kv_store_fp8(kn[layer], vn[layer], kc[layer], vc[layer], meta["slot_mapping"], FP8_K_SCALE,
                             FP8_V_SCALE)
            if events is not None:
                events[layer][0].record()
            pkv.paged_decode_attn_fp8(q[layer], kc[layer], vc[layer], meta["block_tables"], meta["context_lens"],
                                      w.scale, FP8_K_SCALE, FP8_V_SCALE, workspace=ws, out=out[layer])
            if events is not None:
                events[layer][1].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    start.record()
    for k in range(args.steps):
        step(ev[k])
    stop.record()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    ms = max_over_ranks(start.elapsed_time(stop), world, device) / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for per in ev for (a, b) in per)
    step_bytes = L * (decode_alg_bytes_fp8(w) + 2 * w.batch * w.num_kv_heads * w.head_dim * (2 + 1) + 4 * w.batch)
    dec_bytes = decode_alg_bytes_fp8(w)
    hbm_peak = measured_peaks()[0]
    result = {"workload": w.name + "-fp8-e4m3", "ms_per_step": round(ms, 4),
              "value": round(world * step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
              "decode_tokens_per_s": round(world * w.batch / (ms * 1e-3), 1),
              "roofline": roofline_hbm(dec_bytes / (dec_ms * 1e-3) / 1e9, hbm_peak,
                                       kernel="paged_decode_mma_kernel<G=2, e4m3>", alg_bytes_per_launch=dec_bytes,
                                       ms_per_launch=round(dec_ms, 5)),
              "gpu_launches": 2 * L * args.steps}
    del kc, vc
    torch.cuda.empty_cache()
    return result


def bench_verify(args, device, q_len=4):
    """Speculative-decoding verify pass (q_len query tokens per sequence), one layer of the batch-256 workload."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b256_28l(num_layers=1)
    t = wl.verify_tensors(w, q_len, device)
    meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
    ws = pkv.decode_workspace(w.batch, q_len * w.num_q_heads, w.head_dim, 0, device=device)
    out = torch.empty_like(t["q"])
    flush = L2Flush(device)
    times = []
    for i in range(args.warmup + max(10, args.steps)):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.paged_verify_attn(t["q"], t["k_cache"], t["v_cache"], meta["block_tables"], meta["context_lens"],
                              w.scale, workspace=ws, out=out)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    assert pkv.device_error() == 0
    ms = statistics.median(times)
    nbytes = (sum(w.context_lens) * w.num_kv_heads * w.head_dim * 2 * 2 + 2 * w.batch * q_len * w.num_q_heads *
              w.head_dim * 2 + sum(-(-n // w.block_size) for n in w.context_lens) * 4 + 4 * w.batch)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = measured_peaks()[0]
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name.replace("28layers", "1layer") + f"-verify-q{q_len}", "q_len": q_len,
            "ms_median": round(ms, 4), "value": round(gbs, 1), "unit": UNIT,
            "tokens_per_s": round(w.batch * q_len / (ms * 1e-3), 1),
            "roofline": roofline_hbm(gbs, hbm_peak), "l2": "flushed before each rep"}


def bench_long_context(args, device):
    """Long-context small-batch split decode: 4 sequences of 32k-131k tokens, block size 16, 32q/8kv."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.long_context_decode()
    t = wl.decode_tensors(w, device)
    meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0, device=device)
    out = torch.empty_like(t["q"])
    flush = L2Flush(device)
    times = []
    for i in range(args.warmup + max(10, args.steps)):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.paged_decode_attn(t["q"], t["k_cache"], t["v_cache"], meta["block_tables"], meta["context_lens"],
                              w.scale, workspace=ws, out=out)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    assert pkv.device_error() == 0
    ms = statistics.median(times)
    nbytes = decode_alg_bytes(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = measured_peaks()[0]
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name, "ms_median": round(ms, 4), "value": round(gbs, 1), "unit": UNIT,
            "kernel": "paged_decode_mma_kernel (G=4), automatic split + fused combine",
            "roofline": roofline_hbm(gbs, hbm_peak), "l2": "flushed before each rep"}


def bench_decode_b32(args, device):
    """Qwen3-0.6B-shaped decode of one layer at batch 32, contexts uniform in [128, 2048], block size
    256, 512-block pool (~143 MB of K/V: L2-sized, so L2 is flushed before each rep)."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b32()
    t = wl.decode_tensors(w, device)
    meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, w.head_dim, 0, device=device)
    out = torch.empty_like(t["q"])
    flush = L2Flush(device)
    times, both = [], []
    for i in range(args.warmup + max(20, args.steps)):
        flush_l2(flush)
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        pkv.kv_store(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], meta["slot_mapping"])
        e1.record()
        pkv.paged_decode_attn(t["q"], t["k_cache"], t["v_cache"], meta["block_tables"], meta["context_lens"],
                              w.scale, workspace=ws, out=out)
        e2.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e1.elapsed_time(e2))
            both.append(e0.elapsed_time(e2))
    assert pkv.device_error() == 0
    ms = statistics.median(times)
    nbytes = decode_alg_bytes(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = measured_peaks()[0]
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name, "batch": w.batch, "context_tokens": sum(w.context_lens), "alg_bytes": nbytes,
            "ms_median": round(ms, 5), "ms_min": round(min(times), 5), "reps": len(times),
            "store_and_decode_ms_median": round(statistics.median(both), 5),
            "value": round(gbs, 1), "unit": UNIT, "decode_tokens_per_s": round(w.batch / (ms * 1e-3), 1),
            "kernel": "paged_decode_mma_kernel<G=2>, automatic split + fused combine",
            "roofline": roofline_hbm(gbs, hbm_peak), "l2": "flushed before each rep"}


def bench_kv_store(args, device):
    """kv_store at the prefill batch's size (7,168 new tokens, L2 flushed) and at 65,536 tokens
    (537 MB moved: the HBM roofline case), both bf16, 8 KV heads, head_dim 128."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    hbm_peak = measured_peaks()[0]
    flush = L2Flush(device)
    result = {}
    p = wl.qwen3_prefill_prefix()
    t = wl.prefill_tensors(p, device)
    meta = md.prefill_metadata(p.block_tables, p.num_cached, p.num_new, p.block_size, always_tables=True)
    cases = [("prefill_batch", t["k"], t["v"], t["k_cache"], t["v_cache"],
              torch.from_numpy(meta["slot_mapping"]).to(device))]
    n_big = 65536
    gen = torch.Generator(device=device)
    gen.manual_seed(1007)
    bs, hkv, d = 16, 8, 128
    nblk = n_big // bs + 64
    kc = torch.empty(nblk, bs, hkv, d, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    slots = torch.randperm(nblk * bs, generator=gen, device=device)[:n_big].to(torch.int32)
    kb = torch.randn(n_big, hkv, d, generator=gen, device=device).bfloat16()
    vb = torch.randn(n_big, hkv, d, generator=gen, device=device).bfloat16()
    cases.append(("65536_tokens", kb, vb, kc, vc, slots))
    for name, k, v, kcache, vcache, sm in cases:
        n = k.shape[0]
        nbytes = 2 * 2 * n * k.shape[1] * k.shape[2] * k.element_size() + 4 * n
        times = []
        for i in range(args.warmup + max(10, args.steps)):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pkv.kv_store(k, v, kcache, vcache, sm)
            e1.record()
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        gbs = nbytes / (ms * 1e-3) / 1e9
        result[name] = {"tokens": n, "alg_bytes": nbytes, "ms_median": round(ms, 5), "value": round(gbs, 1),
                        "unit": UNIT, "roofline": roofline_hbm(gbs, hbm_peak)}
    assert pkv.device_error() == 0
    result["l2"] = "flushed before each rep"
    result["kernel"] = "kv_store_kernel"
    del t, kc, vc, kb, vb
    torch.cuda.empty_cache()
    return result


def bench_cuda_graph(args, device):
    """Small-batch decode (batch 8, the same Qwen3-0.6B shape, 28 layers of store + decode):
    eager launches against one replay of the step captured in a CUDA graph."""
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b256_28l(batch=8)
    st = DecodeState(w, device)
    L = w.num_layers
    reps = max(20, args.steps)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    eager_ms = timed(st.step)
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        st.step()
    torch.cuda.current_stream(device).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st.step()
    graph_ms = timed(graph.replay)
    assert st.pkv.device_error() == 0
    step_bytes = L * (decode_alg_bytes(w) + store_alg_bytes(w.batch, w))
    gbs = step_bytes / (graph_ms * 1e-3) / 1e9
    hbm_peak = measured_peaks()[0]
    del st, graph
    torch.cuda.empty_cache()
    return {"workload": w.name.replace("b256", "b8"), "batch": w.batch, "layers": L,
            "launches_per_step": 2 * L, "eager_ms_per_step": round(eager_ms, 4),
            "graph_ms_per_step": round(graph_ms, 4), "speedup": round(eager_ms / graph_ms, 3),
            "value": round(gbs, 1), "unit": UNIT, "decode_tokens_per_s": round(w.batch / (graph_ms * 1e-3), 1),
            "roofline": roofline_hbm(gbs, hbm_peak),
            "l2": "inputs (~4 GB per step) larger than L2, no flush"}


def bench_copy_blocks(args, device):
    """Copy-on-write burst: 64 block pairs across 28 layers' K and V pools (block size 256,
    8 KV heads, head_dim 128, bf16: 512 KiB per block per pool), L2 flushed before each rep."""
    import pagedattention_kv_cache_gb300 as pkv

    L, pairs, bs, hkv, d = 28, 64, 256, 8, 128
    nb = 2 * pairs
    gen = torch.Generator(device=device)
    gen.manual_seed(1008)
    ks = [torch.randn(nb, bs, hkv, d, generator=gen, device=device).bfloat16() for _ in range(L)]
    vs = [torch.randn(nb, bs, hkv, d, generator=gen, device=device).bfloat16() for _ in range(L)]
    dst = pairs + torch.randperm(pairs, generator=gen, device=device)
    bp = torch.stack([torch.arange(pairs, device=device), dst], dim=1).to(torch.int32).contiguous()
    flush = L2Flush(device)
    times = []
    for i in range(args.warmup + max(10, args.steps)):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.copy_blocks(ks, vs, bp)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    assert pkv.device_error() == 0
    ms = statistics.median(times)
    nbytes = pairs * L * 2 * (bs * hkv * d * 2) * 2 + pairs * 8
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_peak = measured_peaks()[0]
    del ks, vs
    torch.cuda.empty_cache()
    return {"workload": f"copy-blocks-{pairs}pairs-{L}layers-bs{bs}", "pairs": pairs, "layers": L,
            "alg_bytes": nbytes, "ms_median": round(ms, 4), "value": round(gbs, 1), "unit": UNIT,
            "kernel": "copy_blocks_kernel",
            "roofline": roofline_hbm(gbs, hbm_peak), "l2": "flushed before each rep"}


class L2Flush:
    """Between timed reps: write a buffer twice the size of L2, then read another one as large,
    so L2 holds none of the timed call's inputs and no dirty lines whose write-back would land
    inside the next timed call."""

    def __init__(self, device):
        n = torch.cuda.get_device_properties(device).L2_cache_size // 2  # floats: 2x L2 bytes
        self.dirty = torch.empty(n, dtype=torch.float32, device=device)
        self.clean = torch.zeros(n, dtype=torch.float32, device=device)

    def __call__(self):
        self.dirty.add_(1)
        self.clean.sum()


def flush_l2(flush):
    flush()


def bench_prefill(args, device, p=None):
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    p = p or wl.qwen3_prefill_prefix()
    t = wl.prefill_tensors(p, device)
    meta = md.prefill_metadata(p.block_tables, p.num_cached, p.num_new, p.block_size, always_tables=True)
    gm = md.to_device(meta, device)
    out = torch.empty_like(t["q"])
    flush = L2Flush(device)

    def run():
        pkv.kv_store(t["k"], t["v"], t["k_cache"], t["v_cache"], gm["slot_mapping"])
        e0.record()
        pkv.paged_varlen_prefill_attn(t["q"], gm["cu_seqlens_q"], gm["cu_seqlens_k"], meta["max_seqlen_q"],
                                      meta["max_seqlen_k"], p.scale, k_cache=t["k_cache"], v_cache=t["v_cache"],
                                      block_tables=gm["block_tables"], out=out)
        e1.record()

    times = []
    reps = max(10, args.steps)
    for i in range(args.warmup + reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush_l2(flush)
        run()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    flops = prefill_flops(p)
    return {"workload": p.name, "flops_per_call": flops, "ms_median": round(ms, 4), "ms_min": round(min(times), 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2), "reps": reps, "l2": "flushed before each rep",
            "alg_bytes_per_call": prefill_alg_bytes(p)}


# ---------------------------------------------------------------- CPU oracle

def oracle_decode_sample(w, state=None, budget_s: float = 12.0, max_seqs: int = 64, seed: int = 0):
    """Time the oracle's decode attention on whole sequences of layer 0 until ``budget_s`` elapses.

    Returns (algorithmic bytes processed, seconds, sequences).  With a GPU
    state the sequences' blocks are copied from the device pools; without,
    the same-shaped blocks are drawn on the CPU.
    """
    from oracle import attention as oa

    rng = np.random.default_rng(seed)
    order = rng.permutation(w.batch)[:max_seqs].tolist()
    elt = torch.finfo(w.dtype).bits // 8
    done_bytes, elapsed, nseq = 0, 0.0, 0
    gen = torch.Generator().manual_seed(seed)
    for b in order:
        table = w.block_tables[b]
        ctx = w.context_lens[b]
        if state is not None:
            idx = torch.tensor(table, device=state.k_cache[0].device)
            kc = state.k_cache[0].index_select(0, idx).float().cpu().numpy()
            vc = state.v_cache[0].index_select(0, idx).float().cpu().numpy()
            q = state.q[0][b:b + 1].float().cpu().numpy()
        else:
            shape = (len(table), w.block_size, w.num_kv_heads, w.head_dim)
            kc = torch.randn(shape, generator=gen).to(w.dtype).float().numpy()
            vc = torch.randn(shape, generator=gen).to(w.dtype).float().numpy()
            q = torch.randn((1, w.num_q_heads, w.head_dim), generator=gen).to(w.dtype).float().numpy()
        local_table = np.arange(len(table), dtype=np.int32)[None, :]
        t0 = time.perf_counter()
        oa.paged_decode_attention(q, kc, vc, local_table, np.array([ctx]), w.scale)
        elapsed += time.perf_counter() - t0
        done_bytes += ctx * w.num_kv_heads * w.head_dim * 2 * elt + 2 * w.num_q_heads * w.head_dim * elt
        nseq += 1
        if elapsed >= budget_s:
            break
    return done_bytes, elapsed, nseq


class OracleAllCores:
    """The oracle's decode attention over whole sequences of one layer, fanned out over every host
    core (oracle.parallel: spawned workers, the layer's pool in shared files)."""

    def __init__(self, w, rows, state=None, seed: int = 0):
        from oracle import metadata as om
        from oracle.parallel import OraclePool, host_cores

        self.w, self.rows = w, list(rows)
        self.pool = OraclePool(host_cores())
        self.cores = self.pool.workers
        tables = [w.block_tables[b] for b in self.rows]
        lens = [w.context_lens[b] for b in self.rows]
        if state is not None:
            shape = tuple(state.k_cache[0].shape)
            views, specs = self.pool.shared({"k_cache": (shape, np.float32), "v_cache": (shape, np.float32)})
            for name, src in (("k_cache", state.k_cache[0]), ("v_cache", state.v_cache[0])):
                dst = torch.from_numpy(views[name])
                for i in range(0, shape[0], 256):  # exact bf16 -> float32 widening, a slab at a time
                    dst[i:i + 256].copy_(src[i:i + 256].float())
            q = state.q[0][self.rows].float().cpu().numpy()
            meta = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(tables, lens)], w.block_size)
            bt = meta["block_tables"]
        else:
            # the sample's blocks drawn on the host (same shapes), numbered in order
            nblk = [-(-n // w.block_size) for n in lens]
            shape = (sum(nblk), w.block_size, w.num_kv_heads, w.head_dim)
            views, specs = self.pool.shared({"k_cache": (shape, np.float32), "v_cache": (shape, np.float32)})
            gen = torch.Generator().manual_seed(seed)
            for name in ("k_cache", "v_cache"):
                dst = torch.from_numpy(views[name])
                for i in range(0, shape[0], 64):
                    blk = dst[i:i + 64]
                    blk.copy_(torch.randn(blk.shape, generator=gen).to(w.dtype).float())
            q = torch.randn((len(self.rows), w.num_q_heads, w.head_dim), generator=gen).to(w.dtype).float().numpy()
            starts = np.cumsum([0] + nblk[:-1])
            local = [list(range(int(s0), int(s0) + k)) for s0, k in zip(starts, nblk)]
            meta = om.prepare_decode([dict(block_table=t, length=n) for t, n in zip(local, lens)], w.block_size)
            bt = meta["block_tables"]
        del views
        specs.update(q=q, block_tables=bt, context_lens=meta["context_lens"], scale=w.scale)
        self.specs = specs
        elt = torch.finfo(w.dtype).bits // 8
        self.nbytes = sum(n * w.num_kv_heads * w.head_dim * 2 * elt + 2 * w.num_q_heads * w.head_dim * elt
                          for n in lens)
        self.pool.decode(self.specs, min(len(self.rows), self.cores))  # workers started and importing done

    def time(self) -> float:
        t0 = time.perf_counter()
        self.pool.decode(self.specs, len(self.rows))
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()


def cpu_baseline(w, state=None, budget_s: float = 8.0):
    """The oracle on every host core (all 256 sequences of layer 0), and on one thread (a bounded
    sample of whole sequences of the same layer)."""
    one_bytes, one_secs, one_seqs = oracle_decode_sample(w, state, budget_s)
    multi = OracleAllCores(w, range(w.batch), state)
    try:
        secs = multi.time()
    finally:
        multi.close()
    return {"value": round(multi.nbytes / secs / 1e9, 4), "unit": UNIT, "cores": multi.cores, "kind": "oracle",
            "sample": f"float64 numpy oracle, layer 0 decode attention of all {w.batch} sequences of the batch "
                      f"({multi.nbytes / 1e6:.0f} MB of algorithmic bytes) in {secs:.2f} s on {multi.cores} "
                      f"worker processes, one sequence per task",
            "one_thread": {"value": round(one_bytes / one_secs / 1e9, 4), "unit": UNIT, "cores": 1,
                           "sample": f"{one_seqs} whole sequences of layer 0 ({one_bytes / 1e6:.0f} MB) in "
                                     f"{one_secs:.1f} s"}}


def run_reference(args):
    world, rank, local = dist_info()
    if rank != 0:
        return 0
    from pagedattention_kv_cache_gb300 import workloads as wl

    w = wl.qwen3_decode_b256_28l()
    rows = np.random.default_rng(0).permutation(w.batch)[:64].tolist()
    ref = OracleAllCores(w, rows, None, seed=1)
    try:
        for _ in range(args.warmup):
            ref.time()
        total_s = sum(ref.time() for _ in range(args.steps))
    finally:
        ref.close()
    value = ref.nbytes * args.steps / total_s / 1e9
    sample = (f"float64 numpy oracle on {ref.cores} worker processes, decode attention of the same 64 whole "
              f"sequences of layer 0 per step ({ref.nbytes / 1e6:.0f} MB of algorithmic bytes), blocks drawn on "
              f"the host")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": "64 whole sequences of layer 0 per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": ref.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    dist_init(world, local, "nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    hbm_peak, tc_peak, tc_sust, peak_src = measured_peaks()

    res = bench_decode(args, device, world)
    w = res["w"]
    dec_ms = statistics.mean(res["decode_ms"])
    dec_bytes = decode_alg_bytes(w)
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    e2e = bench_e2e(args, res, device, world)
    prefill = bench_prefill(args, device)
    prefill["roofline"] = {"bound": "tensor", "achieved": prefill["tflops"], "peak": tc_peak, "unit": "TFLOP/s",
                           "frac": round(prefill["tflops"] / tc_peak, 4), "peak_source": f"{peak_src} bf16 burst"}
    line = {
        "metric": METRIC, "value": round(res["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["ms_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "layers": w.num_layers, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                   "context": "uniform [1024, 8192]", "kv_bytes_resident": 2 * w.num_layers * w.num_blocks *
                   w.block_size * w.num_kv_heads * w.head_dim * 2, "l2": "inputs (~139 GB) larger than L2, no flush",
                   "parallelism": f"replicas x{world}"},
        "decode_tokens_per_s": round(world * w.batch / (res["ms_step"] * 1e-3), 1),
        "roofline": roofline_hbm(achieved, hbm_peak, traffic=decode_traffic_record(),
                                 kernel="paged_decode_mma_kernel<G=2>", alg_bytes_per_launch=dec_bytes,
                                 ms_per_launch=round(dec_ms, 5), peak_source=f"{peak_src} HBM copy"),
        "e2e": e2e,
        "prefill": prefill,
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, res["st"])
    res["st"] = None
    torch.cuda.empty_cache()
    line["fp8_kv"] = bench_fp8(args, device, world)
    line["verify"] = bench_verify(args, device)
    line["decode_b32"] = bench_decode_b32(args, device)
    line["long_context"] = bench_long_context(args, device)
    line["kv_store"] = bench_kv_store(args, device)
    line["cuda_graph_decode"] = bench_cuda_graph(args, device)
    line["copy_blocks"] = bench_copy_blocks(args, device)
    from pagedattention_kv_cache_gb300 import workloads as wl
    lh = bench_prefill(args, device, wl.long_history_prefill())
    lh["roofline"] = {"bound": "tensor", "achieved": lh["tflops"], "peak": prefill["roofline"]["peak"],
                      "unit": "TFLOP/s", "frac": round(lh["tflops"] / prefill["roofline"]["peak"], 4)}
    line["prefill_long_history"] = lh
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_profile_case(args):
    """Small single-kernel cases for ncu captures (a few GB on the device, inputs larger than L2)."""
    import pagedattention_kv_cache_gb300 as pkv
    from pagedattention_kv_cache_gb300 import metadata as md
    from pagedattention_kv_cache_gb300 import workloads as wl

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if args.profile == "decode":
        w = wl.qwen3_decode_b256_28l(batch=128, num_layers=1)
        st = DecodeState(w, device)
        for _ in range(3):
            st.step()
    elif args.profile == "decode-long":
        w = wl.long_context_decode()
        st = DecodeState(w, device)
        for _ in range(3):
            st.step()
    elif args.profile == "decode-fp8":
        # one layer of the FP8 bench step at batch 64 (about 0.6 GB of codes)
        w = wl.qwen3_decode_b256_28l(batch=64, num_layers=1)
        shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 7)
        kc, vc = [(torch.randn(shape, generator=gen, device=device) / s).clamp_(-448, 448).to(torch.float8_e4m3fn)
                  .view(torch.uint8) for s in (FP8_K_SCALE, FP8_V_SCALE)]
        q = torch.randn(w.batch, w.num_q_heads, w.head_dim, generator=gen, device=device).bfloat16()
        meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
        for _ in range(3):
            pkv.paged_decode_attn_fp8(q, kc, vc, meta["block_tables"], meta["context_lens"], w.scale, FP8_K_SCALE,
                                      FP8_V_SCALE)
    elif args.profile == "verify":
        w = wl.qwen3_decode_b256_28l(batch=64, num_layers=1)
        t = wl.verify_tensors(w, 4, device)
        meta = md.to_device(md.decode_metadata(w.block_tables, w.context_lens, w.block_size), device)
        for _ in range(3):
            pkv.paged_verify_attn(t["q"], t["k_cache"], t["v_cache"], meta["block_tables"], meta["context_lens"],
                                  w.scale)
    elif args.profile == "prefill":
        p = wl.qwen3_prefill_prefix()
        t = wl.prefill_tensors(p, device)
        meta = md.prefill_metadata(p.block_tables, p.num_cached, p.num_new, p.block_size, always_tables=True)
        gm = md.to_device(meta, device)
        for _ in range(3):
            pkv.kv_store(t["k"], t["v"], t["k_cache"], t["v_cache"], gm["slot_mapping"])
            pkv.paged_varlen_prefill_attn(t["q"], gm["cu_seqlens_q"], gm["cu_seqlens_k"], meta["max_seqlen_q"],
                                          meta["max_seqlen_k"], p.scale, k_cache=t["k_cache"], v_cache=t["v_cache"],
                                          block_tables=gm["block_tables"])
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    print(f"profile case {args.profile} done", flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["decode", "decode-long", "decode-fp8", "verify", "prefill"],
                    help="run a small single-kernel case for ncu instead of the benchmark")
    args = ap.parse_args()
    if args.profile:
        return run_profile_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
