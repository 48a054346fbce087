#!/usr/bin/env python3
"""Benchmark of the fused softmax-attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

One step = one call of the Llama-8B-like grouped-query prefill chunk (B=1, Hq=32, Hkv=8,
D=128, Lq=512 queries at positions 15872..16383 of a 16K-token bf16 KV cache, causal) through
the C ABI.  `value` is attention TFLOP/s (4*D flops per visible query-key pair per head, the
convention the pages' FlashAttention numbers imply) over K timed steps with inputs resident
in HBM and L2 flushed (a 512 MB write) before every step; the step is replayed from a CUDA
graph of the C-ABI call so host enqueue time stays out of the device timing.  `e2e` is the
same metric through the same call with pinned HOST buffers: every step's host-to-device copy
of q/k/v and device-to-host copy of out/lse are inside its timed region, the steps pipelined
as a serving loop runs them (the next step's inputs copy in while this step computes).

The other hot paths are measured in the same run and reported under "paths": paged GQA
decode (KV GB/s), MLA paged decode at batch 128 x 2048 and 768 x 1024 (KV GB/s), and the
Gemma-2B-like multi-query prefill sweep (TFLOP/s).  Each carries its dominant kernel's
roofline against MEASURED_PEAKS.json.

--impl reference times the fp64 CPU oracle on the host cores on bounded samples of the same
workload (the reference arm: this project's reference implementation is that oracle).
With torchrun (N > 1) every rank runs its own replica of the workload (weak scaling; the
path needs no exchange), times are max-reduced over ranks and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention TFLOP/s (prefill) and KV GB/s (decode) + % of GB300 roofline"
FLUSH_BYTES = 512 << 20
# GB300 data-sheet figures the targets are stated against (about 8 TB/s of HBM3e and about
# 2.2 PFLOP/s of dense bf16; the nominal 2.25 is used, and 8.0 rather than 7.9 TB/s, so each
# fraction against them is the lower one).  Every roofline reports its fraction of the
# measured peak (copy / cuBLAS) and, beside it, of these.
SPEC_PEAKS = {"hbm": 8000.0, "bf16": 2250.0}
# The headline workload, named the same way by both arms.
WORKLOAD = ("gqa_prefill_chunk: B=1 Hq=32 Hkv=8 D=128 Lq=512 at 15872..16383 Lkv=16384 "
            "causal bf16 N(0,1)*0.5 scale 1/sqrt(128)")


# ------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# The sources a kernel is compiled from: its translation unit and the headers it includes.
KERNEL_SOURCES = {
    "prefill": ("prefill.cu", "prefill_common.cuh", "sm103.cuh", "internal.h"),
    "decode": ("decode.cu", "sm103.cuh", "internal.h"),
    "mla": ("mla.cu", "sm103.cuh", "internal.h"),
    "gated_delta": ("gated_delta.cu", "sm103.cuh", "internal.h"),
}


def src_hash(kernel: str) -> str:
    """First 16 hex digits of sha256 over the kernel's sources, concatenated in order."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "softmax_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, or None if the summary is absent
    or was taken on a different version of the kernel source."""
    path = os.path.join(ROOT, "profiles", profile)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m_t or not m_h or m_h.group(1) != src_hash(kernel):
        return None
    return int(m_t.group(1))


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed loops run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        max_mhz = max(r[1] for r in rows)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max_mhz,
                "reasons": reasons, "samples": len(loaded)}


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def time_graph(fn, steps: int, warmup: int, flush, dist: Dist):
    """W eager warm-up calls, then K steps: flush L2 (untimed), replay a CUDA graph of `fn`
    between two events on the current stream.  Returns (per-step ms list, wall seconds,
    launch mode)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    mode = "graph"
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize()
        run = graph.replay
    except Exception:  # noqa: BLE001 - fall back to eager launches
        mode = "eager"
        torch.cuda.synchronize()
        run = fn
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s, e in ev:
        flush()
        s.record()
        run()
        e.record()
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t0
    return [s.elapsed_time(e) for s, e in ev], wall, mode


def roofline(bound, achieved, peak, unit, traffic, pk):
    spec = SPEC_PEAKS["bf16" if unit == "TFLOP/s" else "hbm"]
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{pk['source']} ({'burst' if unit == 'TFLOP/s' else 'copy'})",
            "peak_spec": spec, "frac_spec": round(achieved / spec, 4)}


def summary(value, unit, ms, kernel_ms, rl):
    """One config's entry in the compact per-config record of the result line."""
    return {"value": round(value, 1), "unit": unit, "ms": round(ms, 4),
            "kernel_ms": round(kernel_ms, 4), "frac": rl["frac"], "frac_spec": rl["frac_spec"]}


# ------------------------------------------------------------------------------------------
# workloads on the GPU
# ------------------------------------------------------------------------------------------
def prefill_flops(c: workloads.DenseCase) -> float:
    pairs = workloads.causal_pairs(c.Lq, c.Lkv) if c.causal else c.Lq * c.Lkv
    return 4.0 * c.D * pairs * c.Hq * c.B


def bench_prefill(fa, c, steps, warmup, flush, dist, pk, e2e=False):
    dev = torch.device("cuda")
    q, k, v = workloads.dense_inputs(c)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty(c.B, c.Hq, c.Lq, dtype=torch.float32, device=dev)
    nbytes = fa.prefill_workspace_size(qd, kd, vd, causal=c.causal, scale=c.sm_scale)
    splits = fa.prefill_num_splits(qd, kd, vd, causal=c.causal, scale=c.sm_scale)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)

    def call():
        fa.fa_prefill_ex(qd, kd, vd, causal=c.causal, scale=c.sm_scale, out=out, lse=lse,
                         workspace=ws)

    ms, wall, mode = time_graph(call, steps, warmup, flush, dist)
    flops = prefill_flops(c)
    mean_ms = dist.max(statistics.mean(ms))
    res = {"ms": mean_ms, "tflops": flops / (mean_ms * 1e-3) / 1e12, "flops": flops,
           "splits": splits, "launches_per_step": 1 + (splits > 1), "mode": mode,
           "wall_s": dist.max(wall), "p10_ms": sorted(ms)[len(ms) // 10],
           "p90_ms": sorted(ms)[(9 * len(ms)) // 10]}
    if e2e:
        res["e2e"] = prefill_e2e(fa, c, q, k, v, (qd, kd, vd, out, lse, ws), steps, warmup,
                                 flush, dist, flops)
    torch.cuda.synchronize()
    del qd, kd, vd, out, lse, ws
    return res


def prefill_e2e(fa, c, q, k, v, dev_set, steps, warmup, flush, dist, flops):
    """End-to-end throughput of the C-ABI call from pinned host buffers: every step copies
    its q/k/v host-to-device and reads its out/lse back, all inside the timed region.  The
    steps are pipelined as a serving loop would run them: two device buffer sets, the
    host-to-device copies of step i+1 on a copy stream while step i computes on the main
    stream, the device-to-host reads on a third stream; L2 is flushed before every
    compute.  The value is K steps of work over the whole region's time."""
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    qd, kd, vd, out, lse, ws = dev_set
    sets = [dev_set, (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd),
                      torch.empty_like(out), torch.empty_like(lse), torch.empty_like(ws))]
    oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    main = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    n_timed = max(3, steps // 4)
    free = [None, None]  # event: buffer set b's last step has been read back
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    for i in range(warmup + n_timed):
        if i == warmup:
            torch.cuda.synchronize()
            t0.record(main)
            h2d_s.wait_stream(main)
            d2h_s.wait_stream(main)
        b = i % 2
        sq, sk, sv, so, sl, sw = sets[b]
        with torch.cuda.stream(h2d_s):
            if free[b] is not None:
                h2d_s.wait_event(free[b])
            sq.copy_(qh, non_blocking=True)
            sk.copy_(kh, non_blocking=True)
            sv.copy_(vh, non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(h2d_s)
        flush()
        main.wait_event(landed)
        fa.fa_prefill_ex(sq, sk, sv, causal=c.causal, scale=c.sm_scale, out=so, lse=sl,
                         workspace=sw)
        done = torch.cuda.Event()
        done.record(main)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(done)
            oh.copy_(so, non_blocking=True)
            lh.copy_(sl, non_blocking=True)
            free[b] = torch.cuda.Event()
            free[b].record(d2h_s)
    main.wait_stream(d2h_s)
    main.wait_stream(h2d_s)
    t1.record(main)
    torch.cuda.synchronize()
    dist.barrier()
    e2e_ms = dist.max(t0.elapsed_time(t1) / n_timed)
    del sets
    return {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(e2e_ms, 4), "steps": n_timed,
            "overlap": "step i+1 host-to-device copy overlaps step i compute and readback",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (q, k, v)),
            "d2h_bytes_per_step": out.numel() * out.element_size() + lse.numel() * 4}


def decode_bytes(c: workloads.PagedCase, lens) -> dict:
    L = lens.long()
    kv = int(L.sum()) * c.Hkv * c.D * 2 * 2
    pages = int(((L + c.page_size - 1) // c.page_size).sum()) * 4
    q = c.B * c.Hq * c.D * 2
    out = c.B * c.Hq * c.D * 2 + c.B * c.Hq * 4
    return {"kv": kv, "kernel": kv + pages + q + c.B * 4, "total": kv + pages + q + out + c.B * 4}


def bench_decode(fa, c, steps, warmup, flush, dist, pk):
    """Whole call through the automatic path (KV GB/s of the call's algorithmic bytes); the
    roofline takes the dominant kernel alone where the call has a second (merge) launch.  The
    other decode kernel's whole call is timed beside it for comparison."""
    dev = torch.device("cuda")
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, kp, vp, table, lens))
    max_len = int(lens.max())
    out = torch.empty_like(qd)
    lse = torch.empty(c.B, c.Hq, dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, fa.fa_decode_workspace_size(c.B, c.Hq, c.D, max_len)),
                     dtype=torch.uint8, device=dev)
    plan = fa.fa_decode_get_plan(qd, kd, vd, td, ld, max_len)
    other = fa.FA_DECODE_CUDA_CORES if plan["path"] == fa.FA_DECODE_TENSOR_CORES \
        else fa.FA_DECODE_TENSOR_CORES

    def call(path):
        def f():
            fa.fa_decode_paged(qd, kd, vd, td, ld, max_len, c.sm_scale, out=out, lse=lse,
                               workspace=ws, path=path)
        return f

    b = decode_bytes(c, lens)
    ms_f, _, mode = time_graph(call(fa.FA_DECODE_AUTO), steps, warmup, flush, dist)
    f_ms = dist.max(statistics.mean(ms_f))
    if plan["launches"] == 1:
        k_ms, k_bytes = f_ms, b["total"]
    elif plan["path"] == fa.FA_DECODE_CUDA_CORES:
        chunk = fa.fa_decode_chunk_tokens(c.B, c.Hq, max_len)
        n_chunks = -(-max_len // chunk)
        op = torch.empty(c.B * c.Hq, n_chunks, c.D, dtype=torch.float32, device=dev)
        ol = torch.empty(c.B * c.Hq, n_chunks, dtype=torch.float32, device=dev)

        def states():
            fa.fa_decode_paged_states(qd, kd, vd, td, ld, max_len, c.sm_scale, o_parts=op,
                                      lse_parts=ol)
        ms_k, _, _ = time_graph(states, steps, warmup, flush, dist)
        k_ms, k_bytes = dist.max(statistics.mean(ms_k)), b["kernel"]
        del op, ol
    else:
        k_ms, k_bytes = f_ms, b["total"]
    try:
        ms_o, _, _ = time_graph(call(other), steps, warmup, flush, dist)
        o_ms = dist.max(statistics.mean(ms_o))
        alt = {"path": "tensor cores" if other == fa.FA_DECODE_TENSOR_CORES else "CUDA cores",
               "value": round(b["total"] / (o_ms * 1e-3) / 1e9, 1), "ms": round(o_ms, 4)}
    except fa.FAError as e:
        alt = {"unavailable": str(e)}
    tc = plan["path"] == fa.FA_DECODE_TENSOR_CORES
    res = {"value": round(b["total"] / (f_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "ms": round(f_ms, 4), "bytes": b["total"], "mode": mode,
           "path": "tensor cores" if tc else "CUDA cores", "n_splits": plan["n_splits"],
           "launches_per_step": plan["launches"],
           "roofline": roofline("hbm", k_bytes / (k_ms * 1e-3) / 1e9, pk["hbm"], "GB/s",
                                profiled_traffic("decode_paged_gqa_tc.md" if tc
                                                 else "decode_paged_gqa.md",
                                                 "prefill" if tc else "decode"), pk),
           "kernel_ms": round(k_ms, 4), "other_path": alt}
    del qd, kd, vd, td, ld, out, lse, ws
    torch.cuda.empty_cache()
    return res


def gated_delta_bytes(c: workloads.GatedDeltaCase) -> int:
    """Algorithmic bytes of one call: q, k, v, g, beta read once, out and the final state
    written once."""
    qk = 2 * c.B * c.Hk * c.T * c.dk * 2
    v_out = 2 * c.B * c.Hv * c.T * c.dv * 2
    gb = 2 * c.B * c.Hv * c.T * 4
    return qk + v_out + gb + c.B * c.Hv * c.dv * c.dk * 4


def bench_gated_delta(fa, c, steps, warmup, flush, dist, pk):
    """Gated-delta chunked prefill: the whole call (chunk preparation and the recurrence
    kernel), KV GB/s of its algorithmic bytes against the HBM peak, and tokens per second."""
    dev = torch.device("cuda")
    q, k, v, g, beta, _ = (t.to(dev) if t is not None else None
                           for t in workloads.gated_delta_inputs(c))
    out = torch.empty(c.B, c.Hv, c.T, c.dv, dtype=torch.bfloat16, device=dev)
    st = torch.empty(c.B, c.Hv, c.dv, c.dk, dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, fa.gated_delta_workspace_size(q, k, v, g, beta)), dtype=torch.uint8,
                     device=dev)

    def call():
        fa.gated_delta_prefill(q, k, v, g, beta, scale=c.scale, out=out, final_state=st,
                               workspace=ws)

    ms, _, mode = time_graph(call, steps, warmup, flush, dist)
    f_ms = dist.max(statistics.mean(ms))
    nbytes = gated_delta_bytes(c)
    res = {"value": round(nbytes / (f_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms": round(f_ms, 4),
           "tokens_per_s": round(c.B * c.T / (f_ms * 1e-3), 1), "bytes": nbytes,
           "launches_per_step": 2, "mode": mode,
           "roofline": roofline("hbm", nbytes / (f_ms * 1e-3) / 1e9, pk["hbm"], "GB/s",
                                profiled_traffic("gated_delta_prefill.md", "gated_delta"), pk)}
    del q, k, v, g, beta, out, st, ws
    torch.cuda.empty_cache()
    return res


MLA_GRID = ((128, 2048), (768, 1024), (64, 1024), (64, 2048), (128, 1024), (768, 2048))
# the configured pair again with 64-token pages (page-sized TMA copies instead of row gathers)
MLA_PAGED = ((128, 2048, 64), (768, 1024, 64))


def bench_prefill_paged(fa, c, steps, warmup, flush, dist, pk):
    """Chunked prefill against a paged cache: TFLOP/s of the whole call (kernel, plus the
    merge when the planner splits the KV loop) against the bf16 burst peak."""
    dev = torch.device("cuda")
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, kp, vp, table, lens))
    max_len = int(lens.max())
    out = torch.empty_like(qd)
    lse = torch.empty(c.B, c.Hq, c.Lq, dtype=torch.float32, device=dev)
    nbytes = fa.fa_prefill_paged_workspace_size(c.B, c.Hq, c.Hkv, c.Lq, c.D, max_len)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)

    def call():
        fa.fa_prefill_paged(qd, kd, vd, td, ld, max_len, causal=c.causal, scale=c.sm_scale,
                            out=out, lse=lse, workspace=ws)

    ms, _, mode = time_graph(call, steps, warmup, flush, dist)
    mean_ms = dist.max(statistics.mean(ms))
    flops = workloads.paged_prefill_flops(c, lens.tolist())
    tflops = flops / (mean_ms * 1e-3) / 1e12
    res = {"value": round(tflops, 2), "unit": "TFLOP/s", "ms": round(mean_ms, 4),
           "flops": flops, "seq_lens": lens.tolist(), "workspace_bytes": nbytes,
           "launches_per_step": 1 + (nbytes > 0), "mode": mode,
           "roofline": roofline("tensor", tflops, pk["bf16"], "TFLOP/s",
                                profiled_traffic("prefill_paged_gqa.md", "prefill"), pk)}
    del qd, kd, vd, td, ld, out, lse, ws
    torch.cuda.empty_cache()
    return res


def mla_bytes(c: workloads.MlaCase) -> dict:
    T = sum(c.lens())
    kv = T * (c.Dc + c.Dr) * 2
    pages = sum(-(-n // c.page_size) for n in c.lens()) * 4
    q = c.B * c.H * (c.Dc + c.Dr) * 2
    out = c.B * c.H * c.Dc * 2 + c.B * c.H * 4
    return {"kv": kv, "kernel": kv + pages + q + c.B * 4, "total": kv + pages + q + out + c.B * 4}


def bench_mla(fa, c, steps, warmup, flush, dist, pk):
    dev = torch.device("cuda")
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    qnd, qpd, cd, kd, td, ld = (t.to(dev) for t in (qn, qp, ckv, kpe, table, lens))
    max_len = c.max_len
    out = torch.empty_like(qnd)
    lse = torch.empty(c.B, c.H, dtype=torch.float32, device=dev)
    ws = torch.empty(fa.mla_decode_workspace_size(c.B, c.H, c.Dc, max_len), dtype=torch.uint8,
                     device=dev)
    chunk = fa.mla_decode_chunk_tokens(c.B, c.H, max_len)
    n_chunks = -(-max_len // chunk)
    op = torch.empty(c.B * c.H, n_chunks, c.Dc, dtype=torch.float32, device=dev)
    ol = torch.empty(c.B * c.H, n_chunks, dtype=torch.float32, device=dev)

    def full():
        fa.mla_decode_paged(qnd, qpd, cd, kd, td, ld, max_len, c.scale, out=out, lse=lse,
                            workspace=ws)

    def states():
        fa.mla_decode_paged_states(qnd, qpd, cd, kd, td, ld, max_len, c.scale, o_parts=op,
                                   lse_parts=ol)

    b = mla_bytes(c)
    # One chunk per sequence: the MLA kernel writes the final output.  When that leaves a
    # short last wave, the call also cuts that wave's sequences into chunks and merges them
    # (a second, small launch); the roofline then takes the whole call's time, merge
    # included.  Otherwise: the kernel (timed on its own through the states entry point)
    # plus a merge.
    direct = n_chunks == 1
    tail_split = direct and ws.numel() > 0
    ms_f, _, mode = time_graph(full, steps, warmup, flush, dist)
    f_ms = dist.max(statistics.mean(ms_f))
    if direct:
        k_ms = f_ms
    else:
        ms_k, _, _ = time_graph(states, steps, warmup, flush, dist)
        k_ms = dist.max(statistics.mean(ms_k))
    res = {"value": round(b["total"] / (f_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "ms": round(f_ms, 4), "bytes": b["total"], "chunk": chunk, "mode": mode,
           "launches_per_step": 1 if direct and not tail_split else 2,
           "last_wave_split": tail_split,
           # the direct launch also writes the output; the states launch is counted by its
           # reads only
           "roofline": roofline("hbm", b["total" if direct else "kernel"] / (k_ms * 1e-3) / 1e9,
                                pk["hbm"], "GB/s",
                                profiled_traffic(f"mla_decode_b{c.B}_s{c.seq_len}"
                                                 + (f"_ps{c.page_size}" if c.page_size > 1 else "")
                                                 + ".md", "mla"), pk),
           "kernel_ms": round(k_ms, 4)}
    del qnd, qpd, cd, kd, td, ld, out, lse, ws, op, ol
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ------------------------------------------------------------------------------------------
def oracle_rate(c: workloads.DenseCase, q, k, v, n_rows: int, offset: int = 0):
    """Time the fp64 oracle on n_rows query rows of the workload (spread over heads and
    queries); returns (seconds, flops)."""
    import oracle
    total = c.B * c.Hq * c.Lq
    stride = max(1, total // max(1, n_rows))
    rows = [((offset + r * stride) % total) for r in range(n_rows)]
    off = c.Lkv - c.Lq
    flops = 0.0
    for r in rows:
        i = r % c.Lq
        keys = min(c.Lkv, i + off + 1) if c.causal else c.Lkv
        flops += 4.0 * c.D * max(0, keys)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=c.causal, scale=c.sm_scale, rows=rows)
    return time.perf_counter() - t0, flops


def cpu_baseline(c, budget_s: float = 12.0):
    import oracle
    q, k, v = workloads.dense_inputs(c)
    dt, fl = oracle_rate(c, q, k, v, 32)
    n = int(max(32, min(8192, 32 * budget_s / max(dt, 1e-3))))
    dt, fl = oracle_rate(c, q, k, v, n, offset=7)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} of {c.B * c.Hq * c.Lq} query rows, strided, all visible keys; "
                      f"{dt:.1f} s"}


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    import oracle
    c = workloads.gqa_prefill_chunk()
    q, k, v = workloads.dense_inputs(c)
    dt, fl = oracle_rate(c, q, k, v, 16)
    per_row = dt / 16
    total_steps = args.steps + args.warmup
    rows_per_step = int(max(1, min(4096, args.ref_seconds / max(1e-6, per_row) / total_steps)))
    for w in range(args.warmup):
        oracle_rate(c, q, k, v, rows_per_step, offset=w)
    t_sum, f_sum = 0.0, 0.0
    for s in range(args.steps):
        dt, fl = oracle_rate(c, q, k, v, rows_per_step, offset=1000 + s * 13)
        t_sum += dt
        f_sum += fl
    value = f_sum / t_sum / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_sum / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "flops_per_step": prefill_flops(c),
                   "parallelism": "replica x1"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} query rows per step of "
                                   f"{c.B * c.Hq * c.Lq}, all their visible keys"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
def mqa_point(r, mc, pk):
    """Roofline of one multi-query sweep point: HBM-bound where its arithmetic intensity is
    below the ridge point of the measured peaks, tensor-bound above it."""
    bytes_ = (mc.Lq * mc.Hq * 2 + 2 * mc.Lkv * mc.Hkv) * mc.D * 2 + mc.Lq * mc.Hq * 4
    bound = "hbm" if r["flops"] / bytes_ < pk["bf16"] * 1e3 / pk["hbm"] else "tensor"
    ach = (bytes_ / (r["ms"] * 1e-3) / 1e9) if bound == "hbm" else r["tflops"]
    return {"value": round(r["tflops"], 2), "unit": "TFLOP/s", "ms": round(r["ms"], 4),
            "splits": r["splits"], "launches_per_step": r["launches_per_step"],
            "roofline": roofline(bound, ach, pk["hbm"] if bound == "hbm" else pk["bf16"],
                                 "GB/s" if bound == "hbm" else "TFLOP/s",
                                 profiled_traffic(f"prefill_mqa_lq{mc.Lq}.md", "prefill"), pk)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="CPU time budget of the --impl reference run (all steps)")
    ap.add_argument("--only", choices=("decode", "paged", "mla", "mqa", "gdn"), default=None,
                    help="run the headline plus only this path (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
            return
        import softmax_attention_gb300 as fa
        torch.cuda.set_device(dist.local)
        fa.load_library()
        pk = peaks()
        flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

        def flush():
            flush_buf.zero_()

        clocks = ClockSampler(dist.local)
        clocks.start()
        c = workloads.gqa_prefill_chunk(seed=1 + dist.rank)
        head = bench_prefill(fa, c, args.steps, args.warmup, flush, dist, pk, e2e=True)
        head_rl = roofline("tensor", head["tflops"], pk["bf16"], "TFLOP/s",
                           profiled_traffic("prefill_gqa_chunk.md", "prefill"), pk)
        # every configured workload's figure, compact: the last key of the result line
        configs = {"C2": summary(head["tflops"], "TFLOP/s", head["ms"], head["ms"], head_rl)}
        paths = {}
        if not args.quick or args.only:
            sub = max(20, args.steps // 4) if not args.quick else 3
            want = (lambda name: args.only in (None, name))
            if want("decode"):
                pc = workloads.paged_gqa_decode(seed=1 + dist.rank)
                r = bench_decode(fa, pc, sub, args.warmup, flush, dist, pk)
                paths["paged_gqa_decode"] = r
                configs["C3"] = dict(summary(r["value"], "GB/s", r["ms"], r["kernel_ms"],
                                             r["roofline"]), path=r["path"])
            # the MLA grid of the flashinfer PR's results: batch {64, 128, 768} x {1024, 2048}
            mla_points = [(b_, s_, 1) for b_, s_ in MLA_GRID] + list(MLA_PAGED)
            for batch, seq, ps in (mla_points if want("mla") else ()):
                mc = workloads.mla_decode(batch, seq, seed=1 + dist.rank, page_size=ps)
                key = f"mla_decode_b{batch}_s{seq}" + (f"_ps{ps}" if ps > 1 else "")
                try:
                    r = bench_mla(fa, mc, sub, args.warmup, flush, dist, pk)
                except fa.FAError as e:
                    paths[key] = {"unavailable": str(e)}
                    continue
                paths[key] = r
                name = {(128, 2048, 1): "C4a", (768, 1024, 1): "C4b"}.get((batch, seq, ps))
                if name:
                    configs[name] = summary(r["value"], "GB/s", r["ms"], r["kernel_ms"],
                                            r["roofline"])
            sweep = {}
            for lq in (workloads.MQA_SWEEP_LQ if want("mqa") else ()):
                mc = workloads.mqa_prefill(lq, seed=1 + dist.rank)
                r = bench_prefill(fa, mc, sub, args.warmup, flush, dist, pk)
                sweep[str(lq)] = mqa_point(r, mc, pk)
            if sweep:
                paths["mqa_prefill_sweep"] = sweep
                configs["C5"] = {lq: summary(v["value"], "TFLOP/s", v["ms"], v["ms"],
                                             v["roofline"]) for lq, v in sweep.items()}
            if want("paged"):
                ppc = workloads.paged_gqa_prefill(seed=1 + dist.rank)
                r = bench_prefill_paged(fa, ppc, sub, args.warmup, flush, dist, pk)
                paths["paged_gqa_prefill"] = r
                configs["N1"] = summary(r["value"], "TFLOP/s", r["ms"], r["ms"], r["roofline"])
            if want("gdn"):
                gc = workloads.gated_delta_prefill(seed=1 + dist.rank)
                r = bench_gated_delta(fa, gc, sub, args.warmup, flush, dist, pk)
                paths["gated_delta_prefill"] = r
                configs["N3"] = summary(r["value"], "GB/s", r["ms"], r["ms"], r["roofline"])
        clk = clocks.stop() if dist.rank == 0 else None
        flops = head["flops"]
        total_tflops = dist.world * flops / (head["ms"] * 1e-3) / 1e12
        cpu = None
        if dist.rank == 0 and dist.world == 1 and not args.no_cpu:
            cpu = cpu_baseline(c)
        if dist.rank == 0:
            # Verbose per-path detail first, on a line of its own; the result line (last) keeps
            # to the compact per-config record so that it stays short.
            print("detail " + json.dumps({"paths": paths, "p10_ms": round(head["p10_ms"], 4),
                                          "p90_ms": round(head["p90_ms"], 4),
                                          "e2e_overlap": head["e2e"].pop("overlap", None)}),
                  flush=True)
            line = {
                "metric": METRIC, "value": round(total_tflops, 2), "unit": "TFLOP/s",
                "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(head["ms"], 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "flops_per_step": flops,
                           "parallelism": f"replica x{dist.world}", "kv_splits": head["splits"],
                           "l2": "flushed (512 MB write) before every timed step",
                           "launch": head["mode"]},
                "roofline": head_rl,
                "cpu_baseline": cpu,
                "e2e": head["e2e"],
                "gpu_launches": head["launches_per_step"] * args.steps,
                "clocks": clk,
                "configs": configs,
            }
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
