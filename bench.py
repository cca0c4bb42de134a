#!/usr/bin/env python
"""Benchmark of the GB300 cached GQA + RoPE path.

A step is one decode step of one layer on the Llama-style workload (64 cache
slots x 4096 positions, A = 32 active rows at distinct slots, positions uniform
in [1, 4096), H_q = 32, H_kv = 8, D = 128, theta = 5e5): split-half RoPE + K/V
store of the 32 new tokens (rope_kv_store_out_), then cached GQA attention of
each token over its row's prefix (cached_gqa_attention_out_).  Headline value:
decode tokens/s (A tokens per step).  Beside it: the KV-cache bytes per second
of the attention call against the measured HBM copy bandwidth, and the causal
prefill of 16 prompts x 1024 tokens into empty rows (TFLOP/s against the
measured BF16 dense peak).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; L2 (129 MB) is flushed between timed steps, outside
the events, by writing a 256 MB buffer and then reading another one (so the
write-back of dirty lines does not fall inside the next step).  ``e2e`` repeats the step through the
public API (the prepared decode_step_out_ call) from pinned host memory: one
H2D copy of the step's inputs (staged back to back in one pinned buffer), the
call, D2H of the attention output, all inside a host wall-clock timer,
issued as one CUDA graph captured once and replayed per step (its output
checked byte for byte against the plain call's; the plain sequence of API
calls is reported beside it as ``e2e.plain``).

Multi-GPU: the path has no exchange step; with N ranks (torchrun) every rank
runs its own replica on its own GPU, ranks meet at a barrier around the timed
region and the value is all tokens over the slowest rank's time.

``--impl reference`` times the FP64 CPU oracle on a bounded sample of the same
workload instead (the only CPU arm there is: the pages ship no code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "decode tokens/s + KV-cache HBM GB/s (% of peak); prefill TFLOP/s (% BF16 peak)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp16", action="store_true", help="skip the FP16-storage measurements")
    ap.add_argument("--no-decode-workloads", action="store_true",
                    help="skip the attention call on the divergent-length and long-context decode workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    ap.add_argument("--only", choices=["decode", "decode-single", "prefill", "prefill-varlen"], default=None,
                    help="run just the timed decode steps, just the prefill calls, or just the chunked prefill call "
                         "(for profiler captures)")
    ap.add_argument("--decode-workload", choices=["llama", "divergent", "long", "d64", "g1", "g1d64"],
                    default="llama", help="with --only decode: the decode workload to run")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput of N replicas: every rank processes the same
    units, so the job's rate is all ranks' units over the slowest rank's
    time (taken across ranks)."""
    return units_per_rank * world / max_over_ranks(seconds, world)


def spread(ms, world: int):
    """Median of per-step device times (ms), taken as the slowest rank's
    median, and the distribution around it on this rank: the median is what
    every rate here is computed from; p10/p90/mean/min show the spread."""
    a = np.asarray(ms, dtype=np.float64)
    med = max_over_ranks(float(np.median(a)), world)
    return med, {"median_ms": round(med, 5), "p10_ms": round(float(np.percentile(a, 10)), 5),
                 "p90_ms": round(float(np.percentile(a, 90)), 5), "mean_ms": round(float(a.mean()), 5),
                 "min_ms": round(float(a.min()), 5), "n": int(a.size)}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            target = str(self.dev)
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2], *parts[3:7]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        busy = [r[0] for r in rows]
        return {"sm_mhz": float(np.median(busy)), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def e2e_line(plain_value, plain_spread, graph, h2d, d2h):
    """The end-to-end entry: the step replayed as one CUDA graph when capture
    worked (its output checked against the plain call's), else the plain
    synchronous loop; the plain loop is reported beside it either way."""
    plain = {"value": round(plain_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
             "spread": plain_spread, "mode": "plain: H2D copy, prepared decode_step_out_ call, D2H copy, "
                                             "stream synchronize, per step"}
    if graph is None or "value" not in graph:
        out = dict(plain)
        out["graph"] = graph
        return out
    out = dict(graph)
    out["mode"] = "cuda_graph: " + graph["note"] + ", stream synchronize, per step"
    del out["note"]
    out["plain"] = plain
    return out


# ---------------------------------------------------------------------- profiles
def profile_traffic(kernel_source: str, summary_name: str):
    """DRAM bytes per launch from a committed ncu summary, if that summary was
    taken on the current source of the kernel (its sha256 matches)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    if not os.path.exists(path):
        return None
    src = open(os.path.join(ROOT, "kv_cached_gqa_rope_gb300", "csrc", kernel_source), "rb").read()
    sha = hashlib.sha256(src).hexdigest()
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_workload"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------- decode
def decode_bytes(wl, positions):
    """Algorithmic HBM bytes of one decode step.  Attention call: each active
    row's K and V prefix (p+1 keys, all KV heads), the rotated Q read and the
    output written.  Step (decode_step_out_ or the two public calls): plus the
    store (q, k, v read; q_rot and one K and one V cell per KV head written).
    Single-launch step: the prefixes, q, k, v read, the output and the cells
    written (no q_rot round trip)."""
    p = positions.astype(np.int64)
    kv_prefix = int(np.sum(p + 1)) * wl.H_kv * wl.D * 2 * 2
    q_bytes = wl.A * wl.H_q * wl.D * 2
    kv_new = 2 * wl.A * wl.H_kv * wl.D * 2
    attn = kv_prefix + 2 * q_bytes
    store = 2 * (wl.A * (wl.H_q + 2 * wl.H_kv) * wl.D * 2)
    fused = kv_prefix + 2 * q_bytes + 2 * kv_new
    return attn, attn + store, fused


class L2Flush:
    """Evicts the previous step's data from L2 between timed steps: writes a
    256 MB buffer (twice the 129 MB L2), then reads another 256 MB buffer, so
    that L2 holds only clean lines of unrelated data when the step starts.
    A write alone leaves L2 full of dirty lines whose write-back to HBM would
    run inside the next timed step and take HBM time from it."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = torch.zeros((), dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.sink)


def hold_gpu(us: float):
    """Keep the GPU busy for about `us` microseconds (a spin kernel) so that
    the host queues every timed step before the first one starts: the CUDA
    events then see device time only, never a host launch gap."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is None:
        return
    sleep(int(min(us, 2e6) * 2000))   # cycles at about 2 GHz; the length only needs to be rough


def host_call_us(named_calls, n=200):
    """Host time of one prepared C-ABI call (validation + launch), in us."""
    out = {}
    for name, c in named_calls:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            c()
        out[name] = round((time.perf_counter() - t0) / n * 1e6, 2)
        torch.cuda.synchronize()
    return out


def prefill_flops(wl):
    return 4.0 * wl.D * wl.H_q * wl.A * wl.T * (wl.T + 1) / 2.0


def run_ours(args, rank, world, local):
    import kv_cached_gqa_rope_gb300 as kv
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()
    wl = W.LLAMA_DECODE
    if args.only == "decode":
        wl = {"llama": W.LLAMA_DECODE, "divergent": W.DIVERGENT_DECODE, "long": W.LONG_DECODE,
              "d64": W.HEAD_SHAPE_DECODE[0], "g1": W.HEAD_SHAPE_DECODE[1],
              "g1d64": W.HEAD_SHAPE_DECODE[2]}[args.decode_workload]
    inp = W.make_decode_inputs(wl)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    pos, rows = inp.positions.to(dev), inp.cache_rows.to(dev)
    kc, vc = inp.build_cache(dev)
    q_rot = torch.empty_like(q)
    out = torch.empty_like(q)
    ws1 = kv.new_workspace(kv.rope_kv_store_workspace_size(), dev)
    ws2 = kv.new_workspace(kv.cached_gqa_attention_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D), dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    store = kv.prepare_rope_kv_store_out_(q, k, v, pos, rows, wl.theta, q_rot, kc, vc, ws1, stream)
    attend = kv.prepare_cached_gqa_attention_out_(q_rot, kc, vc, pos, rows, wl.scale, out, ws2, stream)
    ws3 = kv.new_workspace(kv.decode_step_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D), dev)
    step = kv.prepare_decode_step_out_(q, k, v, pos, rows, wl.theta, wl.scale, kc, vc, out, ws3, stream)
    single = kv.prepare_decode_step_out_(q, k, v, pos, rows, wl.theta, wl.scale, kc, vc, out, ws3, stream,
                                         single_launch=True)

    for _ in range(max(args.warmup, 3)):
        if args.only == "decode-single":  # profiler run of the single-launch step: nothing else
            single()
            continue
        store()
        attend()
        if args.only is None:  # profiler runs (--only) launch only the kernels they capture
            step()
            single()
    torch.cuda.synchronize()
    if args.only == "decode-single":
        K = max(3, args.steps)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush()
            ev[i][0].record(stream)
            single()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if kv.kvgqa_read_status(ws3):
            raise RuntimeError("device status flags set in the single-launch step")
        med, sp = spread([a.elapsed_time(b) for a, b in ev], world)
        return {"impl": "ours", "only": "decode-single", "single_launch_step_ms": round(med, 5),
                "tokens_per_s": round(whole_job_rate(wl.A, med / 1e3, world), 1), "spread": sp} if rank == 0 else None
    if args.only == "prefill":
        res = run_prefill(args, kv, dev, stream, flush, world, bf16_peak, bf16_sust, peak_src)
        res_v = run_prefill_varlen(args, kv, dev, stream, flush, world, bf16_peak, peak_src)
        return {"impl": "ours", "only": "prefill", "prefill": res, "prefill_varlen": res_v} if rank == 0 else None
    if args.only == "prefill-varlen":
        res_v = run_prefill_varlen(args, kv, dev, stream, flush, world, bf16_peak, peak_src)
        return {"impl": "ours", "only": "prefill-varlen", "prefill_varlen": res_v} if rank == 0 else None
    calls = [("store", store), ("attention", attend)] + ([("step", step), ("single_launch_step", single)]
                                                          if args.only is None else [])
    host_us = host_call_us(calls, n=min(200, 10 * args.steps))
    if kv.kvgqa_read_status(ws1) or kv.kvgqa_read_status(ws2) or kv.kvgqa_read_status(ws3):
        raise RuntimeError("device status flags set during warm-up")

    K = args.steps

    def timed(body, per_step_host_us):
        """K iterations of body() with the L2 flushed before each, CUDA events
        around each body on the launching stream; per-iteration ms."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        torch.cuda.synchronize()
        hold_gpu(K * (per_step_host_us + 50.0))
        for i in range(K):
            flush()
            body(evs[i])
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def step_body(e):
        e[0].record(stream); step(); e[1].record(stream)

    def single_body(e):
        e[0].record(stream); single(); e[1].record(stream)

    def two_call_body(e):
        e[0].record(stream); store(); attend(); e[1].record(stream)

    def attention_body(e):
        store(); e[0].record(stream); attend(); e[1].record(stream)

    # (1) the step as a user runs it: decode_step_out_ (the store kernel, then
    # the attention, which streams the cache while the store runs); the
    # profiler runs (--only decode) time the two public calls instead
    sampler = ClockSampler(dev.index) if rank == 0 and args.only is None else None
    if sampler:
        sampler.start()
    barrier(world)
    if args.only is None:
        step_ms = timed(step_body, host_us["step"])
    else:
        step_ms = timed(two_call_body, host_us["store"] + host_us["attention"])
    barrier(world)
    step_med_ms, step_spread = spread(step_ms, world)
    tokens_per_s = whole_job_rate(wl.A, step_med_ms / 1e3, world)
    total_ms = step_med_ms * K  # K steps at the slowest rank's median
    attn_bytes, step_bytes, fused_bytes = decode_bytes(wl, inp.positions.numpy())
    # (2) the attention call alone: the dominant kernel, for the roofline
    attn_ms = timed(attention_body, host_us["store"] + host_us["attention"])
    attn_med_ms, attn_spread = spread(attn_ms, world)
    attn_avg_s = attn_med_ms / 1e3
    achieved = attn_bytes / attn_avg_s / 1e9
    if args.only == "decode":
        flags = kv.kvgqa_read_status(ws1) | kv.kvgqa_read_status(ws2)
        if flags:
            raise RuntimeError(f"device status flags {flags} after the timed region")
        return {"impl": "ours", "only": "decode", "value": round(tokens_per_s, 1), "unit": UNIT,
                "ms_per_step": round(total_ms / K, 5), "attention_gbs": round(achieved, 1)} if rank == 0 else None
    # (3) the same step as the two public calls, and in one launch
    two_ms = timed(two_call_body, host_us["store"] + host_us["attention"])
    two_avg_ms, two_spread = spread(two_ms, world)
    fused_ms = timed(single_body, host_us["single_launch_step"])
    flags = kv.kvgqa_read_status(ws1) | kv.kvgqa_read_status(ws2) | kv.kvgqa_read_status(ws3)
    if flags:
        raise RuntimeError(f"device status flags {flags} after the timed region")
    fused_avg_ms, fused_spread = spread(fused_ms, world)

    # ---- FP16 storage: the same step and attention call on the same workload
    # held as IEEE binary16 (the caches converted; unused cells 65504)
    fp16 = None
    if not args.no_fp16:
        q16, k16, v16, kc16, vc16 = (W.to_f16(t) for t in (q, k, v, kc, vc))
        q_rot16, out16 = torch.empty_like(q16), torch.empty_like(q16)
        ws16 = [kv.new_workspace(n, dev) for n in (
            kv.rope_kv_store_workspace_size(), kv.cached_gqa_attention_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D),
            kv.decode_step_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D))]
        store16 = kv.prepare_rope_kv_store_out_(q16, k16, v16, pos, rows, wl.theta, q_rot16, kc16, vc16, ws16[0], stream)
        attend16 = kv.prepare_cached_gqa_attention_out_(q_rot16, kc16, vc16, pos, rows, wl.scale, out16, ws16[1], stream)
        step16 = kv.prepare_decode_step_out_(q16, k16, v16, pos, rows, wl.theta, wl.scale, kc16, vc16, out16, ws16[2],
                                             stream)
        for _ in range(3):
            store16(); attend16(); step16()
        torch.cuda.synchronize()

        def step16_body(e):
            e[0].record(stream); step16(); e[1].record(stream)

        def attn16_body(e):
            store16(); e[0].record(stream); attend16(); e[1].record(stream)

        s16 = spread(timed(step16_body, host_us["step"]), world)[0]
        a16 = spread(timed(attn16_body, host_us["store"] + host_us["attention"]), world)[0] / 1e3
        if any(kv.kvgqa_read_status(w) for w in ws16):
            raise RuntimeError("device status flags set in the FP16 decode")
        fp16 = {"decode": {"step": "decode_step_out_", "step_ms": round(s16, 5),
                           "tokens_per_s": round(wl.A * world / (s16 / 1e3), 1),
                           "attention_ms": round(a16 * 1e3, 5), "kv_gbs": round(attn_bytes / a16 / 1e9, 1),
                           "hbm_frac": round(attn_bytes / a16 / 1e9 / hbm_peak, 4)}}
        del q16, k16, v16, kc16, vc16, q_rot16, out16, ws16, store16, attend16, step16

    # ---- end to end: pinned host inputs -> device -> the step call -> host output.
    # The step's inputs (q, k, v, positions, rows) sit back to back in one
    # pinned staging buffer and move with one host-to-device copy per step;
    # the decode call reads them through views of the device copy.
    srcs = (inp.q, inp.k, inp.v, inp.positions, inp.cache_rows)
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    d_views = []
    for t, o in zip(srcs, offs):
        n = t.numel() * t.element_size()
        h_stage[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        d_views.append(d_stage[o:o + n].view(t.dtype).view(t.shape))
    d_q, d_k, d_v, d_pos, d_rows = d_views
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in srcs)
    d2h = h_out.numel() * h_out.element_size()

    e2e_call = kv.prepare_decode_step_out_(d_q, d_k, d_v, d_pos, d_rows, wl.theta, wl.scale, kc, vc, out, ws3,
                                           stream)

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        e2e_call()
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    e2e_ms = []
    barrier(world)
    for _ in range(K):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_med_ms, e2e_spread = spread(e2e_ms, world)
    e2e_value = whole_job_rate(wl.A, e2e_med_ms / 1e3, world)

    # The same step, its copies included, captured once as a CUDA graph and
    # replayed per step (one graph launch instead of four API calls, the way
    # a serving loop that keeps its buffers would issue it).  The call is
    # prepared on a stream of its own: capture needs a non-default stream.
    e2e_graph = None
    try:
        gstream = torch.cuda.Stream()
        g_call = kv.prepare_decode_step_out_(d_q, d_k, d_v, d_pos, d_rows, wl.theta, wl.scale, kc, vc, out, ws3,
                                             gstream)
        with torch.cuda.stream(gstream):
            for _ in range(3):
                g_call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gstream, capture_error_mode="relaxed"):
            d_stage.copy_(h_stage, non_blocking=True)
            g_call()
            h_out.copy_(out, non_blocking=True)
        want = h_out.clone()  # the plain loop's last output
        h_out.zero_()
        for _ in range(3):
            with torch.cuda.stream(gstream):
                graph.replay()
            gstream.synchronize()
        if not torch.equal(h_out.view(torch.int16), want.view(torch.int16)):
            raise RuntimeError("the graph replay's output differs from the plain call's")
        g_ms = []
        barrier(world)
        for _ in range(K):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(gstream):  # replay() launches on the current stream
                graph.replay()
            gstream.synchronize()
            g_ms.append((time.perf_counter() - t0) * 1e3)
        if kv.kvgqa_read_status(ws3):
            raise RuntimeError("device status flags set in the graph replay")
        g_med_ms, g_spread = spread(g_ms, world)
        e2e_graph = {"value": round(whole_job_rate(wl.A, g_med_ms / 1e3, world), 1), "unit": UNIT,
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "spread": g_spread,
                     "note": "one CUDA graph per step: the H2D copy, decode_step_out_'s two kernels, the D2H copy"}
    except Exception as ex:  # capture unsupported here: the plain loop stands alone
        e2e_graph = {"unavailable": f"{type(ex).__name__}: {ex}"[:200]}

    # ---- the attention call on the other decode workloads of the same path
    decode_workloads = None
    if not args.no_decode_workloads:
        decode_workloads = [run_attention_workload(args, kv, w_, dev, stream, flush, world, hbm_peak)
                            for w_ in (W.DIVERGENT_DECODE, W.LONG_DECODE) + W.HEAD_SHAPE_DECODE]

    # ---- prefill: 16 prompts x 1024 tokens into empty rows
    prefill = None
    prefill_varlen = None
    if not args.no_prefill:
        prefill = run_prefill(args, kv, dev, stream, flush, world, bf16_peak, bf16_sust, peak_src)
        prefill_varlen = run_prefill_varlen(args, kv, dev, stream, flush, world, bf16_peak, peak_src)
        if fp16 is not None:
            fp16["prefill"] = run_prefill(args, kv, dev, stream, flush, world, bf16_peak, bf16_sust, peak_src,
                                          f16=True)
    clocks = sampler.stop() if sampler else None

    if rank != 0:
        return None
    traffic = profile_traffic("flash_decode.cu", "flash_decode_splitk_llama_decode.md")
    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "slots": wl.slots, "max_seq": wl.max_seq, "active_rows": wl.A,
                   "H_q": wl.H_q, "H_kv": wl.H_kv, "head_dim": wl.D, "theta": wl.theta,
                   "positions": "uniform [1,4096), seed 20261203", "l2": "flushed between timed steps (256 MB write, then 256 MB read of another buffer: no dirty lines left to write back inside a step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "decode": {"step": "decode_step_out_: the store kernel, then the split-K attention, which streams "
                           "cache tiles without a new cell while the store runs (two launches)",
                   "step_bytes": step_bytes,
                   "step_gbs": round(step_bytes / (total_ms / K / 1e3) / 1e9, 1),
                   "two_call_step_ms": round(two_avg_ms, 5),
                   "two_call_tokens_per_s": round(wl.A * world / (two_avg_ms / 1e3), 1),
                   "attention_ms": round(attn_avg_s * 1e3, 5), "attention_bytes": attn_bytes,
                   "kv_gbs": round(achieved, 1), "hbm_frac": round(achieved / hbm_peak, 4),
                   "single_launch_step_ms": round(fused_avg_ms, 5),
                   "single_launch_tokens_per_s": round(wl.A * world / (fused_avg_ms / 1e3), 1),
                   "single_launch_step_bytes": fused_bytes,
                   "spread": {"step": step_spread, "two_call_step": two_spread, "attention": attn_spread,
                              "single_launch_step": fused_spread}},
        "roofline": {"kernel": "flash_decode_splitk_kernel (the cached_gqa_attention_out_ call; split-K with the combine run by the last CTA of each cut segment)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     # achieved is from the median launch (CUDA events on the launching stream, L2
                     # flushed before each launch); the same at the mean launch duration beside it
                     "launch_ms": {"median": attn_spread["median_ms"], "mean": attn_spread["mean_ms"],
                                   "n": attn_spread["n"]},
                     "achieved_at_mean": round(attn_bytes / (attn_spread["mean_ms"] / 1e3) / 1e9, 1),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s"},
        "e2e": e2e_line(e2e_value, e2e_spread, e2e_graph, h2d, d2h),
        "gpu_launches": 2 * K,  # rope_kv_store_kernel + flash_decode_splitk_kernel per step
        "host_us_per_call": host_us,
        "clocks": clocks,
    }
    if decode_workloads is not None:
        line["decode_workloads"] = decode_workloads
    if prefill is not None:
        line["prefill"] = prefill
    if prefill_varlen is not None:
        line["prefill_varlen"] = prefill_varlen
    if fp16 is not None:
        line["fp16"] = fp16
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def run_attention_workload(args, kv, wl, dev, stream, flush, world, hbm_peak):
    """The attention call (cached_gqa_attention_out_) on another decode
    workload, timed like the roofline number: the store call outside the
    events, the attention call inside, L2 flushed before each step."""
    inp = W.make_decode_inputs(wl)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    pos, rows = inp.positions.to(dev), inp.cache_rows.to(dev)
    kc, vc = inp.build_cache(dev)
    q_rot, out = torch.empty_like(q), torch.empty_like(q)
    ws1 = kv.new_workspace(kv.rope_kv_store_workspace_size(), dev)
    ws2 = kv.new_workspace(kv.cached_gqa_attention_workspace_size(wl.A, wl.H_q, wl.H_kv, wl.D), dev)
    store = kv.prepare_rope_kv_store_out_(q, k, v, pos, rows, wl.theta, q_rot, kc, vc, ws1, stream)
    attend = kv.prepare_cached_gqa_attention_out_(q_rot, kc, vc, pos, rows, wl.scale, out, ws2, stream)
    for _ in range(max(args.warmup, 3)):
        store()
        attend()
    K = max(10, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    hold_gpu(K * 80.0)
    for i in range(K):
        flush()
        store()
        ev[i][0].record(stream)
        attend()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if kv.kvgqa_read_status(ws1) or kv.kvgqa_read_status(ws2):
        raise RuntimeError(f"device status flags set ({wl.name})")
    med_ms, sp = spread([a.elapsed_time(b) for a, b in ev], world)
    avg_s = med_ms / 1e3
    attn_bytes = decode_bytes(wl, inp.positions.numpy())[0]
    gbs = attn_bytes / avg_s / 1e9
    return {"workload": wl.name, "H_q": wl.H_q, "H_kv": wl.H_kv, "head_dim": wl.D,
            "attention_ms": round(avg_s * 1e3, 5), "attention_bytes": attn_bytes,
            "kv_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
            "tokens_per_s": round(wl.A * world / avg_s, 1), "spread": sp}


def run_prefill(args, kv, dev, stream, flush, world, bf16_peak, bf16_sust, peak_src, f16=False):
    pw = W.PREFILL
    pin = W.make_prefill_inputs(pw)
    q, k, v, rows = pin.q.to(dev), pin.k.to(dev), pin.v.to(dev), pin.cache_rows.to(dev)
    kc, vc = pin.build_cache(dev)
    if f16:  # the same workload held as IEEE binary16
        q, k, v, kc, vc = (W.to_f16(t) for t in (q, k, v, kc, vc))
    out = torch.empty(pw.A, pw.T, pw.H_q, pw.D, dtype=q.dtype, device=dev)
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(pw.A, pw.T, pw.H_q, pw.H_kv, pw.D), dev)

    call = kv.prepare_prefill_gqa_cached_rows_out_(q, k, v, rows, pw.theta, pw.scale, kc, vc, out, ws, stream)

    try:
        for _ in range(3):
            call()
        torch.cuda.synchronize()
    except kv.KvgqaError as e:
        return {"workload": pw.name, "unavailable": str(e)}
    K = max(10, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    hold_gpu(K * 100.0)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    avg, sp = spread([a.elapsed_time(b) for a, b in ev], world)
    flops = prefill_flops(pw)
    tflops = flops / (avg / 1e3) / 1e12
    if kv.kvgqa_read_status(ws):
        raise RuntimeError("device status flags set in prefill")
    return {"workload": pw.name, "ms_per_call": round(avg, 5), "causal_flops": flops,
            "tflops": round(tflops, 1), "frac_of_bf16_peak": round(tflops / bf16_peak, 4),
            "peak": bf16_peak,
            "peak_source": f"{peak_src} burst bf16_tflops" + (" (FP16 dense rate = BF16 rate, nominal ratio 1)" if f16 else ""),
            "note": "whole call: RoPE + store of all prompts, then causal attention", "gpu_launches": 2 * K,
            "spread": sp}


def varlen_flops(wl, offsets, lengths):
    """Algorithmic FLOPs of the chunked prefill: query t of prompt a sees keys
    0 .. off_a + t, each key costing 2*D for q.k and 2*D for p.v, per head."""
    keys = sum(n * o + n * (n + 1) // 2 for o, n in zip(offsets, lengths))
    return 4.0 * wl.D * wl.H_q * keys


def run_prefill_varlen(args, kv, dev, stream, flush, world, bf16_peak, peak_src):
    """The chunked prefill (prefill_varlen_gqa_cached_rows_out_) on a
    serving-shaped mix of the prefill workload's shapes: 16 prompts of
    lengths uniform in [1, 1024] (padded to 1024), each continuing a prefix
    at an offset uniform in [0, 2048 - length] of its row."""
    pw = W.PREFILL
    offs, lens = W.random_offsets_lengths(pw)
    inp = W.make_varlen_inputs(pw, offs, lens)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    off_t, len_t, rows = inp.offsets.to(dev), inp.lengths.to(dev), inp.cache_rows.to(dev)
    kc, vc = inp.build_cache(dev)
    out = torch.empty_like(q)
    ws = kv.new_workspace(kv.prefill_gqa_cached_rows_workspace_size(pw.A, pw.T, pw.H_q, pw.H_kv, pw.D), dev)
    call = kv.prepare_prefill_varlen_gqa_cached_rows_out_(q, k, v, off_t, len_t, rows, pw.theta, pw.scale, kc, vc,
                                                          out, ws, stream)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    K = max(10, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    hold_gpu(K * 100.0)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if kv.kvgqa_read_status(ws):
        raise RuntimeError("device status flags set in the chunked prefill")
    avg, sp = spread([a.elapsed_time(b) for a, b in ev], world)
    flops = varlen_flops(pw, offs, lens)
    tflops = flops / (avg / 1e3) / 1e12
    return {"workload": pw.name + "_chunks_len_u1_1024_off_u", "tokens": int(sum(lens)),
            "ms_per_call": round(avg, 5), "flops": flops, "tflops": round(tflops, 1),
            "frac_of_bf16_peak": round(tflops / bf16_peak, 4), "peak": bf16_peak,
            "peak_source": f"{peak_src} burst bf16_tflops",
            "note": "whole call: RoPE + store of every prompt's tokens at its offset, then attention over the row "
                    "prefix and the prompt", "gpu_launches": 2 * K, "spread": sp}


# ---------------------------------------------------------------------- CPU oracle
def oracle_decode_sample(target_seconds: float):
    """Time the FP64 oracle on the decode step of the same workload: RoPE +
    store of all 32 tokens, then attention of every (token, head), on a host
    cache holding the 32 active rows.  Repeats whole steps until about
    ``target_seconds`` have passed; returns (tokens, seconds, steps)."""
    import oracle
    wl = W.LLAMA_DECODE
    inp = W.make_decode_inputs(wl)
    rows = list(range(wl.A))
    kc, vc = inp.compact_cache(rows, length=wl.max_seq)
    kc_b, vc_b = W.bf16_bits(kc), W.bf16_bits(vc)
    qb, kb, vb = W.bf16_bits(inp.q), W.bf16_bits(inp.k), W.bf16_bits(inp.v)
    pos = inp.positions.numpy()
    crow = np.arange(wl.A)
    tokens, steps = 0, 0
    t0 = time.perf_counter()
    while True:
        q_rot, kc2, vc2 = oracle.rope_kv_store(qb, kb, vb, pos, crow, wl.theta, kc_b, vc_b)
        oracle.cached_gqa_attention(q_rot, kc2, vc2, pos, crow, wl.scale)
        tokens += wl.A
        steps += 1
        if time.perf_counter() - t0 >= target_seconds:
            break
    return tokens, time.perf_counter() - t0, steps


def cpu_baseline(target_seconds: float):
    tokens, secs, steps = oracle_decode_sample(target_seconds)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(tokens / secs, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{steps} whole decode step(s) of the same workload (32 tokens each) by the FP64 numpy "
                      f"oracle in {secs:.1f} s; numpy/BLAS may use up to {cores} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    tokens, secs, steps = oracle_decode_sample(args.cpu_seconds)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    value = tokens / secs
    wl = W.LLAMA_DECODE
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": 0, "ms_per_step": round(secs / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "slots": wl.slots, "max_seq": wl.max_seq, "active_rows": wl.A,
                       "H_q": wl.H_q, "H_kv": wl.H_kv, "head_dim": wl.D},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{steps} whole decode step(s), {secs:.1f} s"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup()
    line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
