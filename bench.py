"""Benchmark of the routed MoE FFN hot path on GB300 (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one full forward (route grouping when T > 1, gate/up + SwiGLU, down + combine) over one
batch of the named workload with its inputs resident in HBM. Default workload: ``fp8_decode``
(T=1, H=7168, I=2048, E=256, top-8, E4M3 with 128x128 block scales). Between timed steps a
buffer of twice the L2 size is written (outside the timed events) and the route set rotates
through 8 seeded draws, so every step streams its experts from HBM.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path does not
shard: replicas only, no collective on the data path); the barrier and the max over ranks are
only for timing. ``--impl reference`` times the FP64 CPU oracle on the host cores instead.
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
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_ffn_histogram_gb300 import inputs  # noqa: E402

METRIC = "MoE FFN tokens/s; effective weight GB/s as % of GB300 HBM peak"
UNIT = "tokens/s"
N_ROUTE_SETS = 8


# ---- distributed (replicas only) -------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (the slowest replica sets the job time)."""
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---- measured peaks ------------------------------------------------------------------------------

def load_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"])
    return 1900.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---- clocks during the timed region ----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            if uuid and not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
        except Exception:
            uuid = None
        self.sel = ["--id=" + uuid] if uuid else []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- algorithmic bytes -----------------------------------------------------------------------------

def matrix_bytes(fmt, n, k):
    if fmt == "fp8":
        return n * k + (n // 128) * (k // 128) * 4
    return n * k // 2 + n * (k // 16)


def alg_bytes(wl):
    """Per call: distinct selected experts' codes + scales of the three projections, plus x,
    out, ids and weights (and the small f16 activation round trip through the workspace)."""
    ids = wl.ids.cpu().numpy().reshape(-1)
    distinct = len({int(e) for e in ids if 0 <= e < wl.E})
    P = wl.T * wl.topk
    w_gu = distinct * 2 * matrix_bytes(wl.fmt, wl.I, wl.H)
    w_d = distinct * matrix_bytes(wl.fmt, wl.H, wl.I)
    act = P * wl.I * 2 + P * (wl.I // 64) * 4
    x = wl.T * wl.H * 2
    out = wl.T * wl.H * 2
    idw = P * 8
    return dict(distinct=distinct, gate_up=w_gu + x + act, down=w_d + act + out + idw,
                total=w_gu + w_d + x + out + idw, weights=w_gu + w_d)


def sweep_rows(T, per=8):
    """Token counts of the even sweeps of <= per tokens the narrow tiers split T into (never a
    trailing sweep of one), the split the library makes."""
    n = (T + per - 1) // per
    rows, start = [], 0
    for i in range(n):
        r = (T - start + (n - i) - 1) // (n - i)
        rows.append(r)
        start += r
    return rows


def sweeps_alg_bytes(wl):
    """Per call of the sweep tier: each sweep reads its own union of selected experts once."""
    ids = wl.ids.cpu().numpy()
    total, start = 0, 0
    for r in sweep_rows(wl.T):
        distinct = len({int(e) for e in ids[start:start + r].reshape(-1) if 0 <= e < wl.E})
        total += distinct * (2 * matrix_bytes(wl.fmt, wl.I, wl.H) + matrix_bytes(wl.fmt, wl.H, wl.I))
        start += r
    return total + 2 * wl.T * wl.H * 2 + wl.T * wl.topk * 8


def kernel_source_sha(files=None):
    """Hash of the kernel's sources: the listed csrc files (its translation unit and the headers
    it includes), or every .cu/.cuh file of csrc when no list is given."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_ffn_histogram_gb300", "csrc")
    names = sorted(files) if files else sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh")))
    for fn in names:
        h.update(fn.encode())
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(config, kernel):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the kernel's
    current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(config, {}).get(kernel)
    if not ent or ent.get("source_sha") != kernel_source_sha(ent.get("files")):
        return None
    return ent.get("dram_bytes_per_launch")


# ---- the CPU oracle (baseline / reference arm) ------------------------------------------------------

def oracle_sample(name, route_set, device, n_tokens=None):
    """One bounded oracle sample of the workload: the sampled tokens' selected experts are
    generated (same seeded bytes as the full bank) and copied to the host, outside the timing."""
    c = inputs.CONFIGS[name]
    tmp = inputs.make_workload(name, device="cpu", bank=object(), route_set=route_set)
    T = tmp.T if n_tokens is None else min(n_tokens, tmp.T)
    ids = tmp.ids[:T].numpy()
    used = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < c["E"]})
    remap = {e: i for i, e in enumerate(used)}
    sub_ids = np.vectorize(lambda e: remap.get(int(e), -1))(ids).astype(np.int32)
    bank = inputs.make_bank(name, device=device, experts=used).numpy()
    x = tmp.x[:T].view(torch.int16).numpy().view(np.uint16)
    wts = tmp.wts[:T].numpy()
    return dict(x=x, ids=sub_ids, wts=wts, bank=bank, fmt=c["fmt"], T=T)


def run_oracle(sample, limit=inputs.LIMIT):
    import oracle
    fn = oracle.moe_fp8 if sample["fmt"] == "fp8" else oracle.moe_nvfp4
    t0 = time.perf_counter()
    fn(sample["x"], sample["ids"], sample["wts"], sample["bank"], limit)
    return time.perf_counter() - t0


def cpu_baseline(name, device, budget_s=20.0):
    """Oracle tokens/s on a bounded sample of the workload, about budget_s of CPU work: each of
    the seeded route sets in turn (its tokens' experts generated once, outside the timing) is
    run repeatedly for its share of the budget."""
    import oracle
    oracle.build()
    c = inputs.CONFIGS[name]
    n_tok = 1 if c["T"] <= 8 else 2
    share = budget_s / N_ROUTE_SETS
    secs, toks, runs, sets = 0.0, 0, 0, 0
    for rs in range(N_ROUTE_SETS):
        s = oracle_sample(name, rs, device, n_tokens=min(c["T"], n_tok))
        spent = 0.0
        while True:
            dt = run_oracle(s)
            secs += dt
            spent += dt
            toks += s["T"]
            runs += 1
            if spent + dt > share:               # the next run would overrun this set's share
                break
        sets += 1
        del s
        if secs >= budget_s:                     # slow runs: no further set once the budget is spent
            break
    return {"value": toks / secs, "unit": UNIT, "cores": oracle.hardware_threads(),
            "kind": "oracle",
            "sample": f"{toks} token(s) of {name}: {sets} seeded route set(s) of {n_tok} token(s), "
                      f"{runs} oracle runs in all, FP64 C++ oracle, {secs:.1f} s"}


# ---- our arm ---------------------------------------------------------------------------------------

def make_route_sets(name, device, bank, E=None, T=None):
    return [inputs.make_workload(name, device=device, bank=bank, route_set=i, E=E, T=T)
            for i in range(N_ROUTE_SETS)]


HOLD_CYCLES = 1_000_000      # about 0.5 ms of SM clock


def hold_stream():
    """Keep the current stream busy with a bounded spin kernel while the host enqueues the timed
    work (the blocking-kernel technique of nvbench), so that the CUDA events bracket device work
    rather than the binding's Python marshalling. Issued after the L2 flush and before the start
    event, outside the timed region; the end-to-end loop does not use it."""
    torch.cuda._sleep(HOLD_CYCLES)


def stream_ceiling_us(nbytes, dev, flush, reps):
    """Median device time (us) of one plain streaming-read kernel (moe_stream_read) over nbytes,
    timed like a forward step: L2 flushed, stream held, CUDA events around the launch. What one
    kernel of that many bytes reaches on the device, the ceiling a step of the same bytes is read
    against (launch latency and the ramp at either end weigh more the fewer bytes a call moves)."""
    from moe_expert_ffn_histogram_gb300 import capi
    n = int(nbytes) // 16 * 16
    buf = torch.empty(n + 256, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ts = []
    for i in range(3 + reps):
        flush.zero_()
        hold_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        capi.stream_read(buf, n, sink)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(a.elapsed_time(b) * 1e3)
    del buf
    ts.sort()
    return ts[len(ts) // 2]


def ceiling_entry(nbytes, t_us, ceil_us, peak, key):
    """One stream_ceiling entry: the plain read of the same bytes, and how the timed work compares."""
    gbs = nbytes / (ceil_us * 1e-6) / 1e9
    return {"bytes": int(nbytes), "read_us": round(ceil_us, 2), "read_gbs": round(gbs, 1),
            "read_frac_of_peak": round(gbs / peak, 4), key: round(ceil_us / t_us, 4)}


CEILING_RULE = ("one plain streaming-read kernel (moe_stream_read) over the same number of "
                "algorithmic bytes, timed like the step (L2 flushed, CUDA events around the launch, "
                "median); *_vs_read = read time / measured time (1.0: as fast as a plain read)")


# ---- harness statistics ---------------------------------------------------------------------------

def nearest_rank(sorted_vals, percentile: int):
    """The sample at nearest rank ceil(percentile * n / 100) of an ascending list (1 <= percentile
    <= 100): an observed sample, never an interpolation ("memra-engine 0.108.0
    src/bin/ep_step_fp8_gate.rs", benchmark harness, `nearest_rank_ns`)."""
    n = len(sorted_vals)
    if n == 0 or not 1 <= percentile <= 100:
        raise ValueError("nearest_rank needs samples and 1 <= percentile <= 100")
    rank = -(-percentile * n // 100)
    return sorted_vals[min(max(rank, 1), n) - 1]


def step_stats_us(step_ms):
    """mean, min, p50, p90, p95, p99 and max of the per-step times, in microseconds."""
    srt = sorted(step_ms)
    out = {"mean": statistics.mean(srt) * 1e3, "min": srt[0] * 1e3}
    for q in (50, 90, 95, 99):
        out[f"p{q}"] = nearest_rank(srt, q) * 1e3
    out["max"] = srt[-1] * 1e3
    return {k: round(v, 3) for k, v in out.items()}


def output_checksum(values) -> int:
    """Order- and bit-sensitive 64-bit fold of fp32 values: state = rotl(state, 7) ^ bits(v),
    starting from 0x9e3779b97f4a7c15 (the gate binary's `output_checksum`, "memra-engine 0.108.0
    src/bin/ep_step_fp8_gate.rs", benchmark harness). bf16 results are widened to fp32 first.
    The fold is linear over XOR, so it is evaluated in closed form: v_i enters rotated by
    7 * (n - 1 - i) mod 64, which depends only on i mod 64, so each residue class is XOR-reduced
    first and the 64 partial results are rotated once each; the start value enters rotated by
    7 * n mod 64."""
    a = np.ascontiguousarray(np.asarray(values, dtype=np.float32)).reshape(-1)
    n = a.size
    bits = a.view(np.uint32).astype(np.uint64)
    pad = (-n) % 64
    if pad:
        bits = np.concatenate([bits, np.zeros(pad, dtype=np.uint64)])
    cols = np.bitwise_xor.reduce(bits.reshape(-1, 64), axis=0) if bits.size else np.zeros(64, np.uint64)
    mask = (1 << 64) - 1

    def rotl(v, r):
        r %= 64
        return ((v << r) | (v >> (64 - r))) & mask if r else v

    acc = rotl(0x9E3779B97F4A7C15, 7 * n)
    for j in range(64):
        acc ^= rotl(int(cols[j]), 7 * (n - 1 - j))
    return acc


def graded_fraction(alg_bytes, flops, seconds, hbm_gbs, bf16_tflops):
    """The grouped-GEMM workload's graded fraction: max(bytes / HBM peak, FLOPs / bf16 peak) over
    the measured time (the roofline of a contraction next to its ridge point)."""
    floor = max(alg_bytes / (hbm_gbs * 1e9), flops / (bf16_tflops * 1e12))
    return floor / seconds, floor


# ---- our arm ---------------------------------------------------------------------------------------

def prefill_alg_bytes(wl):
    """Per call of the grouped-GEMM tier: the distinct experts' weights, x and out, the 16-bit
    activation written and read once per routed pair, ids and weights."""
    b = alg_bytes(wl)
    P = wl.T * wl.topk
    return b["weights"] + 2 * wl.T * wl.H * 2 + 2 * P * wl.I * 2 + P * 8


def measure_workload(name, args, dev, bank, world, peak, peak_kind, tpeak, want_router=True):
    """Times one workload through the C ABI and returns its part of the bench line."""
    from moe_expert_ffn_histogram_gb300 import capi
    c = inputs.CONFIGS[name]
    E = c["E"] if args.bank_experts is None else args.bank_experts
    sets = make_route_sets(name, dev, bank, E, args.tokens)
    wl0 = sets[0]
    T = wl0.T
    fmt_code = capi.FMT_FP8 if c["fmt"] == "fp8" else capi.FMT_NVFP4
    ws = capi.alloc_workspace(T, wl0.H, wl0.I, wl0.E, wl0.topk, fmt_code, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd(wl, o):
        capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit, out=o, workspace=ws)

    # untimed reference run of every route set (also warm-up): the timed steps must reproduce it
    refs = []
    for j in range(N_ROUTE_SETS):
        flush.zero_()
        o = torch.empty(T, wl0.H, dtype=torch.bfloat16, device=dev)
        fwd(sets[j], o)
        refs.append(o)
    out = torch.empty(T, wl0.H, dtype=torch.bfloat16, device=dev)
    for i in range(args.warmup):
        flush.zero_()
        fwd(sets[i % N_ROUTE_SETS], out)
    torch.cuda.synchronize()
    outs = [torch.empty(T, wl0.H, dtype=torch.bfloat16, device=dev) for _ in range(args.steps)]

    # ---- timed region: whole forward per step, device events on the launching stream
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    if args.profile_range:            # a profiler started with its capture off records from here
        torch.cuda.cudart().cudaProfilerStart()
    for i in range(args.steps):
        flush.zero_()
        hold_stream()
        if args.profile_range:
            torch.cuda.nvtx.range_push(f"{name}/step")
        ev[i][0].record(stream)
        fwd(sets[i % N_ROUTE_SETS], outs[i])
        ev[i][1].record(stream)
        if args.profile_range:
            torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if args.profile_range:
        torch.cuda.cudart().cudaProfilerStop()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    clk = clocks.stop()
    same = sum(int(torch.equal(outs[i].view(torch.int16), refs[i % N_ROUTE_SETS].view(torch.int16)))
               for i in range(args.steps))
    checksum = 0
    for r in refs:
        checksum ^= output_checksum(r.float().cpu().numpy())
    del outs

    # ---- the same calls captured once per route set in a CUDA graph and replayed
    graph_ms, graph_err = [], None
    try:
        graphs = []
        for j in range(N_ROUTE_SETS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fwd(sets[j], out)
            graphs.append(g)
        torch.cuda.synchronize()
        for i in range(args.warmup + args.steps):
            flush.zero_()
            hold_stream()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            graphs[i % N_ROUTE_SETS].replay()
            b_.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                graph_ms.append(a_.elapsed_time(b_))
        del graphs
    except Exception as exc:                       # report, do not fail the bench line
        graph_err = f"{type(exc).__name__}: {exc}"[:200]
        torch.cuda.synchronize()

    # ---- T <= 8: the same work as three stage kernels (each timed alone)
    stage_ms = {"plan": [], "gate_up": [], "down_combine": []}
    if T <= 8:
        for i in range(args.steps):
            wl = sets[i % N_ROUTE_SETS]
            flush.zero_()
            hold_stream()
            e0, e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
            e0.record(stream)
            capi.plan(wl.ids, wl.H, wl.I, wl.E, fmt_code, ws)
            e1.record(stream)
            capi.gate_up(wl.x, wl.ids, wl.bank, wl.limit, ws)
            e2.record(stream)
            capi.down_combine(wl.ids, wl.wts, wl.bank, out, ws)
            e3.record(stream)
            torch.cuda.synchronize()
            stage_ms["plan"].append(e0.elapsed_time(e1))
            stage_ms["gate_up"].append(e1.elapsed_time(e2))
            stage_ms["down_combine"].append(e2.elapsed_time(e3))
    # ---- prefill: the library's own per-stage events (moe_stage_timing) around each kernel
    prefill_stage_ms = {}
    if T > 8:
        capi.stage_timing(True)
        try:
            for i in range(args.steps):
                flush.zero_()
                hold_stream()
                fwd(sets[i % N_ROUTE_SETS], out)
                for k, v in capi.stage_times():
                    prefill_stage_ms.setdefault(k, []).append(v)
        finally:
            capi.stage_timing(False)

    # ---- the router in front of the path (informational): a synthetic bf16 router matrix
    router_ms = []
    if want_router and E % 16 == 0 and E <= 1024:
        rg = torch.Generator(device=dev)
        rg.manual_seed(4242)
        rw = (torch.randn(E, wl0.H, generator=rg, device=dev) * wl0.H ** -0.5).to(torch.bfloat16)
        rbias = torch.zeros(E, dtype=torch.float32, device=dev)
        rws = torch.empty(int(capi.load().moe_router_workspace_bytes(T, wl0.H, E)), dtype=torch.uint8, device=dev)
        for i in range(args.warmup + args.steps):
            flush.zero_()
            hold_stream()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            capi.router(sets[i % N_ROUTE_SETS].x, rw, 8, 2.5, True, bias=rbias, workspace=rws)
            b_.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                router_ms.append(a_.elapsed_time(b_))

    # ---- end to end through the public API: pinned host inputs in, result out, every step.
    # A step's inputs (x, ids, weights) sit in one pinned host buffer and go over in one copy
    # into one device buffer that the three input tensors view.
    def al(n):
        return (n + 255) // 256 * 256
    xb, ib = wl0.x.numel() * 2, wl0.ids.numel() * 4
    wb = wl0.wts.numel() * 4
    o_ids, o_w = al(xb), al(xb) + al(ib)
    tot = o_w + al(wb)
    hbuf = []
    for st_ in sets:
        hb = torch.zeros(tot, dtype=torch.uint8).pin_memory()
        hb[:xb].copy_(st_.x.cpu().contiguous().view(torch.uint8).reshape(-1))
        hb[o_ids:o_ids + ib].copy_(st_.ids.cpu().contiguous().view(torch.uint8).reshape(-1))
        hb[o_w:o_w + wb].copy_(st_.wts.cpu().contiguous().view(torch.uint8).reshape(-1))
        hbuf.append(hb)
    dbuf = torch.empty(tot, dtype=torch.uint8, device=dev)
    dx = dbuf[:xb].view(torch.bfloat16).view(wl0.x.shape)
    dids = dbuf[o_ids:o_ids + ib].view(torch.int32).view(wl0.ids.shape)
    dw = dbuf[o_w:o_w + wb].view(torch.float32).view(wl0.wts.shape)
    hout = torch.empty(T, wl0.H, dtype=torch.bfloat16).pin_memory()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        j = i % N_ROUTE_SETS
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dbuf.copy_(hbuf[j], non_blocking=True)
        capi.forward(dx, dids, dw, bank, inputs.LIMIT, out=out, workspace=ws)
        hout.copy_(out, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    h2d = tot
    d2h = T * wl0.H * 2

    # ---- aggregate (replicas: units add up, the slowest rank sets the time)
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    units = sum_over_ranks(float(T * args.steps), world, dev)
    value = units / total_s
    e2e_s = max_over_ranks(sum(e2e_ms) / 1e3, world, dev)
    e2e_value = sum_over_ranks(float(T * args.steps), world, dev) / e2e_s

    by = [alg_bytes(s_) for s_ in sets]
    mean_total = statistics.mean(b_["total"] for b_ in by)
    ms = statistics.mean(step_ms)
    call_gbs = mean_total / (ms * 1e-3) / 1e9
    if T == 1:
        # dominant kernel: gate_up_kernel (two thirds of the bytes), timed by its own CUDA events
        # in the stage loop above (launched alone, so without the PDL overlap of the step)
        gu_ms = statistics.mean(stage_ms["gate_up"])
        dn_ms = statistics.mean(stage_ms["down_combine"])
        gu_bytes = statistics.mean(b_["gate_up"] for b_ in by)
        dn_bytes = statistics.mean(b_["down"] for b_ in by)
        ach = gu_bytes / (gu_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "gate_up_kernel", "achieved": round(ach, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(ach / peak, 4),
                "traffic": profiled_traffic(name, "gate_up"), "alg_bytes_per_launch": int(gu_bytes),
                "avg_launch_us": round(gu_ms * 1e3, 2),
                "down": {"kernel": "down_combine_kernel", "alg_bytes_per_launch": int(dn_bytes),
                         "avg_launch_us": round(dn_ms * 1e3, 2),
                         "achieved": round(dn_bytes / (dn_ms * 1e-3) / 1e9, 1),
                         "frac": round(dn_bytes / (dn_ms * 1e-3) / 1e9 / peak, 4)},
                "step": {"kernels": "gate_up_kernel + down_combine_kernel (PDL)",
                         "alg_bytes": int(mean_total), "achieved": round(call_gbs, 1),
                         "frac": round(call_gbs / peak, 4)},
                "note": "CUDA events on the launching stream"}
        reps = max(args.steps, 10)
        roof["stream_ceiling"] = {
            "rule": CEILING_RULE,
            "step": ceiling_entry(mean_total, ms * 1e3, stream_ceiling_us(mean_total, dev, flush, reps),
                                  peak, "step_vs_read"),
            "gate_up": ceiling_entry(gu_bytes, gu_ms * 1e3, stream_ceiling_us(gu_bytes, dev, flush, reps),
                                     peak, "kernel_vs_read"),
            "down": ceiling_entry(dn_bytes, dn_ms * 1e3, stream_ceiling_us(dn_bytes, dev, flush, reps),
                                  peak, "kernel_vs_read")}
        launches_per_step = 2
    elif T <= 8:
        ach = mean_total / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "fused_forward_kernel", "achieved": round(ach, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(ach / peak, 4),
                "traffic": profiled_traffic(name, "fused"), "alg_bytes_per_launch": int(mean_total),
                "avg_launch_us": round(ms * 1e3, 2),
                "note": "step = barrier memset + the fused kernel (CUDA events); bytes over the "
                        "realised union of each route set"}
        roof["stream_ceiling"] = {
            "rule": CEILING_RULE,
            "step": ceiling_entry(mean_total, ms * 1e3,
                                  stream_ceiling_us(mean_total, dev, flush, max(args.steps, 10)),
                                  peak, "step_vs_read")}
        launches_per_step = 1
    elif "gate_up_gemm" not in prefill_stage_ms:
        # T > 8 below the grouped tier's crossover: ceil(T/8) sweeps through the fused kernel
        sb = statistics.mean(sweeps_alg_bytes(s_) for s_ in sets)
        ach = sb / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "fused_forward_kernel (sweeps of <= 8 tokens)",
                "achieved": round(ach, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": None, "alg_bytes_per_launch": int(sb),
                "avg_launch_us": round(ms * 1e3, 2),
                "note": "step = the sweeps (CUDA events); bytes: each sweep's union of experts"}
        launches_per_step = len(sweep_rows(T))
    else:
        # dominant kernel: the gate/up grouped GEMM (two thirds of the flops), timed by the
        # library's stage events; every (token, slot) pair is one GEMM row
        P = T * 8
        gu_flops = 2.0 * 2 * P * wl0.H * wl0.I
        dn_flops = 2.0 * P * wl0.H * wl0.I
        gu_ms = statistics.mean(prefill_stage_ms["gate_up_gemm"])
        dn_ms = statistics.mean(prefill_stage_ms["down_gemm"])
        ach = gu_flops / (gu_ms * 1e-3) / 1e12
        step_tf = (gu_flops + dn_flops) / (ms * 1e-3) / 1e12
        pb = statistics.mean(prefill_alg_bytes(s_) for s_ in sets)
        graded, floor_s = graded_fraction(pb, gu_flops + dn_flops, ms * 1e-3, peak, tpeak)
        roof = {"bound": "tensor", "kernel": "prefill_tw_gemm_kernel (gate/up)",
                "achieved": round(ach, 1), "peak": tpeak, "peak_kind": "measured bf16 dense burst",
                "unit": "TFLOP/s", "frac": round(ach / tpeak, 4),
                "traffic": profiled_traffic(name, "gate_up_gemm"),
                "alg_flops_per_launch": gu_flops, "avg_launch_us": round(gu_ms * 1e3, 2),
                "down": {"kernel": "prefill_tw_gemm_kernel (down)", "alg_flops_per_launch": dn_flops,
                         "avg_launch_us": round(dn_ms * 1e3, 2),
                         "achieved": round(dn_flops / (dn_ms * 1e-3) / 1e12, 1),
                         "frac": round(dn_flops / (dn_ms * 1e-3) / 1e12 / tpeak, 4),
                         "traffic": profiled_traffic(name, "down_gemm")},
                "step": {"alg_flops": gu_flops + dn_flops, "achieved": round(step_tf, 1),
                         "frac": round(step_tf / tpeak, 4), "hbm_bytes": int(pb),
                         "hbm_frac": round(pb / (ms * 1e-3) / 1e9 / peak, 4),
                         "stages_us": {k: round(statistics.mean(v) * 1e3, 1)
                                       for k, v in prefill_stage_ms.items()}},
                "graded": {"frac": round(graded, 4), "floor_us": round(floor_s * 1e6, 1),
                           "rule": "max(alg bytes / HBM peak, FLOPs / bf16 peak) / step time",
                           "target_frac": 0.5},
                "note": "f16 x f16 -> f32 MMA (same nominal rate as bf16); kernel times from the "
                        "library's stage events on the launching stream"}
        # route plan and tile list (three launches from 4096 pairs on, the middle one building the
        # tile list; else two), x prep, gate/up GEMM, activation prep (only without a clamp limit
        # <= 255), down GEMM, combine
        launches_per_step = ((3 if P >= 4096 else 2) + 4
                             + (0 if math.isfinite(inputs.LIMIT) and inputs.LIMIT <= 255 else 1))

    return {
        "workload": name, "value": round(value, 2), "unit": UNIT, "ms_per_step": round(ms, 5),
        "dtype": "e4m3/bf16->f32" if c["fmt"] == "fp8" else "e2m1/bf16->f32",
        "config": {"workload": name, "T": T, "H": wl0.H, "I": wl0.I, "E": E, "topk": 8,
                   "format": "fp8_e4m3_block128" if c["fmt"] == "fp8" else "nvfp4",
                   "routes": c["routes"], "route_sets": N_ROUTE_SETS,
                   "l2": "flushed between steps (write of 2x L2 outside the timed events)",
                   "parallelism": f"replicas x{world}"},
        "effective_weight_gbs": round(call_gbs, 1),
        "hbm_frac_of_peak": round(call_gbs / peak, 4),
        "step_us": step_stats_us(step_ms),
        "output_check": {"bit_identical_steps": same, "steps": args.steps,
                         "against": "an untimed run of the same route set before the timed region",
                         "checksum": f"{checksum:016x}",
                         "checksum_of": "XOR over the 8 route sets of the gate binary's output fold"},
        "stage_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in stage_ms.items() if v},
        "roofline": roof,
        "gpu_launches": launches_per_step * args.steps,
        "graph": ({"ms_per_step": round(statistics.mean(graph_ms), 5),
                   "value": round(T / (statistics.mean(graph_ms) * 1e-3), 2), "unit": UNIT,
                   "note": "the same forward replayed from a CUDA graph per route set"}
                  if graph_ms else {"error": graph_err}),
        "router": None if not router_ms else {
            "us": round(statistics.mean(router_ms) * 1e3, 2), "T": T, "E": E, "H": wl0.H,
            "weight_gbs": round(E * wl0.H * 2 / (statistics.mean(router_ms) * 1e-3) / 1e9, 1),
            "note": "moe_router (logits GEMV/GEMM + top-8), not part of the step"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(statistics.mean(e2e_ms), 5)},
        "clocks": clk,
    }


SIDE_WORKLOADS = ("fp8_batchm", "nvfp4_decode", "fp8_prefill", "nvfp4_prefill")


def bench_ours(args):
    from moe_expert_ffn_histogram_gb300 import _build, capi
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    if args.lib:
        capi._lib = capi.load(args.lib)          # an alternative build of the same library
    else:
        _build.build()
        capi.load()
    peak, peak_kind = load_peaks()
    tpeak = load_tensor_peak()
    banks = {}

    def bank_for(name):
        c = inputs.CONFIGS[name]
        key = (c["fmt"], c["bank_seed"], args.bank_experts)
        if key not in banks:
            banks.clear()                          # one resident bank at a time
            torch.cuda.empty_cache()
            E = c["E"] if args.bank_experts is None else args.bank_experts
            banks[key] = inputs.make_bank(name, dev, experts=None if E == c["E"] else range(E))
        return banks[key]

    name = args.config
    head = measure_workload(name, args, dev, bank_for(name), world, peak, peak_kind, tpeak)
    side = {}
    todo = [w for w in (args.workloads.split(",") if args.workloads else []) if w and w != name]
    # group by bank so that each bank is generated once
    todo.sort(key=lambda w: (inputs.CONFIGS[w]["fmt"] != inputs.CONFIGS[name]["fmt"], w))
    for w in todo:
        r = measure_workload(w, args, dev, bank_for(w), world, peak, peak_kind, tpeak)
        side[w] = {k: r[k] for k in ("value", "unit", "ms_per_step", "dtype", "config", "step_us",
                                     "effective_weight_gbs", "hbm_frac_of_peak", "roofline", "e2e",
                                     "output_check", "stage_us", "gpu_launches", "graph", "router",
                                     "clocks")}

    result = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"],
        "data": "synthetic (seeded N(0,0.02) weights quantised, N(0,1) bf16 activations)",
        "config": head["config"],
        "effective_weight_gbs": head["effective_weight_gbs"],
        "hbm_frac_of_peak": head["hbm_frac_of_peak"],
        "p50_ms": round(head["step_us"]["p50"] / 1e3, 5),
        "p99_ms": round(head["step_us"]["p99"] / 1e3, 5),
        "step_us": head["step_us"],
        "output_check": head["output_check"],
        "stage_us": head["stage_us"],
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "graph": head["graph"],
        "router": head["router"],
        "e2e": head["e2e"],
        "clocks": head["clocks"],
        "workloads": side,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(name, dev, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.config
    c = inputs.CONFIGS[name]
    gen_dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    n_tok = 1 if c["T"] <= 8 else 2
    samples = [oracle_sample(name, i % N_ROUTE_SETS, gen_dev, n_tokens=n_tok)
               for i in range(min(N_ROUTE_SETS, args.warmup + args.steps))]
    for i in range(args.warmup):
        run_oracle(samples[i % len(samples)])
    secs, toks = [], 0
    for i in range(args.steps):
        s = samples[i % len(samples)]
        secs.append(run_oracle(s))
        toks += s["T"]
    value = toks / sum(secs)
    sample_desc = f"{n_tok} token(s) of {name} per step (bounded sample), FP64 C++ oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(secs) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "T": c["T"], "H": c["H"], "I": c["I"], "E": c["E"],
                   "topk": 8, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.hardware_threads(),
                         "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="fp8_decode", choices=sorted(inputs.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket each workload's timed steps with cudaProfilerStart/Stop and one "
                         "NVTX range per step ('<workload>/step'; the library adds a range per "
                         "forward and per stage), for `ncu --profile-from-start off` or "
                         "`--nvtx --nvtx-include`")
    ap.add_argument("--lib", default=None, help="path of an alternative build of the library")
    ap.add_argument("--bank-experts", type=int, default=None,
                    help="use only the first N experts of the bank (small profiling captures)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count T (small profiling captures)")
    ap.add_argument("--workloads", default=",".join(SIDE_WORKLOADS),
                    help="comma-separated further workloads measured in the same run and reported "
                         "under 'workloads' ('' for none)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least 3 untimed warm-up steps, always
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
