#!/usr/bin/env python
"""Throughput of the RDKV hot path on one B300: KV tokens scored + compressed
per second per layer.

A step is one pass of the whole path over one (layer, sequence) pool of the
synthetic Llama-3-8B-shaped layer (32 query heads, 8 KV heads, d = 128,
N = 8192 keys, window of the last 512 queries, 3 bits on average):
row LSE (pass 1), token weights (pass 2), channel weights, sigma_t, V
allocation, sigma_c over kept tokens, K allocation, V and K quantise/pack,
V and K dequantise.  Inputs are resident in HBM; L2 is flushed (256 MB write)
between timed steps and the flush is not timed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own synthetic layer (no data-path
collective: the pools are independent) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens scored+compressed/s per layer (M tok/s) and % of tensor/HBM roofline"
UNIT = "M tok/s"
DEFAULT_WORKLOAD = "full_model_l32_b16_n16384"
FULL_MODEL = "full_model_l32_b16_n16384"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 10 for the full-model batch, 200 for one pool)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--overlap", type=int, default=0,
                    help="full-model batch: 1 runs each layer's post-scoring chain beside the next layer's passes "
                         "(measured no faster: the passes slow down by what the chain saves)")
    ap.add_argument("--layers", type=int, default=None,
                    help="full-model batch: run only this many layers (a reduced case, e.g. for a profiler)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="full-model batch: run only this many sequences per layer (a reduced case)")
    ap.add_argument("--e2e-steps", type=int, default=2, help="end-to-end steps of the full-model batch")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle time for the CPU baseline")
    ap.add_argument("--soak-s", type=float, default=1.0, help="untimed replays before timing (clock samples)")
    ap.add_argument("--trizone", action="store_true",
                    help="time one TriZone decode step over the workload's compressed pool instead")
    ap.add_argument("--core", action="store_true",
                    help="time the KV-CoRE Gram accumulation and spectrum of the workload's K cache instead")
    ap.add_argument("--sculpt", action="store_true",
                    help="time KVSculpt's zone targets (block attention) and ridge values instead")
    ap.add_argument("--chain", action="store_true",
                    help="time the post-scoring chain of one full-model layer call by call instead")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# multi-process plumbing (barrier and max over ranks only; no data exchange)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_group(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(dist, x: float, device=None) -> float:
    """Max of x over ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, steps: int, tokens_per_pool: int, slowest_s: float) -> float:
    """Whole-job throughput in M tok/s: every rank compresses one pool per step
    (weak scaling), and the job takes as long as its slowest rank."""
    return world * steps * tokens_per_pool / slowest_s / 1e6


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, mx, reasons = [], [], set()
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for name, v in zip(self.NAMES, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------
def pass_flops(wl) -> float:
    """2 d flops per visible (query row, key) pair per query head; masked work not counted."""
    pairs = wl.W * (wl.q_pos0 + 1) + wl.W * (wl.W - 1) // 2
    return 2.0 * wl.d * pairs * wl.Hq


def sustained_peak():
    """The measured sustained bf16 rate (a seconds-long GEMM loop under the power cap), if recorded."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)).get("bf16_tflops_sustained")
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1800.0, 6400.0, "fallback"


def fma_clock_mhz() -> float:
    """The SM clock the fp32 FMA peak is taken at: the measured maximum."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p)).get("sm_max_mhz", 2032.0))
    return 2032.0


# the sources that define the scoring passes: their kernels and their launch plan
PASS_SOURCES = ("common.cuh", "score.cuh", "score_host.cuh")


def csrc_hash() -> str:
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "kv_cache_compression_flash_b300", "csrc")
    for f in PASS_SOURCES:
        h.update(open(os.path.join(cdir, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on this source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    cur = csrc_hash()
    for line in open(PROFILE_TRAFFIC):
        f = line.split()
        if len(f) == 4 and f[0] == kernel and f[1] == workload and f[3] == cur:
            return float(f[2])
    return None


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_cores():
    """Threads the oracle uses: its BLAS pool (elementwise NumPy work is single-threaded)."""
    import numpy as np
    np.ones((64, 64)) @ np.ones((64, 64))           # loads the BLAS library
    try:
        import threadpoolctl
        blas = [i["num_threads"] for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if blas:
            return max(blas)
    except ImportError:
        pass
    return len(os.sched_getaffinity(0))


def oracle_group_step(wl, host, g):
    """The oracle's RDKV pass over KV group g alone (G query heads, one KV head)."""
    import numpy as np
    import oracle as O
    G = wl.G
    Q = host["Q"][g * G:(g + 1) * G].float().numpy().astype(np.float64)
    Kx = host["K"][g:g + 1].float().numpy().astype(np.float64)
    Vx = host["V"][g:g + 1].float().numpy().astype(np.float64)
    O.rdkv_compress(Q, Kx, Vx, wl.q_pos0, wl.avg_bits[0])


KVZIP_ORACLE_ROWS = 1024


def time_oracle_kvzip(wl, host, min_seconds=10.0):
    """KVzip+: the oracle's score pass (materialised attention, the norms, the
    column maxima) for one query head over the last KVZIP_ORACLE_ROWS query
    rows against all keys, repeated until min_seconds; its time per visible
    (row, key) pair is scaled to the whole layer (all heads, all N x N causal
    pairs).  Returns (layer tokens/s, slices, seconds)."""
    import numpy as np
    import oracle as O
    R, N, d = KVZIP_ORACLE_ROWS, wl.N, wl.d
    f = lambda t: t.float().numpy().astype(np.float64)
    Kg, Vg, h = f(host["K"][:1]), f(host["V"][:1]), f(host["h"][N - R:])
    slices, t0 = 0, time.perf_counter()
    while True:
        hd = slices % wl.G
        Qh = f(host["Q"][hd:hd + 1, N - R:])
        O.attention_scores(Qh, Kg, N - R, V=Vg, h=h, W_O=f(host["W_O"][:, hd * d:(hd + 1) * d]))
        slices += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    pairs_slice = R * (N - R) + R * (R + 1) // 2
    pairs_layer = wl.Hq * N * (N + 1) // 2
    layer_s = dt / slices / pairs_slice * pairs_layer
    return N / layer_s, slices, dt


def time_oracle(wl, host, min_seconds=10.0):
    """Runs the oracle group by group until min_seconds; returns (layer tokens/s, groups, seconds)."""
    groups, t0 = 0, time.perf_counter()
    while True:
        oracle_group_step(wl, host, groups % wl.Hkv)
        groups += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return wl.N * groups / wl.Hkv / dt, groups, dt


def workload_config(wl):
    c = {"workload": wl.name, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N, "W": wl.W, "d": wl.d,
         "avg_bits": wl.avg_bits[len(wl.avg_bits) // 2], "widths": list(wl.widths), "pools_per_step_per_gpu": 1,
         "l2": "flushed between timed steps (256 MB write, untimed)", "parallelism": "replicas"}
    if wl.mode == "kvzip_plus":
        c.update({"mode": "kvzip_plus", "D": wl.D, "evict_fraction": wl.evict_fraction, "avg_bits": None})
    return c


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    if wl.mode == "kvzip_plus":
        host = synth.make_layer(wl)
        time_oracle_kvzip(wl, host, min_seconds=0.0)          # warm
        v, n, dt = time_oracle_kvzip(wl, host, min_seconds=20.0)
        sample = (f"{n} slices of the fp64 oracle's KVzip+ score pass in {dt:.1f} s (one slice = 1 query head x "
                  f"the last {KVZIP_ORACLE_ROWS} query rows x all {wl.N} keys); time per visible pair scaled to "
                  f"the whole layer")
        value = v / 1e6
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "warmup": 1, "ms_per_step": 1e3 * dt / n, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    pools = FULL_MODEL_ORACLE_POOLS if wl.name == FULL_MODEL else ((0, 0),)
    hosts = [synth.make_layer(wl, l, q) for l, q in pools]
    for i in range(args.warmup):
        oracle_group_step(wl, hosts[i % len(hosts)], (i // len(hosts)) % wl.Hkv)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_group_step(wl, hosts[i % len(hosts)], (i // len(hosts)) % wl.Hkv)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = wl.N / wl.Hkv * args.steps / total / 1e6
    sample = (f"each step = the fp64 oracle's full RDKV pass (scores, weights, allocation, packing) over one "
              f"KV group ({wl.G} query heads, 1 of {wl.Hkv} KV heads, N={wl.N}, W={wl.W}) of the (layer, sequence) "
              f"pools {list(pools)} in turn; counted as N/Hkv layer tokens")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": full_model_config(wl) if wl.name == FULL_MODEL else workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def make_step(wl, host, dev, avg, h_dev=None):
    """The workload's step: RDKV compression, or KVzap's eviction by KVzip+ score."""
    from kv_cache_compression_flash_b300.pipeline import KvzipStep, RdkvLayerStep
    if wl.mode == "kvzip_plus":
        h = h_dev if h_dev is not None else host["h"].to(dev)
        return KvzipStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, wl.evict_fraction, h, host["W_O"].to(dev), device=dev)
    return RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, avg, device=dev)


def run_ours(args):
    import torch

    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_group(world, "nccl")
    L.lib()

    wl = synth.WORKLOADS[args.workload]
    host = synth.make_layer(wl, layer=rank)                  # each rank: its own pool
    in_keys = ("Q", "K", "V", "h") if wl.mode == "kvzip_plus" else ("Q", "K", "V")
    pinned = {k: host[k].pin_memory() for k in in_keys}
    Q, K, V = (pinned[k].to(dev) for k in ("Q", "K", "V"))
    avg = wl.avg_bits[len(wl.avg_bits) // 2]                 # the middle budget of a sweep
    step = make_step(wl, host, dev, avg)
    step.capture(Q, K, V)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    for _ in range(args.warmup):
        flush.zero_()
        step.replay_step()
        flush.zero_()
        step.replay()
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise SystemExit("device error during warm-up")

    clocks = ClockSampler(local).start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:  # clocks under load before the timed region
        for _ in range(20):
            flush.zero_()
            step.replay_step()
        torch.cuda.synchronize()

    # the timed steps: the whole step replayed as one graph, events around it
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        step_evs[i][0].record()
        step.replay_step()
        step_evs[i][1].record()
    torch.cuda.synchronize()
    barrier(dist, dev)
    clk = clocks.stop()
    if L.device_error() != 0:
        raise SystemExit("device error during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in step_evs]
    total_s = reduce_max(dist, sum(step_ms) / 1e3, dev)
    value = replica_value(world, args.steps, wl.N, total_s)

    # the segments (pass 1, pass 2, the rest), each its own graph with events
    # between them, for the per-segment times and the roofline of the pass kernel
    n_seg = min(args.steps, 50)
    for i in range(n_seg):
        flush.zero_()
        step.replay(evs[i])
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise SystemExit("device error while timing the segments")
    seg = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(3)] for i in range(n_seg)]
    seg_avg = [statistics.fmean(s[j] for s in seg) for j in range(3)]

    # ---- roofline of the dominant kernel (the slower scoring pass) -------------
    peak_tf, _, peak_kind = measured_peaks()
    dom = 0 if seg_avg[0] >= seg_avg[1] else 1
    kname = ("lse_pass_kernel", "colreduce_pass_kernel")[dom]
    achieved = pass_flops(wl) / (seg_avg[dom] / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf if peak_tf else None, "peak_kind": f"{peak_kind} bf16 burst",
                "traffic": recorded_traffic(kname, wl.name),
                "duration_note": "segment time: the pass kernel plus its small merge kernel"}

    # a budget sweep: the post-scoring segment (allocation, packing, dequantisation)
    # at every average budget of the workload, the scores computed once
    sweep = {}
    if len(wl.avg_bits) > 1:
        for b in wl.avg_bits:
            sb = step if b == avg else make_step(wl, host, dev, b)
            if sb is not step:
                sb.capture(Q, K, V)
            ts = []
            for i in range(min(args.steps, 20)):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                sb.graphs["rest"].replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            sweep[str(b)] = {"rest_ms": statistics.fmean(ts), "step_ms": seg_avg[0] + seg_avg[1] + statistics.fmean(ts),
                             "M_tok_s": wl.N / ((seg_avg[0] + seg_avg[1] + statistics.fmean(ts)) / 1e3) / 1e6}
        if L.device_error() != 0:
            raise SystemExit("device error during the budget sweep")

    e2e = run_e2e(args, step, pinned, (Q, K, V), flush, dist, dev, world, wl, avg)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.fmean(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl),
        "segments_ms": {"pass1_lse": seg_avg[0], "pass2": seg_avg[1], "rest": seg_avg[2]},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": step.kernel_launches() * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"], "window": "1 s soak of the same step, then the timed steps"},
    }
    if sweep:
        out["budget_sweep"] = sweep
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl.mode == "kvzip_plus":
        v, n, dt = time_oracle_kvzip(wl, host)
        out["cpu_baseline"] = {"value": v / 1e6, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
                               "sample": f"{n} slices of the fp64 oracle's KVzip+ score pass in {dt:.1f} s (one "
                                         f"slice = 1 query head x the last {KVZIP_ORACLE_ROWS} query rows x all "
                                         f"{wl.N} keys); time per visible pair scaled to the whole layer"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, groups, dt = time_oracle(wl, host)
        out["cpu_baseline"] = {"value": v / 1e6, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
                               "sample": f"{groups} KV groups of this layer through the fp64 oracle in {dt:.1f} s "
                                         f"(one group = {wl.G} query heads x 1 KV head; N/Hkv tokens each)"}
    if rank == 0:
        print(json.dumps(out))
        log_result(out)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_e2e(args, step, pinned, dev_inputs, flush, dist, dev, world, wl, avg):
    """Pinned host Q, K, V in; the packed streams and widths a caller keeps, out.

    Two pools in flight, as a serving loop would run them: while step i
    computes, step i+1's inputs cross the host link and step i-1's streams come
    back.  Every step still copies its own inputs in and its own result out
    (the used part of every stream, the counts and the widths); the time is
    the wall clock over all steps.  Inputs arrive by copy every step, so no L2
    flush is needed between steps."""
    import torch
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in pinned)
    # the second pool: its own inputs, outputs and captured graphs
    step2 = make_step(wl, {"W_O": step.W_O.cpu()} if hasattr(step, "W_O") else None, dev, avg,
                      h_dev=torch.empty_like(step.h) if hasattr(step, "h") else None)
    inputs2 = tuple(torch.empty_like(x) for x in dev_inputs)
    for x, k in zip(inputs2, ("Q", "K", "V")):
        x.copy_(pinned[k])
    step2.capture(*inputs2)
    slots = [(step, dev_inputs), (step2, inputs2)]

    def landing(st):
        streams = (st.v_streams, st.k_streams)
        return {"bits_v": torch.empty(st.bits_v.numel(), dtype=torch.uint8, pin_memory=True),
                "bits_k": torch.empty(st.bits_k.numel(), dtype=torch.uint8, pin_memory=True),
                "counts": [torch.empty(8, dtype=torch.int64, pin_memory=True) for _ in streams],
                "streams": [[tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                                   for t in (s.codes[i], s.scales[i], s.ids[i], s.goff[i])) for i in range(4)]
                            for s in streams]}
    lands = [landing(st) for st, _ in slots]
    cp, comp, out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_comp = [torch.cuda.Event() for _ in slots]
    ev_in = [torch.cuda.Event() for _ in slots]
    ev_out = [torch.cuda.Event() for _ in slots]
    d2h = [0]

    def issue_step(i):
        s = i % 2
        st, (Q, K, V) = slots[s]
        land = lands[s]
        if i >= 2:
            cp.wait_event(ev_comp[s])          # step i-2 no longer reads these inputs
        with torch.cuda.stream(cp):
            Q.copy_(pinned["Q"], non_blocking=True)
            K.copy_(pinned["K"], non_blocking=True)
            V.copy_(pinned["V"], non_blocking=True)
            if "h" in pinned:                  # KVzip+: the window's hidden states are an input too
                st.h.copy_(pinned["h"], non_blocking=True)
            ev_in[s].record(cp)
        comp.wait_event(ev_in[s])
        if i >= 2:
            comp.wait_event(ev_out[s])         # step i-2's streams have left
        with torch.cuda.stream(comp):
            st.replay_step()
            for j, sm in enumerate((st.v_streams, st.k_streams)):
                land["counts"][j].copy_(sm.counts, non_blocking=True)
            land["bits_v"].copy_(st.bits_v, non_blocking=True)
            land["bits_k"].copy_(st.bits_k, non_blocking=True)
            ev_comp[s].record(comp)

    def drain_step(i):
        s = i % 2
        st, _ = slots[s]
        land = lands[s]
        ev_comp[s].synchronize()               # the counts of step i are on the host
        nbytes = 2 * 64 + st.bits_v.numel() + st.bits_k.numel()
        out.wait_event(ev_comp[s])
        with torch.cuda.stream(out):
            for j, sm in enumerate((st.v_streams, st.k_streams)):
                c = land["counts"][j].tolist()
                for k, wd in enumerate((2, 4, 8, 16)):
                    nu, ng = c[k], c[4 + k]
                    lc, ls, li, lg = land["streams"][j][k]
                    lc[:ng * 8 * wd].copy_(sm.codes[k][:ng * 8 * wd], non_blocking=True)
                    li[:nu].copy_(sm.ids[k][:nu], non_blocking=True)
                    lg[:nu].copy_(sm.goff[k][:nu], non_blocking=True)
                    nbytes += ng * 8 * wd + nu * 12
                    if wd != 16:
                        ls[:ng].copy_(sm.scales[k][:ng], non_blocking=True)
                        nbytes += ng * 2
            ev_out[s].record(out)
        d2h[0] = nbytes

    for i in range(2):                         # warm the two-pool loop
        issue_step(i)
        if i:
            drain_step(i - 1)
    drain_step(1)
    torch.cuda.synchronize()
    barrier(dist, dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        issue_step(i)
        if i:
            drain_step(i - 1)
    drain_step(args.steps - 1)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    barrier(dist, dev)
    total = reduce_max(dist, elapsed, dev)
    return {"value": replica_value(world, args.steps, wl.N, total), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h[0],
            "path": "pinned host Q,K,V -> device, graph replay of the C-ABI calls, packed streams + widths -> "
                    "host; two pools in flight (copies of one step overlap the compute of the next)"}


def run_trizone(args):
    """One decode step over a compressed pool (TriZone zones A, B and C), timed
    with events around a graph replay, L2 flushed before each step.  The pool is
    the workload's layer through the full RDKV path; the query is the last
    window row; zone C holds 64 new tokens."""
    import torch
    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    t = synth.make_layer(wl)
    Q, K, V = (t[k].to(dev) for k in ("Q", "K", "V"))
    avg = wl.avg_bits[len(wl.avg_bits) // 2]
    step = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, avg, device=dev, dequant=False)
    step.run(Q, K, V)
    idx = L.trizone_index(step.k_streams, step.v_streams, step.bits_v)
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise SystemExit("device error while compressing")
    q = Q[:, -1, :].contiguous()
    g = torch.Generator().manual_seed(7)
    nc_cap, nc = 128, 64
    kn = torch.randn(wl.Hkv, nc_cap, wl.d, generator=g).bfloat16().to(dev)
    vn = torch.randn(wl.Hkv, nc_cap, wl.d, generator=g).bfloat16().to(dev)
    n_new = torch.tensor([nc], dtype=torch.int32, device=dev)
    out = torch.empty(wl.Hq, wl.d, device=dev)
    lse = torch.empty(wl.Hq, device=dev)
    ws = L.Workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)

    def graph_of(fn):
        with torch.cuda.stream(s):
            fn()
            fn()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s):
                fn()
        torch.cuda.synchronize()
        return gr

    def timed(gr):
        for _ in range(args.warmup):
            gr.replay()
        ts = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                flush.zero_()
                e0.record(s)
                gr.replay()
                e1.record(s)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    us = timed(graph_of(lambda: L.trizone_decode(q, step.k_streams, step.v_streams, idx, kn, vn, n_new,
                                                 out=out, lse=lse, ws=ws)))
    if L.device_error() != 0:
        raise SystemExit("device error during the decode")
    # dense bf16 decode over the uncompressed cache plus zone C, through the library
    # attention of PyTorch: context for the compressed step, not a baseline of the method
    Kd = torch.cat([K, kn[:, :nc]], dim=1).unsqueeze(0)
    Vd = torch.cat([V, vn[:, :nc]], dim=1).unsqueeze(0)
    qd = q.view(1, wl.Hq, 1, wl.d)
    dense_us = timed(graph_of(lambda: torch.nn.functional.scaled_dot_product_attention(qd, Kd, Vd, enable_gqa=True)))
    counts = [step.v_streams.counts.cpu().tolist(), step.k_streams.counts.cpu().tolist()]
    packed = sum(c[4 + i] * 8 * w + (2 * c[4 + i] if w < 16 else 0)
                 for c in counts for i, w in enumerate((2, 4, 8, 16)))
    nkept = int((step.bits_v > 0).sum().item())
    algo = packed + nkept + 2 * wl.Hkv * nc * wl.d * 2 + wl.Hq * wl.d * (2 + 4)
    _, peak_gbs, peak_kind = measured_peaks()
    achieved = algo / (us * 1e-6) / 1e9
    print(json.dumps({
        "metric": "TriZone decode step latency (one query per head, compressed pool + 64 new tokens)",
        "value": us, "unit": "us", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N, "d": wl.d, "avg_bits": avg,
                   "kept_tokens": nkept, "zone_c_tokens": nc, "l2": "flushed before each step (untimed)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                     "frac": achieved / peak_gbs if peak_gbs else None, "peak_kind": f"{peak_kind} copy",
                     "algorithmic_bytes": algo},
        "dense_bf16_sdpa_us": dense_us, "gpu_launches": 2 * args.steps,
    }))
    return 0


def run_core(args):
    """KV-CoRE over the workload's K cache: kvs_gram (all tokens of every KV
    head) and kvs_spectrum, each timed with events, L2 flushed before each."""
    import torch
    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    K = synth.make_layer(wl)["K"].to(dev)
    G = torch.empty(wl.Hkv, wl.d, wl.d, dtype=torch.float32, device=dev)
    ws = L.Workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        L.gram(K, out=G, ws=ws)
        L.spectrum(G)
    torch.cuda.synchronize()
    tg, ts = [], []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        L.gram(K, out=G, ws=ws)
        e1.record()
        sigma, ner, rank = L.spectrum(G)
        e2.record()
        torch.cuda.synchronize()
        tg.append(e0.elapsed_time(e1) * 1e3)
        ts.append(e1.elapsed_time(e2) * 1e3)
    if L.device_error() != 0:
        raise SystemExit("device error")
    gram_us = statistics.median(tg)
    byts = K.numel() * 2
    flops = 2.0 * wl.Hkv * wl.N * wl.d * wl.d
    peak_tf, peak_gbs, peak_kind = measured_peaks()
    print(json.dumps({
        "metric": "KV-CoRE Gram accumulation over the K cache (all KV heads)", "value": gram_us, "unit": "us",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": wl.name, "Hkv": wl.Hkv, "N": wl.N, "d": wl.d,
                                        "l2": "flushed before each step (untimed)"},
        "roofline": {"bound": "hbm", "achieved": byts / (gram_us * 1e-6) / 1e9, "peak": peak_gbs, "unit": "GB/s",
                     "frac": byts / (gram_us * 1e-6) / 1e9 / peak_gbs if peak_gbs else None,
                     "peak_kind": f"{peak_kind} copy", "algorithmic_bytes": byts,
                     "tensor_tflops": flops / (gram_us * 1e-6) / 1e12},
        "spectrum_us": statistics.median(ts), "ner": [round(float(x), 4) for x in ner.cpu()],
        "rank": [int(x) for x in rank.cpu()], "gpu_launches": 3 * args.steps,
    }))
    return 0


def run_chain(args):
    """The post-scoring chain of one layer of the full-model batch (its 16
    sequences as pools, or --seqs of them), call by call: each call timed
    with events, L2 flushed before each (untimed); its algorithmic bytes
    over its time, against the measured HBM copy rate.  The whole chain as the
    step runs it (two streams) is timed beside the calls."""
    import torch
    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep
    wl = synth.WORKLOADS[FULL_MODEL]
    P = args.seqs or wl.seqs
    dev = torch.device("cuda", 0)
    x = synth.make_pools(wl, 0, range(P), device=dev)
    Q, K, V = x["Q"], x["K"], x["V"]
    st = RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, wl.avg_bits[0], device=dev, n_pools=P)
    st.run(Q, K, V)
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise SystemExit("device error")
    Hq, Hkv, N, W, d = st.shape
    X4 = (P, Hkv, N, d)
    bv, bk = st.pool_bits()
    ws = st.ws
    calls = [
        ("sigma_t", lambda: L.unit_rms(V.view(P * Hkv, N, d), 0, out=st.sig_t, ws=ws["rms0"])),
        ("alloc_v", lambda: L.allocate_bits_pools(st.out["w_t"].view(P, -1), st.sig_t.view(P, -1), st.B_v,
                                                  out=bv, ws=ws["av"])),
        ("channel_stats", lambda: L.channel_stats(Q.view(P * Hq, W, d), K.view(P * Hkv, N, d), st.bits_v,
                                                  out_wc=st.w_c, out_sigma=st.sig_c)),
        ("alloc_k", lambda: L.allocate_bits_pools(st.w_c.view(P, -1), st.sig_c.view(P, -1), st.B_k, out=bk,
                                                  ws=ws["ak"])),
        ("pack_v", lambda: L.quantize_pack_pools(V.view(X4), 0, st.bits_v, None, st.v_streams, ws=ws["pv"])),
        ("pack_k", lambda: L.quantize_pack_pools(K.view(X4), 1, st.bits_k, st.bits_v, st.k_streams, ws=ws["pk"])),
        ("dequant_v", lambda: L.dequantize_pools(st.v_streams, st.bits_v, None, out=st.v_hat.view(X4), ws=ws["dv"])),
        ("dequant_k", lambda: L.dequantize_pools(st.k_streams, st.bits_k, st.bits_v, out=st.k_hat.view(X4),
                                                 ws=ws["dk"])),
        ("chain", lambda: st.rest(Q, K, V)),
    ]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        for _, f in calls:
            f()
    torch.cuda.synchronize()
    times = {n: [] for n, _ in calls}
    for _ in range(args.steps):
        for n, f in calls:
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            times[n].append(e0.elapsed_time(e1))
    if L.device_error() != 0:
        raise SystemExit("device error")
    # algorithmic bytes: what each call must read and write once
    U_v, U_k = P * Hkv * N, P * Hkv * d
    cache = U_v * d * 2                                   # one bf16 cache (K or V) of the layer
    kept = int((st.bits_v > 0).sum())                     # kept tokens (V rows stored, K columns' length)

    def streams_bytes(s):
        cnt = s.counts.view(P, 8).sum(0).tolist()         # units, groups per width slot
        return sum(cnt[4 + i] * 8 * w + (2 * cnt[4 + i] if w < 16 else 0) + 12 * cnt[i]
                   for i, w in enumerate((2, 4, 8, 16)))
    sv, sk = streams_bytes(st.v_streams), streams_bytes(st.k_streams)
    algo = {"sigma_t": cache + 4 * U_v, "alloc_v": 9 * U_v,
            "channel_stats": cache + P * Hq * W * d * 2 + U_v + 8 * U_k, "alloc_k": 9 * U_k,
            "pack_v": kept * d * 2 + sv + U_v, "pack_k": kept * d * 2 + sk + U_v + U_k,
            "dequant_v": sv + U_v + U_v * d * 4, "dequant_k": sk + U_v + U_k + U_v * d * 4}
    algo["chain"] = sum(algo.values())
    _, peak_gbs, peak_kind = measured_peaks()
    out_calls = {}
    for n, _ in calls:
        ms = statistics.median(times[n])
        gbs = algo[n] / (ms * 1e-3) / 1e9
        out_calls[n] = {"ms": ms, "algorithmic_bytes": algo[n], "GB/s": gbs,
                        "frac": gbs / peak_gbs if peak_gbs else None}
    print(json.dumps({
        "metric": "post-scoring chain of one full-model layer, per call", "value": out_calls["chain"]["ms"],
        "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic (seeded, drawn on the device)",
        "config": {"workload": wl.name, "layer": 0, "pools": P, "Hkv": Hkv, "N": N, "d": d, "avg_bits": wl.avg_bits[0],
                   "kept_tokens": kept, "l2": "flushed before each call (untimed)"},
        "peak": {"GB/s": peak_gbs, "kind": f"{peak_kind} copy"}, "calls": out_calls,
        "gpu_launches": (st.kernel_launches() - scoring_launches(st)) * args.steps,
    }))
    return 0


def scoring_launches(st):
    """Launches of one step that belong to its scoring call (not in the chain)."""
    from kv_cache_compression_flash_b300 import _lib as L
    Hq, Hkv, N, W, d = st.shape
    P = st.n_pools
    return L.score_plan_info(P * Hq, P * Hkv, W, N, d, mode=st.BOTH_MODE)[4]


def run_sculpt(args):
    """KVSculpt over the workload's compression zone (all but the window): the
    targets Y and lse of the window queries over the zone (kvs_block_attention)
    and the ridge values of 512 compressed pairs per KV head whose keys are
    every (zone / 512)-th key of the zone (kvs_ridge_values), each timed with
    events, L2 flushed before each step.  The block attention runs on the
    tensor cores (bf16 products, fp32 sums), the ridge on the FMA pipes."""
    import torch
    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    t = synth.make_layer(wl)
    Q, K, V = t["Q"].to(dev), t["K"].to(dev), t["V"].to(dev)
    n_block = wl.N - wl.W
    G = wl.Hq // wl.Hkv
    R, k = G * wl.W, min(512, n_block)
    stride = max(1, n_block // k)
    Kc = K[:, :n_block:stride][:, :k].contiguous()
    lam = 0.05 * R / k  # a twentieth of lambda_max(A^T A) when the attention is spread evenly
    Y = torch.empty(wl.Hq, wl.W, wl.d, dtype=torch.float32, device=dev)
    Vc = torch.empty(wl.Hkv, k, wl.d, dtype=torch.float32, device=dev)
    ws = L.Workspace()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(evs=None):
        if evs:
            evs[0].record()
        _, lse = L.block_attention(Q, K, V, n_block, q_pos0=wl.q_pos0, out=Y)
        if evs:
            evs[1].record()
        L.ridge_values(Q.view(wl.Hkv, R, wl.d), Kc, Y.view(wl.Hkv, R, wl.d), lam, out=Vc, ws=ws)
        if evs:
            evs[2].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ta, tr = [], []
    for _ in range(args.steps):
        flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        step(evs)
        torch.cuda.synchronize()
        ta.append(evs[0].elapsed_time(evs[1]) * 1e3)
        tr.append(evs[1].elapsed_time(evs[2]) * 1e3)
    if L.device_error() != 0:
        raise SystemExit("device error")
    attn_us, ridge_us = statistics.median(ta), statistics.median(tr)
    # algorithmic flops: q.k and p.v per visible (row, key) pair; the ridge's
    # logits, A^T A, A^T Y, Cholesky and the two triangular solves
    n_vis = sum(min(n_block, wl.q_pos0 + r + 1) for r in range(wl.W))
    attn_flops = 4.0 * wl.Hq * n_vis * wl.d
    ridge_flops = wl.Hkv * (2.0 * R * k * wl.d + 2.0 * R * k * k + 2.0 * R * k * wl.d + k ** 3 / 3.0
                            + 2.0 * k * k * wl.d)
    peak_tf, _, peak_kind = measured_peaks()
    print(json.dumps({
        "metric": "KVSculpt zone targets + ridge values (all KV heads)", "value": attn_us + ridge_us, "unit": "us",
        "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "f32",
        "data": "synthetic", "config": {"workload": wl.name, "Hq": wl.Hq, "Hkv": wl.Hkv, "W": wl.W, "N": wl.N,
                                        "d": wl.d, "n_block": n_block, "R": R, "k": k,
                                        "l2": "flushed before each step (untimed)"},
        "block_attention_us": attn_us, "ridge_values_us": ridge_us,
        "roofline": {"bound": "tensor", "achieved": attn_flops / (attn_us * 1e-6) / 1e12, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": attn_flops / (attn_us * 1e-6) / 1e12 / peak_tf,
                     "peak_kind": f"{peak_kind} bf16 dense", "kernel": "block_attention_tc_kernel",
                     "algorithmic_flops": attn_flops},
        "ridge_tflops": ridge_flops / (ridge_us * 1e-6) / 1e12,
        "ridge_fma_frac": ridge_flops / (ridge_us * 1e-6) / (148 * 128 * 2 * fma_clock_mhz() * 1e6),
        # block attention, then the ridge's softmax, A^T A + A^T Y and the cluster solve
        "gpu_launches": 4 * args.steps,
    }))
    return 0


# ---------------------------------------------------------------------------
# the full-model batch: 32 layers x 16 sequences, every layer one pooled step
# ---------------------------------------------------------------------------
def full_model_inputs(wl, dev, layers):
    """Every layer's Q, K, V for all its sequences, drawn on the device (seeded)."""
    from kv_cache_compression_flash_b300 import synth
    return [synth.make_pools(wl, l, range(wl.seqs), device=dev) for l in range(layers)]


def oracle_pool_groups(wl, pools, seconds):
    """The oracle's RDKV pass, one KV group at a time, over sampled (layer,
    sequence) pools of the batch until `seconds`; (layer tokens/s, groups, s)."""
    from kv_cache_compression_flash_b300 import synth
    hosts = [synth.make_layer(wl, l, q) for l, q in pools]
    groups, t0 = 0, time.perf_counter()
    while True:
        oracle_group_step(wl, hosts[groups % len(hosts)], (groups // len(hosts)) % wl.Hkv)
        groups += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return wl.N * groups / wl.Hkv / dt, groups, dt


FULL_MODEL_ORACLE_POOLS = ((0, 0), (15, 15), (31, 0))


def full_model_config(wl):
    return {"workload": wl.name, "layers": wl.layers, "seqs": wl.seqs, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N,
            "W": wl.W, "d": wl.d, "avg_bits": wl.avg_bits[0], "pools_per_step_per_gpu": wl.layers * wl.seqs,
            "pools_per_launch": wl.seqs, "tokens_per_step": wl.layers * wl.seqs * wl.N,
            "l2": "inputs ({:.1f} GB) far larger than L2; no flush".format(
                wl.layers * wl.seqs * (wl.Hq * wl.W + 2 * wl.Hkv * wl.N) * wl.d * 2 / 1e9),
            "parallelism": "replicas"}


def run_full_model(args):
    """One step = every layer of the batch through the whole RDKV path: per
    layer one pooled step over its 16 sequences (pass 1, pass 2, w_c, sigma_t,
    V allocation per pool, sigma_c, K allocation per pool, V and K pack and
    dequantise).  All 32 layers' inputs (38.7 GB) are resident in HBM before
    the timed region; they are far larger than L2, so no flush is needed.
    Events on the launching stream bracket each layer's two scoring passes,
    which gives the pass kernels' times inside the timed steps."""
    import torch
    from kv_cache_compression_flash_b300 import _lib as L
    from kv_cache_compression_flash_b300 import synth
    from kv_cache_compression_flash_b300.pipeline import RdkvLayerStep

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_group(world, "nccl")
    L.lib()
    wl = synth.WORKLOADS[FULL_MODEL]
    reduced = args.layers is not None or args.seqs is not None
    if reduced:   # a smaller slice of the batch (profiling); the line says so in its config
        wl = wl.small(layers=args.layers or wl.layers, seqs=args.seqs or wl.seqs)
    layers, P = wl.layers, wl.seqs
    t_gen = time.perf_counter()
    inputs = full_model_inputs(wl, dev, layers)
    torch.cuda.synchronize()
    gen_s = time.perf_counter() - t_gen
    avg = wl.avg_bits[0]
    steps = [RdkvLayerStep(wl.Hq, wl.Hkv, wl.N, wl.W, wl.d, avg, device=dev, n_pools=P) for _ in range(2)]
    main = torch.cuda.current_stream()
    # With overlap, layer l's post-scoring chain runs on a second stream while
    # layer l+1's scoring passes run on the first (the two step objects take
    # the layers in turn; a layer's passes wait until the chain of the layer
    # two back, which used the same buffers, is done).
    rest_stream = torch.cuda.Stream(device=dev)
    scored = [torch.cuda.Event() for _ in range(2)]
    rested = [torch.cuda.Event() for _ in range(2)]

    def one_step(evs=None):
        for l in range(layers):
            st, x = steps[l % 2], inputs[l]
            if args.overlap and l >= 2:
                main.wait_event(rested[l % 2])
            if evs is not None:
                evs[l][0].record(main)
            st.pass1(x["Q"], x["K"], x["V"])
            if evs is not None:
                evs[l][1].record(main)
            st.pass2(x["Q"], x["K"], x["V"])
            if evs is not None:
                evs[l][2].record(main)
            if args.overlap:
                scored[l % 2].record(main)
                rest_stream.wait_event(scored[l % 2])
                with torch.cuda.stream(rest_stream):
                    st.rest(x["Q"], x["K"], x["V"], stream=rest_stream)
                rested[l % 2].record(rest_stream)
            else:
                st.rest(x["Q"], x["K"], x["V"])
        if args.overlap:
            main.wait_stream(rest_stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise SystemExit("device error during warm-up")
    clocks = ClockSampler(local).start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        one_step()
        torch.cuda.synchronize()
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    ev_pass = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(layers)]
               for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize()
    for i in range(args.steps):
        ev_step[i][0].record(main)
        one_step(ev_pass[i])
        ev_step[i][1].record(main)
    torch.cuda.synchronize()
    barrier(dist, dev)
    clk = clocks.stop()
    if L.device_error() != 0:
        raise SystemExit("device error during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    total_s = reduce_max(dist, sum(step_ms) / 1e3, dev)
    tokens_per_step = layers * P * wl.N                      # layer-tokens: every layer of every sequence
    value = world * args.steps * tokens_per_step / total_s / 1e6
    p1 = statistics.fmean(e[l][0].elapsed_time(e[l][1]) for e in ev_pass for l in range(layers))
    p2 = statistics.fmean(e[l][1].elapsed_time(e[l][2]) for e in ev_pass for l in range(layers))
    rest = statistics.fmean(step_ms) / layers - p1 - p2   # with overlap: the part of the chain not hidden

    peak_tf, _, peak_kind = measured_peaks()
    peak_sus = sustained_peak()
    dom_ms, kname = (p1, "lse_pass_kernel") if p1 >= p2 else (p2, "colreduce_pass_kernel")
    flops = pass_flops(wl) * P                               # one launch covers the layer's 16 pools
    achieved = flops / (dom_ms / 1e3) / 1e12
    peak = peak_sus if peak_sus else peak_tf
    roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak if peak else None,
                "peak_kind": f"{peak_kind} bf16 {'sustained' if peak_sus else 'burst'} (the pass runs inside a "
                             f"seconds-long step)",
                "frac_of_burst": achieved / peak_tf if peak_tf else None,
                "flops_per_launch": flops, "launch_ms": dom_ms,
                "traffic": recorded_traffic(kname, wl.name),
                "duration_note": "CUDA events on the launching stream around each layer's pass (the pass kernel "
                                 "plus its small merge kernel), averaged over every layer of the timed steps"}
    launches = sum(st.kernel_launches() for st in steps[:1]) * layers + layers   # + pass 2's offsets kernel
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.fmean(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, drawn on the device)",
        "config": dict(full_model_config(wl), **({"reduced": True} if reduced else {})),
        "segments_ms_per_layer": {"pass1_lse": p1, "pass2_token_weights": p2, "rest": rest,
                                  "overlap": bool(args.overlap)},
        "roofline": roofline,
        "gpu_launches": launches * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"], "window": f"{args.soak_s:.0f} s soak of the same step, then the timed steps"},
        "input_generation_s": gen_s,
    }
    if not args.no_e2e:
        out["e2e"] = run_full_model_e2e(args, wl, inputs, steps, dist, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, groups, dt = oracle_pool_groups(wl, FULL_MODEL_ORACLE_POOLS, args.cpu_seconds)
        out["cpu_baseline"] = {
            "value": v / 1e6, "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
            "sample": f"{groups} KV groups of the (layer, sequence) pools {list(FULL_MODEL_ORACLE_POOLS)} through the "
                      f"fp64 oracle in {dt:.1f} s (one group = {wl.G} query heads x 1 KV head, N/Hkv layer tokens "
                      f"each); the whole batch's rate is extrapolated from these groups"}
    if rank == 0:
        print(json.dumps(out))
        log_result(out)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_full_model_e2e(args, wl, dev_inputs, steps, dist, dev, world):
    """The same step through the same calls with HOST buffers: every layer's
    Q, K, V come from pinned host memory and its packed streams, widths and
    counts go back to pinned host memory, every copy inside the timed region.
    Two layers in flight: layer l's inputs cross the host link while layer
    l-1 computes and layer l-2's streams come back."""
    import torch
    layers, P = wl.layers, wl.seqs
    host = []
    for l in range(layers):
        try:
            host.append({k: dev_inputs[l][k].cpu().pin_memory() for k in ("Q", "K", "V")})
        except RuntimeError:            # not enough pinnable host memory: reuse the layers already there
            break
    n_host = len(host)
    if n_host == 0:
        return {"value": None, "unit": UNIT, "error": "no pinned host memory for the inputs"}
    slots = [{k: torch.empty_like(dev_inputs[0][k]) for k in ("Q", "K", "V")} for _ in range(2)]
    cp, comp, out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def landing(st):
        return {"bits_v": torch.empty(st.bits_v.numel(), dtype=torch.uint8, pin_memory=True),
                "bits_k": torch.empty(st.bits_k.numel(), dtype=torch.uint8, pin_memory=True),
                "counts": [torch.empty(st.v_streams.counts.numel(), dtype=torch.int64, pin_memory=True)
                           for _ in range(2)],
                "streams": [[tuple(torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
                                   for t in (s.codes[i], s.scales[i], s.ids[i], s.goff[i])) for i in range(4)]
                            for s in (st.v_streams, st.k_streams)]}
    lands = [landing(st) for st in steps]
    h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in ("Q", "K", "V")) * layers
    d2h = [0]

    def issue(l):
        s = l % 2
        st, x, hx, land = steps[s], slots[s], host[l % n_host], lands[s]
        if l >= 2:
            cp.wait_event(ev_comp[s])          # layer l-2 no longer reads this slot
        with torch.cuda.stream(cp):
            for k in ("Q", "K", "V"):
                x[k].copy_(hx[k], non_blocking=True)
            ev_in[s].record(cp)
        comp.wait_event(ev_in[s])
        if l >= 2:
            comp.wait_event(ev_out[s])         # layer l-2's streams have left
        with torch.cuda.stream(comp):
            st.run(x["Q"], x["K"], x["V"], stream=comp)
            for j, sm in enumerate((st.v_streams, st.k_streams)):
                land["counts"][j].copy_(sm.counts, non_blocking=True)
            land["bits_v"].copy_(st.bits_v, non_blocking=True)
            land["bits_k"].copy_(st.bits_k, non_blocking=True)
            ev_comp[s].record(comp)

    def drain(l):
        s = l % 2
        st, land = steps[s], lands[s]
        ev_comp[s].synchronize()               # this layer's counts are on the host
        nbytes = land["bits_v"].numel() + land["bits_k"].numel() + 2 * 8 * 8 * P
        out.wait_event(ev_comp[s])
        with torch.cuda.stream(out):
            for j, sm in enumerate((st.v_streams, st.k_streams)):
                c = land["counts"][j].view(P, 8).tolist()
                for i, wd in enumerate((2, 4, 8, 16)):
                    lc, ls, li, lg = land["streams"][j][i]
                    cu, cg = sm.cap_units[i], sm.cap_groups[i]
                    for q in range(P):
                        nu, ng = c[q][i], c[q][4 + i]
                        g0, u0 = q * cg, q * cu
                        lc[g0 * 8 * wd:(g0 + ng) * 8 * wd].copy_(sm.codes[i][g0 * 8 * wd:(g0 + ng) * 8 * wd],
                                                                 non_blocking=True)
                        li[u0:u0 + nu].copy_(sm.ids[i][u0:u0 + nu], non_blocking=True)
                        lg[u0:u0 + nu].copy_(sm.goff[i][u0:u0 + nu], non_blocking=True)
                        nbytes += ng * 8 * wd + nu * 12
                        if wd != 16:
                            ls[g0:g0 + ng].copy_(sm.scales[i][g0:g0 + ng], non_blocking=True)
                            nbytes += ng * 2
            ev_out[s].record(out)
        return nbytes

    def run_steps(n):
        total = 0
        for i in range(n):
            tot = 0
            for l in range(layers):
                issue(l)
                if l:
                    tot += drain(l - 1)
            tot += drain(layers - 1)
            total = tot
        return total

    run_steps(1)                               # warm
    torch.cuda.synchronize()
    barrier(dist, dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    d2h[0] = run_steps(args.e2e_steps)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    barrier(dist, dev)
    total = reduce_max(dist, elapsed, dev)
    tokens = layers * P * wl.N
    return {"value": world * args.e2e_steps * tokens / total / 1e6, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h[0], "steps": args.e2e_steps,
            "host_layers": n_host,
            "path": "pinned host Q,K,V of every layer -> device, the C-ABI calls of the pooled step, packed "
                    "streams + widths + counts -> pinned host; two layers in flight (copy in / compute / copy out "
                    "on three streams)"}


def log_result(line):
    """Appends the line to the results log (bench_results.jsonl beside bench.py, one JSON line per run)."""
    try:
        with open(os.path.join(ROOT, "bench_results.jsonl"), "a") as f:
            f.write(json.dumps(line) + "\n")
    except OSError:
        pass


def main(argv=None):
    args = parse_args(argv)
    side_leg = args.trizone or args.core or args.sculpt or args.chain
    if args.steps is None:
        args.steps = 10 if (args.workload == FULL_MODEL and not side_leg) else 20 if args.chain else 200
    if args.impl == "reference":
        return run_reference(args)
    if args.chain:
        return run_chain(args)
    if args.workload == FULL_MODEL and not side_leg:
        return run_full_model(args)
    if args.trizone:
        return run_trizone(args)
    if args.core:
        return run_core(args)
    if args.sculpt:
        return run_sculpt(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
