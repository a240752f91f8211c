"""Benchmark: batch-1 decode over a 64-layer q8_0 (or f16) GQA KV cache on GB300.

Workload (default): 64 layers, 40 query heads / 8 KV heads, head_dim 128,
q8_0 K/V from N(0,1)*0.5, RoPE base 1e6, n_kv = 16384.  One step is one
decode token through the layer stack: for every layer, quantise-on-append of
the new K/V row, then split-K decode attention over all n_kv rows, as one
fused launch (kvc_decode_step).  The step is captured once as a CUDA graph of
64 launches and replayed; each replay
rewrites row n_kv-1 with the same values, so every step does the full work of
a decode step at n_kv.  The 64 layers read 2.28 GB of distinct KV per step,
far more than the 129 MB L2, so nothing is served from L2 across steps.

Printed: one JSON line (rank 0).  value = KV GB/s (algorithmic KV bytes of
the step / device time of the step); roofline = the attention kernel alone
(bytes per launch / average launch time) against the measured HBM copy
bandwidth; e2e = the same metric with the step's inputs copied from pinned
host memory and its outputs copied back inside the timed region; host = the
host-resident pipeline at 32k (steps/s, H2D GB/s against the measured pinned
link); cpu_baseline = the CPU oracle on a bounded sample, on the host cores;
step_two_calls = the same step with a separate append kernel per layer.

--impl reference times the CPU oracle (there is no other reference implementation) on
the same workload, a bounded sample per step.
Multi-GPU: replicas only (one independent cache per rank, no collective on
the data path); value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s (% of HBM peak); host-KV steps/s at 32k (% of PCIe bw)"
GB = 1e9


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--n-kv", type=int, default=16384)
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--type", default="q8_0", choices=["q8_0", "f16"])
    ap.add_argument("--host-n", type=int, default=32768, help="host-resident context (0 = skip)")
    ap.add_argument("--host-steps", type=int, default=4)
    ap.add_argument("--cpu-sample-layers", type=int, default=4)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="repeat the oracle sample for at least this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the variant, ragged and churn measurements")
    ap.add_argument("--churn-cycles", type=int, default=64)
    ap.add_argument("--host-matrix", action="store_true",
                    help="host-resident decline matrix: n_kv 32k/64k/128k x depth 0/1/4 x budget 128/512 MiB")
    ap.add_argument("--churn-n", type=int, default=131072)
    ap.add_argument("--rows", default="", help="comma-separated subset of the extra rows to run (default: all)")
    ap.add_argument("--child", default="", help=argparse.SUPPRESS)  # one optional phase, in a process of its own
    return ap.parse_args()


# ----------------------------------------------------------------- shapes --
H, HK, D = 40, 8, 128


def kv_bytes_per_row(type_: str) -> int:
    if type_ == "q8_0":
        return 2 * HK * (D + (D // 32) * 2)  # 2176
    if type_ == "q8_0/q4_0":  # q8_0 K, q4_0 V
        return HK * (D + (D // 32) * 2) + HK * (D // 2 + (D // 32) * 2)  # 1088 + 576 = 1664
    return 2 * HK * D * 2  # 4096


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks --
class Clocks:
    """nvidia-smi samples every 50 ms from start() to stop(); the report keeps
    the samples that fall inside the timed windows marked with window()."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.windows = []
        self.path = os.path.join("/tmp", "kvc_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t_end = time.time() + 10.0  # the first sample shows the sampler is running
        while time.time() < t_end and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def window(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return clock_summary(lines, self.windows)


def clock_summary(lines, windows) -> dict:
    """Median SM clock and throttle reasons of the nvidia-smi samples (CSV lines
    of Clocks.FIELDS) that fall inside the timed windows [(t0, t1)] (epoch
    seconds, 25 ms of slack); with none inside, the sample nearest to them."""
    import datetime

    rows = []
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append((ts, float(parts[2]), float(parts[3]),
                         [n for n, v in zip(names, parts[6:10]) if v.lower() in ("active", "1")]))
        except ValueError:
            continue
    inside = [r for r in rows if any(t0 - 0.025 <= r[0] <= t1 + 0.025 for t0, t1 in windows)]
    note = "samples inside the timed windows"
    if not inside and rows and windows:
        mid = sum(t0 + t1 for t0, t1 in windows) / (2 * len(windows))
        inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        note = "no sample fell inside the timed windows: the nearest one"
    reasons = sorted({n for r in inside for n in r[3]})
    return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
            "sm_max_mhz": inside[-1][2] if inside else None, "reasons": reasons, "samples": len(inside),
            "timed_ms": round(1e3 * sum(t1 - t0 for t0, t1 in windows), 1), "note": note}


def attn_traffic(type_: str, n_kv: int):
    """DRAM read + write bytes of one attention launch, from the committed ncu
    summary of the q8_0 n_kv 16384 launch; None for other workloads or once
    the kernel source no longer matches the hash the summary was taken on."""
    import hashlib
    import re

    if type_ != "q8_0" or n_kv != 16384:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", "attn_kernel_q8_0_16k.md")).read()
        src = open(os.path.join(ROOT, "kv_cache_decode_flash_gb300", "csrc", "k_attn.cu"), "rb").read()
    except OSError:
        return None
    h = re.search(r"kernel_sha256: ([0-9a-f]+)", text)
    t = re.search(r"`traffic_bytes_per_launch`[^|]*\|\s*(\d+)", text)
    if not h or not t or not hashlib.sha256(src).hexdigest().startswith(h.group(1)):
        return None
    return int(t.group(1))


L_STACK = 64  # layers of the decode stack the host-resident rows run

# ------------------------------------------------------------- CPU oracle --
def oracle_sample(n_kv: int, n_layers: int, type_: str, seed: int = 0):
    """Quantised sample layers for the oracle (not timed)."""
    import oracle
    from kv_cache_decode_flash_gb300 import synth

    layers = []
    for l in range(n_layers):
        k = synth.normal(seed, synth.stream_id("k", l), n_kv * HK * D, 0.5).reshape(n_kv, HK, D)
        v = synth.normal(seed, synth.stream_id("v", l), n_kv * HK * D, 0.5).reshape(n_kv, HK, D)
        q = synth.normal(seed, synth.stream_id("q", l), H * D).reshape(H, D)
        if type_ == "q8_0":
            kc, ks = oracle.q8_0_quantize(k)
            vc, vs = oracle.q8_0_quantize(v)
            layers.append((q, oracle.Q8_0, kc, ks, vc, vs))
        else:
            layers.append((q, oracle.F16, oracle.f32_to_f16(k), None, oracle.f32_to_f16(v), None))
    return layers


def time_oracle(layers, n_kv: int, type_: str):
    """Oracle decode attention over the sample layers, one task per (layer,
    query head) on all host cores.  Returns (GB/s, seconds, threads)."""
    import oracle

    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    scale = float(np.float32(1.0 / np.sqrt(D)))

    def task(args):
        (q, t, kc, ks, vc, vs), h = args
        return oracle.attn(q, t, kc, ks, t, vc, vs, scale, heads=(h, h + 1))

    jobs = [(lay, h) for lay in layers for h in range(H)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(task, jobs))
    dt = time.perf_counter() - t0
    nbytes = len(layers) * n_kv * kv_bytes_per_row(type_)
    return nbytes / dt / GB, dt, threads


def oracle_rows(args) -> dict:
    """The oracle timed beside the other rows, each on a bounded sample (a few
    seconds of host time in all), on every host core where the work splits:
    host-resident attention over one layer's pinned-store-sized arrays at 32k
    (the CPU attending where the data lives), a ragged-batch sample, one
    layer's RoPE shift of an 8192-row block (the churn's shift), and KeyDiff
    scores of one 32768-row layer."""
    import oracle
    from kv_cache_decode_flash_gb300 import synth

    res = {}
    # host-resident 32k: one layer, all query heads; steps/s for the 64-layer stack
    lay = oracle_sample(32768, 1, "q8_0", seed=3)
    gbs, dt, threads = time_oracle(lay, 32768, "q8_0")
    res["host_32k_attention"] = {"gbs": round(gbs, 3), "steps_per_s": round(gbs * GB / (L_STACK * 32768 *
                                kv_bytes_per_row("q8_0")), 4), "cores": threads,
                                 "sample": "1 of 64 layers at 32768 rows, 40 query heads (%.1f s)" % dt}
    # ragged batch: the four shortest of the benchmark's 32 lengths, 32 query heads
    lens = sorted(synth.randint(0, synth.stream_id("len"), 32, 1024, 32768).tolist())[:4]
    seqs = []
    for i, n in enumerate(lens):
        k = synth.normal(4, synth.stream_id("k", 0, i), n * HK * D).reshape(n, HK, D)
        v = synth.normal(4, synth.stream_id("v", 0, i), n * HK * D).reshape(n, HK, D)
        q = synth.normal(4, synth.stream_id("q", 0, i), 32 * D).reshape(32, D)
        seqs.append((q, *oracle.q8_0_quantize(k), *oracle.q8_0_quantize(v), n))
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda a: oracle.attn(a[0][0], oracle.Q8_0, a[0][1], a[0][2], oracle.Q8_0, a[0][3], a[0][4],
                                          0.088, heads=(a[1], a[1] + 1)), [(sq, h) for sq in seqs for h in range(32)]))
    dt = time.perf_counter() - t0
    rows = sum(lens)
    res["ragged_q8_0"] = {"gbs": round(rows * kv_bytes_per_row("q8_0") / dt / GB, 3), "cores": threads,
                          "sample": "the 4 shortest of the 32 sequences (%d rows), 32 query heads (%.1f s)"
                                    % (rows, dt)}
    # churn shift: one layer's K of an 8192-row block, RoPE shift with requantisation (one thread)
    kc, ks = lay[0][2][:8192], lay[0][3][:8192]
    t0 = time.perf_counter()
    oracle.rope_shift_q8_0(kc, ks, 0, 1e6, 131072 - 8192)
    dt = time.perf_counter() - t0
    res["churn_shift"] = {"gbs": round(2 * 8192 * HK * (D + (D // 32) * 2) / dt / GB, 3), "cores": 1,
                          "sample": "one layer of an 8192-row block, K read + write (%.2f s)" % dt}
    # KeyDiff: one 32768-row layer, two passes over its K (one thread)
    t0 = time.perf_counter()
    oracle.keydiff_scores(oracle.Q8_0, lay[0][2], lay[0][3])
    dt = time.perf_counter() - t0
    res["keydiff_scores"] = {"gbs": round(2 * 32768 * HK * (D + (D // 32) * 2) / dt / GB, 3), "cores": 1,
                             "sample": "one 32768-row layer, two passes over its K (%.2f s)" % dt}
    return res


# ------------------------------------------------------------ reference --
def run_reference(args, rank: int):
    if rank != 0:
        return
    n_layers = 1
    layers = oracle_sample(args.n_kv, n_layers, args.type)
    for _ in range(max(args.warmup, 0)):
        time_oracle(layers, args.n_kv, args.type)
    times, threads = [], 1
    for _ in range(args.steps):
        gbs, dt, threads = time_oracle(layers, args.n_kv, args.type)
        times.append(dt)
    total = sum(times)
    nbytes = n_layers * args.n_kv * kv_bytes_per_row(args.type) * args.steps
    value = nbytes / total / GB
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "1 of %d layers per step, all %d query heads, n_kv=%d" % (args.layers, H,
                                                                                                args.n_kv)},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(args):
    return {"workload": "decode, %d layers, %d/%d heads, head_dim %d, %s KV, n_kv %d, batch 1"
                        % (args.layers, H, HK, D, args.type, args.n_kv),
            "layers": args.layers, "n_head": H, "n_head_kv": HK, "head_dim": D, "kv_type": args.type,
            "n_kv": args.n_kv, "batch": 1, "rope_base": 1e6,
            "l2": "no flush: each step reads %.2f GB of distinct KV, far above the 129 MB L2"
                  % (args.layers * args.n_kv * kv_bytes_per_row(args.type) / GB),
            "parallelism": "replicas"}


# --------------------------------------------------------------- our arm --
def fill_cache(cache, args, dev, torch):
    from kv_cache_decode_flash_gb300 import synth

    n0 = args.n_kv - 1
    chunk = 4096
    for l in range(args.layers):
        for p0 in range(0, n0, chunk):
            m = min(chunk, n0 - p0)
            k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
            v = synth.normal_torch(0, synth.stream_id("v", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
            cache.append(l, 0, p0, k, v)
    torch.cuda.synchronize()


def measure_link(torch, dev) -> float:
    """Pinned host -> device copy bandwidth at a slot-sized transfer (GB/s)."""
    n = 256 << 20
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return 5 * n / (e0.elapsed_time(e1) * 1e-3) / GB


HOST_CELLS = (("ordered", 0, 128 << 20), ("pipelined", 1, 512 << 20), ("pipelined_depth4", 4, 1 << 30),
              ("declined", 1, 128 << 20))
MATRIX_CELLS = (("N0", 0, 128 << 20), ("N1_128MiB", 1, 128 << 20), ("N1_512MiB", 1, 512 << 20),
                ("N4_128MiB", 4, 128 << 20), ("N4_512MiB", 4, 512 << 20))


SPLIT_CELLS = (("ordered", 0, 128 << 20), ("pipelined", 1, 512 << 20))


def host_pipeline(args, dev, torch, kvc, n=None, cells=HOST_CELLS, link=None, gpu_heads=0):
    """Host-resident KV at n (default args.host_n): steps/s and H2D GB/s for
    each (name, depth, budget) cell, run one after another on one cache (the
    context grows by host_steps + 1 rows per cell).  With gpu_heads > 0 the
    context splits by head: KV heads 0..gpu_heads-1 stay in HBM and only the
    others cross the link.  Ordered/pipelined byte identity is a parity test,
    not measured here."""
    from kv_cache_decode_flash_gb300 import synth

    n = n or args.host_n
    L = args.layers
    t = kvc.KVC_Q8_0 if args.type == "q8_0" else kvc.KVC_F16
    res = {}
    link = link or measure_link(torch, dev)
    scale = float(1.0 / np.sqrt(D))
    if gpu_heads:
        cache = kvc.KVCache(L, H, HK, D, n + 256, 1, t, t, 1e6, 0, kvc.KVC_SPLIT_HEADS, 0, 0, gpu_heads)
    else:
        cache = kvc.KVCache(L, H, HK, D, n + 256, 1, t, t, 1e6, 0, kvc.KVC_HOST_PINNED)
    host_frac = (HK - gpu_heads) / HK  # share of each row that lives in host memory
    try:
        for l in range(L):
            for p0 in range(0, n - 1, 8192):
                m = min(8192, n - 1 - p0)
                k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                v = synth.normal_torch(0, synth.stream_id("v", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                cache.append(l, 0, p0, k, v)
        q = torch.randn(L, 1, H, D, device=dev)
        kn = torch.randn(L, 1, HK, D, device=dev) * 0.5
        vn = torch.randn(L, 1, HK, D, device=dev) * 0.5
        out = torch.empty_like(q)
        pos = n - 1
        for name, depth, budget in cells:
            kvc.kvc_pipeline_depth(cache.ctx, depth)
            kvc.kvc_pipeline_budget(cache.ctx, budget)
            # five timed runs of host_steps steps after one warm-up step; the host link is
            # shared with other work on the machine, so single runs vary: the best run is
            # the transport's rate, the median is reported beside it
            link_cell = measure_link(torch, dev)
            runs = []
            for rep in range(5):
                for step in range(args.host_steps + (1 if rep == 0 else 0)):
                    if step == (1 if rep == 0 else 0):
                        torch.cuda.synchronize()
                        t0 = time.perf_counter()
                    for l in range(L):
                        cache.append(l, 0, pos, kn[l], vn[l])
                        cache.attn_decode(l, [0], q[l], out[l], scale)
                    pos += 1
                torch.cuda.synchronize()
                runs.append((time.perf_counter() - t0) / args.host_steps)
            dt, dt_med = min(runs), statistics.median(runs)
            link_cell = max(link_cell, measure_link(torch, dev))
            st = cache.stats()
            # bytes moved host->device per step: every layer's rows (stable prefix) once
            h2d = L * (pos - 1) * kv_bytes_per_row(args.type) * host_frac
            res[name] = {"steps_per_s": round(1.0 / dt, 3), "ms_per_step": round(1000 * dt, 3),
                         "steps_per_s_median": round(1.0 / dt_med, 3),
                         "h2d_gbs": round(h2d / dt / GB, 2), "frac_of_link": round(h2d / dt / GB / link, 3),
                         "link_gbs_around": round(link_cell, 2),
                         "frac_of_link_around": round(h2d / dt / GB / link_cell, 3),
                         "ring_engaged": st["ring_engaged"], "ring_declined": st["ring_declined"],
                         "rolling": st["rolling"], "tile_rows": st["tile_rows"],
                         "ring_mib": round(st["ring_bytes"] / 2**20, 1),
                         "device_mib": round(st["device_bytes"] / 2**20, 1),
                         "host_mib": round(st["host_pinned_bytes"] / 2**20, 1)}
        res["n_kv"] = n
        if gpu_heads:
            res["gpu_heads"] = gpu_heads
            res["bytes"] = "H2D counts the host heads' rows only (%d of %d KV heads)" % (HK - gpu_heads, HK)
        res["link_gbs"] = round(link, 2)
        res["link"] = "pinned H2D, 256 MiB copies, measured in this run"
        res["note"] = ("n_kv grows by one row per step (decode); H2D counts every layer's rows once per step; "
                       "steps/s is the best of 5 runs of host_steps steps (median beside it); link_gbs_around = the best of "
                       "two link measurements "
                       "taken just before and after the cell (the host link is shared)")
    finally:
        cache.close()
    return res


TIMELINE_CELLS = ((32768, (("ordered", 0, 128 << 20), ("N1_512MiB", 1, 512 << 20), ("N4_512MiB", 4, 512 << 20))),
                  (65536, (("ordered", 0, 128 << 20), ("N1_512MiB", 1, 512 << 20))),
                  (131072, (("ordered", 0, 128 << 20), ("rolling_N4_128MiB", 4, 128 << 20))))


def _measure(iv, lo, hi):
    """Length of the union of intervals [a, b) clipped to [lo, hi)."""
    tot, end = 0.0, lo
    for a, b in sorted(iv):
        a, b = max(a, end), min(b, hi)
        if b > a:
            tot += b - a
            end = b
    return tot


def _intersect(iv1, iv2):
    out = []
    for a1, b1 in iv1:
        for a2, b2 in iv2:
            a, b = max(a1, a2), min(b1, b2)
            if b > a:
                out.append((a, b))
    return out


def timeline_summary(recs, L):
    """Summary of the middle one of three traced steps: recs are
    (kind, layer, bytes, t0_us, t1_us), kind 0 delivery, 1 attention."""
    att = [r for r in recs if r[0] == 1]
    dlv = [r for r in recs if r[0] == 0]
    per = len(att) // 3  # attention launches per step (several per layer with rolling tiles)
    if per < L or len(att) != 3 * per:
        return {"error": "%d attention records for 3 steps of %d layers" % (len(att), L)}
    w0 = att[per - 1][4]  # end of the first step's last attention
    w1 = att[2 * per - 1][4]
    win = w1 - w0
    D_iv = [(r[3], r[4]) for r in dlv]
    A_iv = [(r[3], r[4]) for r in att]
    copy = _measure(D_iv, w0, w1)
    busy = _measure(A_iv, w0, w1)
    hidden = _measure(_intersect([(max(a, w0), min(b, w1)) for a, b in D_iv if b > w0 and a < w1], A_iv), w0, w1)
    inwin = [r for r in dlv if w0 <= r[3] < w1]
    rates = sorted(r[2] / (r[4] - r[3]) / 1e3 for r in inwin if r[4] > r[3])  # GB/s (bytes / us / 1e3)
    moved = sum(r[2] for r in inwin)
    pct = lambda q: round(rates[min(len(rates) - 1, int(q * len(rates)))], 1) if rates else None
    return {"step_ms": round(win / 1e3, 3), "steps_per_s": round(1e6 / win, 2),
            "deliveries": len(inwin), "delivered_gb": round(moved / 1e9, 3),
            "h2d_gbs_over_step": round(moved / win / 1e3, 1),
            "per_delivery_gbs_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
            "copy_busy_frac": round(copy / win, 3), "attn_busy_frac": round(busy / win, 3),
            "copy_hidden_frac": round(hidden / copy, 3) if copy > 0 else None,
            "attn_hidden_frac": round(hidden / busy, 3) if busy > 0 else None,
            "launches_per_step": per,
            "compute_idle_ms": round((win - busy) / 1e3, 3)}


def link_series(torch, dev, n: int = 60, size: int = 64 << 20) -> list:
    """min, p10 and p50 GB/s of n back-to-back pinned host -> device copies of
    `size` bytes, each timed by its own CUDA events (the link on its own)."""
    h = torch.empty(size, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(size, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    d.copy_(h, non_blocking=True)
    ev[0].record()
    for i in range(n):
        d.copy_(h, non_blocking=True)
        ev[i + 1].record()
    torch.cuda.synchronize()
    r = sorted(size / (ev[i].elapsed_time(ev[i + 1]) * 1e-3) / GB for i in range(n))
    return [round(r[0], 1), round(r[n // 10], 1), round(r[n // 2], 1)]


def host_timeline(args, dev, torch, kvc) -> dict:
    """Per-delivery timeline of the host transport (kvc_trace_*): for each
    context length and (depth, budget) cell, one warm-up step, then three
    traced steps; the middle one is summarised (timeline_summary)."""
    from kv_cache_decode_flash_gb300 import synth

    L = args.layers
    out = {"link_gbs": round(measure_link(torch, dev), 2)}
    scale = float(1.0 / np.sqrt(D))
    for n, cells in TIMELINE_CELLS:
        cache = kvc.KVCache(L, H, HK, D, n + 256, 1, kvc.KVC_Q8_0, kvc.KVC_Q8_0, 1e6, 0, kvc.KVC_HOST_PINNED)
        try:
            for l in range(L):
                for p0 in range(0, n - 1, 8192):
                    m = min(8192, n - 1 - p0)
                    k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                    cache.append(l, 0, p0, k, k)
            q = torch.randn(L, 1, H, D, device=dev)
            kn = torch.randn(L, 1, HK, D, device=dev) * 0.5
            o = torch.empty_like(q)
            pos = n - 1

            def step():
                nonlocal pos
                for l in range(L):
                    cache.append(l, 0, pos, kn[l], kn[l])
                    cache.attn_decode(l, [0], q[l], o[l], scale)
                pos += 1

            for name, depth, budget in cells:
                kvc.kvc_pipeline_depth(cache.ctx, depth)
                kvc.kvc_pipeline_budget(cache.ctx, budget)
                step()
                torch.cuda.synchronize()
                probe_before = link_series(torch, dev)
                kvc.kvc_trace_start(cache.ctx, 64 * L)
                for _ in range(3):
                    step()
                torch.cuda.synchronize()
                kvc.kvc_trace_stop(cache.ctx)
                st = cache.stats()
                summ = timeline_summary(kvc.kvc_trace_read(cache.ctx), L)
                summ.update({"ring_engaged": st["ring_engaged"], "rolling": st["rolling"],
                             "tile_rows": st["tile_rows"],
                             "plain_copies_gbs_min_p10_p50": [probe_before[0], probe_before[1], probe_before[2],
                                                              "before"] + link_series(torch, dev) + ["after"]})
                if "h2d_gbs_over_step" in summ:
                    summ["frac_of_link"] = round(summ["h2d_gbs_over_step"] / out["link_gbs"], 3)
                out["%dk_%s" % (n // 1024, name)] = summ
        finally:
            cache.close()
        torch.cuda.empty_cache()
    out["note"] = ("CUDA-event trace of the middle of three decode steps: deliveries are the H2D copies of "
                   "one layer (or rolling tile), attention the launches on the compute stream after their "
                   "wait; copy_hidden_frac = share of copy time overlapped by attention, attn_hidden_frac = share "
                   "of attention time overlapped by copies; plain_copies: 60 back-to-back 64 MiB pinned H2D "
                   "copies just before and after the cell, each timed alone")
    return out


# ------------------------------------------------------- further rows --
def attn_only_gbs(kvc, torch, dev, type_: str, n: int, reps: int = 50):
    """KV GB/s of back-to-back attention launches, one per layer, over enough
    distinct layers that one pass reads at least 512 MB (no L2 reuse)."""
    from kv_cache_decode_flash_gb300 import synth

    layers = max(8, -(-(512 << 20) // (n * kv_bytes_per_row(type_))))

    t = kvc.KVC_F16 if type_ == "f16" else kvc.KVC_Q8_0
    tv = kvc.KVC_Q4_0 if type_ == "q8_0/q4_0" else t
    cache = kvc.KVCache(layers, H, HK, D, n + 64, 1, t, tv, 1e6)
    try:
        for l in range(layers):
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                cache.append(l, 0, p0, k, k)
        q = torch.randn(layers, 1, H, D, device=dev)
        o = torch.empty_like(q)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            for l in range(layers):
                cache.attn_decode(l, [0], q[l], o[l], 0.088, stream=s)
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for l in range(layers):
                cache.attn_decode(l, [0], q[l], o[l], 0.088, stream=torch.cuda.current_stream())
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) * 1e-3 / (reps * layers)
        return {"n_kv": n, "kv_type": type_, "layers": layers, "launch_us": round(dt * 1e6, 3),
                "gbs": round(n * kv_bytes_per_row(type_) / dt / GB, 1)}
    finally:
        cache.close()


def ragged(kvc, torch, dev, type_: str, reps: int = 60):
    """32 sequences, lengths uniform in [1024, 32768] (seed 0), 32/8 heads,
    D 128, one layer; one attention call over the whole batch."""
    from kv_cache_decode_flash_gb300 import synth

    Hq = 32
    lens = synth.randint(0, synth.stream_id("len"), 32, 1024, 32768).tolist()
    t = kvc.KVC_Q8_0 if type_ == "q8_0" else kvc.KVC_F16
    cache = kvc.KVCache(1, Hq, HK, D, sum(lens) + 32 * 256, 32, t, t, 1e6)
    try:
        for sidx, n in enumerate(lens):
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = synth.normal_torch(0, synth.stream_id("k", 0, sidx * 4096 + p0 // 8192), m * HK * D, 1.0, dev).view(m, HK, D)
                v = synth.normal_torch(0, synth.stream_id("v", 0, sidx * 4096 + p0 // 8192), m * HK * D, 1.0, dev).view(m, HK, D)
                cache.append(0, sidx, p0, k, v)
        q = torch.randn(32, Hq, D, device=dev)
        o = torch.empty_like(q)
        ids = list(range(32))
        for _ in range(10):
            cache.attn_decode(0, ids, q, o, 0.088)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            cache.attn_decode(0, ids, q, o, 0.088)
        e1.record()
        torch.cuda.synchronize()
        dt = e0.elapsed_time(e1) * 1e-3 / reps
        rows = sum(lens)
        return {"kv_type": type_, "sequences": 32, "rows": rows, "ms_per_call": round(dt * 1e3, 4),
                "gbs": round(rows * kv_bytes_per_row(type_) / dt / GB, 1)}
    finally:
        cache.close()


def churn(kvc, torch, dev, n: int, cycles: int, layers: int):
    """Cold-store churn on a q8_0 cache of n tokens: evict the oldest 8192
    rows (copy to a scratch sequence, export, drop, remove, slide) and
    re-admit them at the tail (import, shift, copy in), then one decode step
    over the layer stack.  Per-op GB/s; every op is synchronous."""
    from kv_cache_decode_flash_gb300 import synth

    blk = 8192
    row_all = layers * kv_bytes_per_row("q8_0")          # one row, all layers, K+V
    krow_all = layers * HK * (D + (D // 32) * 2)         # K only (what a shift rewrites)
    cache = kvc.KVCache(layers, H, HK, D, n + 2 * blk + 512, 2, kvc.KVC_Q8_0, kvc.KVC_Q8_0, 1e6)
    try:
        for l in range(layers):
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                v = synth.normal_torch(0, synth.stream_id("v", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                cache.append(l, 0, p0, k, v)
        torch.cuda.synchronize()
        size = kvc.kvc_state_size(cache.ctx, 0, 0, blk)
        host = torch.empty(size, dtype=torch.uint8, pin_memory=True)
        again = torch.empty(size, dtype=torch.uint8, pin_memory=True)
        q = torch.randn(layers, 1, H, D, device=dev)
        o = torch.empty_like(q)
        # the host link in each direction for a copy of the state's size between
        # the same pinned buffers and device memory (best of 3)
        devbuf = torch.empty(size, dtype=torch.uint8, device=dev)
        link = {}
        for name, dst, src in (("d2h", again, devbuf), ("h2d", devbuf, host)):
            best = None
            for _ in range(3):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                dst.copy_(src)
                torch.cuda.synchronize()
                dt_ = time.perf_counter() - t0
                best = dt_ if best is None else min(best, dt_)
            link[name] = size / best / GB
        del devbuf
        acc = {k: 0.0 for k in ("seq_cp", "state_get", "seq_rm", "slide", "state_set", "shift", "copy_in", "decode")}

        def timed(name, fn):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            acc[name] += time.perf_counter() - t0

        ok = exact = True
        for c in range(cycles):
            timed("seq_cp", lambda: cache.seq_cp(0, 1, 0, blk))
            timed("state_get", lambda: cache.state_get(1, -1, -1, host))
            cache.seq_rm(1, -1, -1)
            timed("seq_rm", lambda: cache.seq_rm(0, 0, blk))
            timed("slide", lambda: cache.seq_add(0, blk, n, -blk))
            timed("state_set", lambda: cache.state_set(1, host))
            if c in (0, cycles - 1):  # export -> import -> export is byte-exact
                cache.state_get(1, -1, -1, again)
                exact = exact and bool(torch.equal(host, again))
            timed("shift", lambda: cache.seq_add(1, -1, -1, n - blk))
            timed("copy_in", lambda: cache.seq_cp(1, 0, -1, -1))
            cache.seq_rm(1, -1, -1)
            timed("decode", lambda: [cache.attn_decode(l, [0], q[l], o[l], 0.088) for l in range(layers)])
            pos = cache.positions(0)
            ok = ok and bool((np.sort(pos) == np.arange(n)).all())
        byts = {"seq_cp": 2 * blk * row_all, "state_get": size, "seq_rm": 0, "slide": 2 * (n - blk) * krow_all,
                "state_set": size, "shift": 2 * blk * krow_all, "copy_in": 2 * blk * row_all,
                "decode": n * row_all}
        ops = {}
        for k2, v2 in acc.items():
            per = v2 / cycles
            ops[k2] = {"ms": round(per * 1e3, 3), "gbs": round(byts[k2] / per / GB, 1) if byts[k2] else None}
        ops["state_get"]["frac_of_link"] = round(ops["state_get"]["gbs"] / link["d2h"], 3)
        ops["state_set"]["frac_of_link"] = round(ops["state_set"]["gbs"] / link["h2d"], 3)
        return {"n_kv": n, "block": blk, "cycles": cycles, "layers": layers, "positions_ok": ok,
                "state_round_trip_exact": exact,
                "link_gbs": {"d2h": round(link["d2h"], 1), "h2d": round(link["h2d"], 1),
                             "note": "one plain copy of the state's size between the same pinned buffers "
                                     "and device memory, best of 3"},
                "bytes": "seq_cp/copy_in/slide/shift: read+write; state_get/set: bytes exported; decode: KV read",
                "ops": ops}
    finally:
        cache.close()


def keydiff(kvc, torch, dev, n: int, layers: int, reps: int = 10):
    """KeyDiff scores of one layer of an n-token q8_0 cache (two passes over
    that layer's K) and one retention-aware context shift (scores, window,
    seq_rm, slide of the later rows in every layer).  Synchronous API calls."""
    from kv_cache_decode_flash_gb300 import synth

    cache = kvc.KVCache(layers, H, HK, D, n + 512, 1, kvc.KVC_Q8_0, kvc.KVC_Q8_0, 1e6)
    try:
        for l in range(layers):
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                cache.append(l, 0, p0, k, k)
        torch.cuda.synchronize()
        cache.key_scores(0, -1)
        t0 = time.perf_counter()
        for _ in range(reps):
            sc = cache.key_scores(0, -1)
        dt = (time.perf_counter() - t0) / reps
        kbytes = n * HK * (D + (D // 32) * 2)  # one layer's K codes + scales
        t0 = time.perf_counter()
        p0 = cache.evict_window(0, -1, 4, 8192, 1024)
        dt_evict = time.perf_counter() - t0
        return {"n_kv": n, "layers": layers, "score_ms": round(dt * 1e3, 3),
                "score_gbs": round(2 * kbytes / dt / GB, 1), "bytes": "2 passes over one layer's K",
                "evict_ms": round(dt_evict * 1e3, 3), "evicted_from": p0, "rows_after": cache.n_tokens(0),
                "score_range": [round(float(sc.min()), 4), round(float(sc.max()), 4)]}
    finally:
        cache.close()


def cold_store(kvc, torch, dev, n: int, layers: int, cycles: int = 8):
    """Host-RAM cold store over an n-token q8_0 cache: each cycle evicts the
    oldest 8192 rows into the store (copy to a scratch sequence, export into
    pinned host memory, remove, slide) and admits them back at the tail
    (import, shift, copy in), then admits an absent key (a miss).
    Synchronous calls, wall time per operation; the first cycle, which pins
    the store's buffers, is not timed."""
    from kv_cache_decode_flash_gb300 import synth

    blk = 8192
    cache = kvc.KVCache(layers, H, HK, D, n + 2 * blk + 512, 2, kvc.KVC_Q8_0, kvc.KVC_Q8_0, 1e6)
    store = kvc.ColdStore(2 * blk)
    try:
        for l in range(layers):
            for p0 in range(0, n, 8192):
                m = min(8192, n - p0)
                k = synth.normal_torch(0, synth.stream_id("k", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                v = synth.normal_torch(0, synth.stream_id("v", l, p0), m * HK * D, 0.5, dev).view(m, HK, D)
                cache.append(l, 0, p0, k, v)
        torch.cuda.synchronize()
        size = kvc.kvc_state_size(cache.ctx, 0, 0, blk)
        t_ev = t_ad = t_miss = 0.0
        ok = True
        for c in range(cycles + 1):
            t0 = time.perf_counter()
            stored, _ = store.evict(cache, 0, 1, 0, blk, 1000 + c, c % 3)
            t1 = time.perf_counter()
            hit, _ = store.admit(cache, 0, 1, 1000 + c)
            t2 = time.perf_counter()
            miss, _ = store.admit(cache, 0, 1, 1)
            t3 = time.perf_counter()
            ok = ok and stored == 1 and hit == 1 and miss == 0
            if c:
                t_ev += t1 - t0
                t_ad += t2 - t1
                t_miss += t3 - t2
        ok = ok and bool((np.sort(cache.positions(0)) == np.arange(n)).all())
        # restore versus recompute: admits of smaller blocks as well, so that the store's fitted
        # model, restore_us = fixed + per_token * n, separates the fixed cost from the per-row one
        for j, m in enumerate((512, 2048, 4096, 512, 2048, 4096)):
            store.evict(cache, 0, 1, 0, m, 5000 + j, 0)
            store.admit(cache, 0, 1, 5000 + j)
        fixed_us, per_tok_us, samples = store.restore_model()
        crossover = {}
        for rec in (1.0, 10.0, 100.0):  # recompute cost per token (us) a caller might measure
            crossover[str(rec)] = (round(fixed_us / (rec - per_tok_us)) if rec > per_tok_us else None)
        return {"n_kv": n, "block": blk, "layers": layers, "cycles": cycles, "block_state_bytes": size,
                "restore_model": {"fixed_us": round(fixed_us, 1), "per_token_us": round(per_tok_us, 4),
                                  "samples": samples,
                                  "crossover_tokens_by_recompute_us_per_token": crossover,
                                  "note": "least-squares fit over the store's timed admits (8192-row blocks and "
                                          "512 / 2048 / 4096-row ones); restore wins above the crossover"},
                "evict_ms": round(t_ev / cycles * 1e3, 3), "admit_ms": round(t_ad / cycles * 1e3, 3),
                "miss_us": round(t_miss / cycles * 1e6, 1),
                "evict_state_gbs": round(size / (t_ev / cycles) / GB, 1),
                "admit_state_gbs": round(size / (t_ad / cycles) / GB, 1), "ok": ok, "store": store.stats(),
                "note": "evict = seq_cp + export (D2H) + remove + slide of the rest; admit = import (H2D) + "
                        "shift + copy in; GB/s = state bytes of the block / operation time"}
    finally:
        store.close()
        cache.close()


def step_line(args, world: int, L: int, n: int, t_step: float, t_attn: float, t_e2e: float, t_two: float,
              h2d_bytes: int, d2h_bytes: int, clk: dict) -> dict:
    """The JSON line of the decode step from its measured durations (seconds for
    args.steps steps; t_attn: the attention-only graph)."""
    row_bytes = kv_bytes_per_row(args.type)
    step_bytes = L * n * row_bytes
    value = world * step_bytes * args.steps / t_step / GB
    attn_launch_s = t_attn / (args.steps * L)
    achieved = n * row_bytes / attn_launch_s / GB
    peak, peak_kind = peaks()
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * t_step / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "%s KV, fp32 accumulate" % args.type,
        "data": "synthetic (splitmix64 + Box-Muller, N(0,1)*0.5 K/V)", "config": config_dict(args),
        "steps_per_s": round(args.steps / t_step, 2),
        "hbm_frac": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": attn_traffic(args.type, n),
                     "kernel": "attn_kernel (decode attention), %d bytes per launch" % (n * row_bytes),
                     "peak_kind": "%s (MEASURED_PEAKS.json hbm_gbs, burst copy)" % peak_kind,
                     "launch_us": round(attn_launch_s * 1e6, 3),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                                       "profiles/attn_kernel_q8_0_16k.md (null when the kernel changed)"},
        "e2e": {"value": round(world * step_bytes * args.steps / t_e2e / GB, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes},
        "gpu_launches": L * args.steps,
        "step_two_calls": {"ms_per_step": round(1000 * t_two / args.steps, 4),
                           "value": round(world * step_bytes * args.steps / t_two / GB, 2), "unit": "GB/s",
                           "note": "the same step with a separate append kernel before each attention launch"},
        "clocks": clk,
    }


EXTRA_ROWS = ("q8_0_4k", "q8_0_64k", "q8_0_256k", "f16_16k", "f16_4k", "q8_0_q4_0_16k", "q8_0_q4_0_64k",
              "ragged_q8_0", "ragged_f16", "churn", "keydiff", "split_32k_g4", "cold_store", "host_timeline")


def run_child(args, name: str) -> dict:
    """Run one optional phase in a child process and return its JSON result
    (or the error it ended with)."""
    t0 = time.perf_counter()
    log("phase %s" % name)
    cmd = [sys.executable, os.path.abspath(__file__), "--child", name] + [a for a in sys.argv[1:]]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)  # each phase takes about a minute
    except subprocess.TimeoutExpired:
        return {"error": "phase %s: no result within 600 s" % name}
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if r.returncode != 0 or not lines:
        tail = " | ".join((r.stderr or "").strip().splitlines()[-4:])
        log("phase %s failed (exit %d)" % (name, r.returncode))
        return {"error": ("exit %d: %s" % (r.returncode, tail))[:400]}
    log("phase %s done in %.1f s" % (name, time.perf_counter() - t0))
    return json.loads(lines[-1])


def child_phase(args) -> dict:
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.child
    if name == "host":
        return host_pipeline(args, dev, torch, kvc)
    if name == "host_matrix":
        link = measure_link(torch, dev)
        mat = {}
        for hn in (32768, 65536, 131072):
            try:
                mat[str(hn)] = host_pipeline(args, dev, torch, kvc, hn, MATRIX_CELLS, link)
            except Exception as e:  # reported, not fatal
                mat[str(hn)] = {"error": str(e)[:300]}
            torch.cuda.empty_cache()
        return mat
    rows = {
        "q8_0_4k": lambda: attn_only_gbs(kvc, torch, dev, "q8_0", 4096),
        "q8_0_64k": lambda: attn_only_gbs(kvc, torch, dev, "q8_0", 65536),
        "q8_0_256k": lambda: attn_only_gbs(kvc, torch, dev, "q8_0", 262144),
        "f16_16k": lambda: attn_only_gbs(kvc, torch, dev, "f16", 16384),
        "f16_4k": lambda: attn_only_gbs(kvc, torch, dev, "f16", 4096),
        "q8_0_q4_0_16k": lambda: attn_only_gbs(kvc, torch, dev, "q8_0/q4_0", 16384),
        "q8_0_q4_0_64k": lambda: attn_only_gbs(kvc, torch, dev, "q8_0/q4_0", 65536),
        "ragged_q8_0": lambda: ragged(kvc, torch, dev, "q8_0"),
        "ragged_f16": lambda: ragged(kvc, torch, dev, "f16"),
        "churn": lambda: churn(kvc, torch, dev, args.churn_n, args.churn_cycles, args.layers),
        "keydiff": lambda: keydiff(kvc, torch, dev, args.churn_n, args.layers),
        "split_32k_g4": lambda: host_pipeline(args, dev, torch, kvc, 32768, SPLIT_CELLS, gpu_heads=4),
        "cold_store": lambda: cold_store(kvc, torch, dev, args.churn_n, args.layers),
        "host_timeline": lambda: host_timeline(args, dev, torch, kvc),
    }
    return rows[name]()


def log(msg: str):
    print("bench: %s" % msg, file=sys.stderr, flush=True)


def max_over_ranks(vals, device, world: int):
    """Element-wise maximum of the ranks' timed durations (every rank gets it)."""
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def run_ours(args, rank: int, world: int):
    import torch

    from kv_cache_decode_flash_gb300 import kvc

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t = kvc.KVC_Q8_0 if args.type == "q8_0" else kvc.KVC_F16
    L, n = args.layers, args.n_kv
    cache = kvc.KVCache(L, H, HK, D, n + 256, 1, t, t, 1e6, 0, kvc.KVC_DEVICE, local)
    fill_cache(cache, args, dev, torch)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    # the step's inputs live in one buffer (q | k | v of every layer), so that the end-to-end
    # step moves them host -> device in one copy; qbuf / kbuf / vbuf are views into it
    nq, nk = L * H * D, L * HK * D
    inbuf = torch.empty(nq + 2 * nk, device=dev)
    qbuf = inbuf[:nq].view(L, 1, H, D)
    kbuf = inbuf[nq:nq + nk].view(L, 1, HK, D)
    vbuf = inbuf[nq + nk:].view(L, 1, HK, D)
    qbuf.copy_(torch.randn(L, 1, H, D, device=dev, generator=g))
    kbuf.copy_(torch.randn(L, 1, HK, D, device=dev, generator=g) * 0.5)
    vbuf.copy_(torch.randn(L, 1, HK, D, device=dev, generator=g) * 0.5)
    obuf = torch.empty(L, 1, H, D, device=dev)
    scale = float(1.0 / np.sqrt(D))

    s = torch.cuda.Stream(device=dev)
    # one eager step creates row n-1 in every layer (allocations happen here, not in capture)
    with torch.cuda.stream(s):
        for l in range(L):
            cache.decode_step(l, [0], [n - 1], kbuf[l], vbuf[l], qbuf[l], obuf[l], scale, stream=s)
    s.synchronize()
    # the captured step rewrites row n-1: roll the host bookkeeping back by one row
    # (seq_rm of the last position keeps the device pages; the graph re-appends it)
    cache.seq_rm(0, n - 1, -1)

    # the step: one fused append + attention launch per layer
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=s):
        for l in range(L):
            cache.decode_step(l, [0], [n - 1], kbuf[l], vbuf[l], qbuf[l], obuf[l], scale,
                              stream=torch.cuda.current_stream())
    cache.seq_rm(0, n - 1, -1)
    # the same step as two calls per layer (append kernel, then attention), for comparison
    two_call_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(two_call_graph, stream=s):
        for l in range(L):
            cache.append(l, 0, n - 1, kbuf[l], vbuf[l], stream=torch.cuda.current_stream())
            cache.attn_decode(l, [0], qbuf[l], obuf[l], scale, stream=torch.cuda.current_stream())
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph, stream=s):
        for l in range(L):
            cache.attn_decode(l, [0], qbuf[l], obuf[l], scale, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    clocks = Clocks(local)

    def timed(fn, steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(steps):
                fn()
            e1.record(s)
        torch.cuda.synchronize()
        clocks.window(w0, time.time())
        barrier()
        return e0.elapsed_time(e1) * 1e-3

    for _ in range(max(3, args.warmup)):
        step_graph.replay()
    torch.cuda.synchronize()
    clocks.start()
    t_step = timed(step_graph.replay, args.steps)
    for _ in range(3):
        attn_graph.replay()
    t_attn = timed(attn_graph.replay, args.steps)
    for _ in range(3):
        two_call_graph.replay()
    t_two = timed(two_call_graph.replay, args.steps)

    # end to end through the public API: inputs from pinned host memory, outputs back
    hin = torch.empty_like(inbuf, device="cpu").pin_memory()
    ho = torch.empty_like(obuf, device="cpu").pin_memory()
    hin.copy_(inbuf)

    def e2e_step():
        inbuf.copy_(hin, non_blocking=True)  # q, k and v of every layer
        step_graph.replay()
        ho.copy_(obuf, non_blocking=True)

    for _ in range(3):
        with torch.cuda.stream(s):
            e2e_step()
    t_e2e = timed(e2e_step, args.steps)

    # End to end without a graph: every step issues the 64 kvc_decode_step calls from the
    # host through the C entry point (arguments built once, so the binding adds little),
    # with the same pinned copies.  The sequence grows by one row per step, as in decode.
    import ctypes as C

    f_step = kvc.load().kvc_decode_step
    ids = (C.c_int32 * 1)(0)
    pos = (C.c_int32 * 1)(n)
    largs = [(cache.ctx, l, 1, ids, pos, kbuf[l].data_ptr(), vbuf[l].data_ptr(), qbuf[l].data_ptr(),
              obuf[l].data_ptr(), scale, s.cuda_stream) for l in range(L)]
    eager_steps = min(args.steps, 100)
    host_issue = [0.0]

    issue_steps = 8  # host time is taken over the first steps only: later ones wait on a full launch queue
    n_issue = [0]

    def eager_step():
        inbuf.copy_(hin, non_blocking=True)
        h0 = time.perf_counter()
        for a_ in largs:
            rc_ = f_step(*a_)
            if rc_ != 0:
                raise RuntimeError("kvc_decode_step: %d" % rc_)
        if n_issue[0] < issue_steps:
            host_issue[0] += time.perf_counter() - h0
            n_issue[0] += 1
        pos[0] += 1
        ho.copy_(obuf, non_blocking=True)

    for _ in range(3):
        with torch.cuda.stream(s):
            eager_step()
    host_issue[0] = 0.0
    n_issue[0] = 0
    n_eager0 = pos[0]
    t_eager = timed(eager_step, eager_steps)
    clk = clocks.stop()  # over the timed windows of the step, attention-only, two-call and end-to-end legs
    eager_rows = (n_eager0 + pos[0] - 1) / 2.0  # mean rows attended per step

    t_step, t_attn, t_e2e, t_two, t_eager = max_over_ranks([t_step, t_attn, t_e2e, t_two, t_eager], dev, world)

    out = step_line(args, world, L, n, t_step, t_attn, t_e2e, t_two, int(hin.numel() * 4), int(ho.numel() * 4),
                    clk)
    out["e2e_eager"] = {
        "value": round(world * L * eager_rows * kv_bytes_per_row(args.type) * eager_steps / t_eager / GB, 2),
        "unit": "GB/s", "ms_per_step": round(1000 * t_eager / eager_steps, 4), "steps": eager_steps,
        "host_us_per_call": round(1e6 * host_issue[0] / (max(1, n_issue[0]) * L), 2),
        "h2d_bytes_per_step": int(hin.numel() * 4), "d2h_bytes_per_step": int(ho.numel() * 4),
        "note": "no CUDA graph: 64 kvc_decode_step calls per step issued from the host through the C "
                "entry point, each step appending the next position; host_us_per_call is the host time "
                "of one call (argument checks, planning, launch) over the first 8 steps, before the "
                "launch queue fills"}
    cache.close()
    del cache
    torch.cuda.empty_cache()
    if rank == 0:
        # The optional phases run one per child process (a fresh CUDA context each), so
        # that a failing phase is reported as that phase's error and the line above stands.
        if args.host_n > 0:
            out["host"] = run_child(args, "host")
            h = out["host"]
            if isinstance(h, dict) and "pipelined" in h and "ordered" in h:
                # the metric's second half, near the front of the line
                summary = {"n_kv": h.get("n_kv"), "link_gbs": h.get("link_gbs"),
                           "pipelined_steps_per_s": h["pipelined"]["steps_per_s"],
                           "pipelined_steps_per_s_median": h["pipelined"].get("steps_per_s_median"),
                           "pipelined_frac_of_link": h["pipelined"]["frac_of_link"],
                           "ordered_steps_per_s": h["ordered"]["steps_per_s"],
                           "ordered_frac_of_link": h["ordered"]["frac_of_link"]}
                keys = list(out.keys())
                at = keys.index("unit") + 1
                out = {**{k: out[k] for k in keys[:at]}, "host_32k": summary, **{k: out[k] for k in keys[at:]}}
        if args.host_matrix:
            out["host_matrix"] = run_child(args, "host_matrix")
        if not args.no_extra:
            ex = {}
            for name in EXTRA_ROWS:
                if args.rows and name not in args.rows.split(","):
                    continue
                ex[name] = run_child(args, name)
            out["rows"] = ex
    if rank == 0 and not args.no_cpu_baseline and not args.no_extra:
        try:
            out["cpu_rows"] = oracle_rows(args)
        except Exception as e:  # reported, not fatal
            out["cpu_rows"] = {"error": str(e)[:300]}
    if rank == 0 and not args.no_cpu_baseline:
        layers = oracle_sample(n, args.cpu_sample_layers, args.type)
        passes, dt, threads = 0, 0.0, 1
        while passes == 0 or dt < args.cpu_seconds:
            _, d1, threads = time_oracle(layers, n, args.type)
            dt += d1
            passes += 1
        gbs = passes * len(layers) * n * kv_bytes_per_row(args.type) / dt / GB
        out["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": "%d of %d layers x %d passes, all %d query heads, n_kv=%d (%.1f s)"
                                         % (args.cpu_sample_layers, L, passes, H, n, dt)}
    return out


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.child:
        import __graft_entry__

        __graft_entry__.build()
        print(json.dumps(child_phase(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        import __graft_entry__

        __graft_entry__.build()
        out = run_ours(args, rank, world)
        if rank == 0:
            print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
