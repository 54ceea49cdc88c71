"""Benchmark of the R-KV compression step on GB300.

One step = one ``rkv_compress`` call over every (layer, sequence, KV head)
problem of the workload: key statistics, importance, thresholded Gram ->
redundancy and Z, top-k select, and the copy of the kept K/V rows.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-e2e] [--no-cpu-baseline]

Prints one JSON line (rank 0).  ``value`` is compressed KV tokens per second
(P * n_cached token slots per step) over all ranks, device-timed with CUDA
events on the launching stream, inputs resident in HBM (K + V are far larger
than L2, so no L2 flush is needed).  ``e2e`` is the same metric with the
host->device copy of K, V, Q_obs from pinned memory and the device->host copy
of the compacted K, V and the indices inside the timed region.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_kv_cache_02_gb300 import rkv, workloads as wl  # noqa: E402

METRIC = "KV tokens compressed/sec + steps/sec (1 GB300); % tensor-pipe & % HBM roofline"

# DRAM bytes (read + write) per problem measured by ncu on a 1,024-problem
# copy of the Llama-8B-shaped workload and a 768-problem copy of the
# Qwen-14B-shaped one (the committed per-kernel ncu summaries),
# with the sha256 of the kernel source they were measured on; a changed source
# reports traffic null.  Every kernel streams whole problems, so traffic scales
# with the problem count.
NCU_TRAFFIC = {
    "llama8b_full": {
        "importance_tc": ("k_importance_tc.cu", "9debeb48aa3a2eafc245d0af2bc3979d401067cc8e37bdd45a4a9463acc7082d", (310465536 + 12756480) / 1024),
        "gram_tc": ("k_gram_tc.cu", "a97ab1ebb4b6aa45acd0053a51d1b3e57e5b909e2df783f344f566b853e04f48", (317408256 + 9883904) / 1024),
        "compact": ("k_compact.cu", "e1f10483478e846d1525863f92693bb15ce63fdb2c3ec308a1192e61053d2281", (541721600 + 492887808) / 1024),
    },
    # the Qwen-14B-shaped step, captured on 768 problems (K 830 MB)
    "qwen14b": {
        "key_stats": ("k_key_stats.cu", "95b35392fb1c978ea7baa169ce85d537de074573cfd2711b5af30a594ca84177", (830592000 + 31349000) / 768),
        "importance_tc": ("k_importance_tc.cu", "9debeb48aa3a2eafc245d0af2bc3979d401067cc8e37bdd45a4a9463acc7082d", (1215002000 + 25443000) / 768),
        "gram_tc": ("k_gram_tc_pairs.cu", "ed9472e6e08de81ce281fd4c00809133d27de62737a0af54ed516a6480406460", (3823741000 + 34038000) / 768),
        "compact": ("k_compact.cu", "e1f10483478e846d1525863f92693bb15ce63fdb2c3ec308a1192e61053d2281", (1623967000 + 1578236000) / 768),
    },
    # the paged round (bs 128: the pool read in place, 8 heads per block)
    "llama8b_full_paged": {
        "compact_paged": ("k_compact.cu", "e1f10483478e846d1525863f92693bb15ce63fdb2c3ec308a1192e61053d2281", (512742144 + 453292544) / 1024),
    },
}


def measured_traffic(workload: str, kernel: str, problems: int):
    """ncu DRAM bytes per launch for `problems` problems, or None when no
    capture exists for this kernel and workload or the source has changed."""
    import hashlib
    ent = NCU_TRAFFIC.get(workload, {}).get(kernel)
    if ent is None:
        return None
    fn, sha, per_problem = ent
    path = os.path.join(ROOT, "decode_kv_cache_02_gb300", "csrc", fn)
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    except OSError:
        return None
    return per_problem * problems
UNIT = "tokens/s"


# ------------------------------------------------------------------ utils --

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "sm_max_mhz": p.get("sm_max_mhz", 2070.0), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_ms: float, units: float, world: int):
    """Max of the ranks' elapsed times and the sum of their units (the
    whole-job throughput is sum(units) / max(time))."""
    if world == 1:
        return elapsed_ms, units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------- algorithmic work model --

def work_model(w: wl.Workload) -> dict:
    """Algorithmic bytes (HBM) / flops per launch of each kernel, for the
    whole step (all P problems): what each kernel must read and write (or
    the useful flops of the Gram's symmetric half), not what it happens to."""
    P, N, d, G, es = w.problems, w.n_cached, w.head_dim, w.gqa, (2 if w.dtype == "bf16" else 4)
    B, n_obs = w.budget, w.n_obs
    k_bytes = P * N * d * es
    return {
        "key_stats": {"bytes": k_bytes + 2 * P * N * 4},
        "importance": {"bytes": k_bytes + P * G * n_obs * d * es + P * N * 4},
        "importance_tc": {"bytes": k_bytes + P * G * n_obs * d * es + P * N * 4},
        "gram_tc": {"flops": P * N * (N - 1) * d, "bytes": k_bytes + 3 * P * N * 4},
        "gram_simt": {"flops": 2 * P * N * N * d, "bytes": k_bytes + 3 * P * N * 4},
        "select": {"bytes": P * (N - n_obs) * 4 + P * B * 4},
        "gather": {"bytes": 4 * P * B * d * es + P * B * 4},
        # select + gather in one pass: Z read once, idx written, kept K, V moved
        "compact": {"bytes": P * (N - n_obs) * 4 + P * B * 4 + 4 * P * B * d * es},
        # scoring variant: read I and R, write Z
        "variant": {"bytes": 3 * P * N * 4},
    }


# a timed region shorter than this is a burst: the tensor-bound kernel is held
# to the burst bf16 peak (measured over a short loop at full clocks), a longer
# one to the sustained peak (a seconds-long loop under the power cap)
SUSTAINED_REGION_MS = 1000.0


def tensor_peak(peaks: dict, region_ms: float):
    """(peak TFLOP/s, description) for a tensor-bound kernel timed inside a
    region of region_ms milliseconds."""
    if region_ms < SUSTAINED_REGION_MS:
        return peaks["bf16_tflops"], ("bf16 burst (of " + peaks["source"] + "; timed region "
                                      f"{region_ms:.0f} ms < {SUSTAINED_REGION_MS:.0f} ms)")
    return peaks["bf16_tflops_sustained"], ("bf16 sustained (of " + peaks["source"] +
                                            f"; timed region {region_ms:.0f} ms)")


def roofline(kernels: dict, model: dict, peaks: dict, steps: int, w=None,
             region_ms: float = 0.0) -> dict:
    """Roofline of the kernel with the largest device time."""
    name = max(kernels, key=lambda k: kernels[k]["ms"])
    per_launch_ms = kernels[name]["ms"] / max(1, kernels[name]["launches"])
    m = model.get(name, {})
    if name == "gram_tc":
        achieved = m["flops"] / (per_launch_ms * 1e-3) / 1e12
        peak, kind = tensor_peak(peaks, region_ms)
        r = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": peak,
             "unit": "TFLOP/s", "peak_kind": kind,
             "frac_of_burst": achieved / peaks["bf16_tflops"],
             "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    elif name == "gram_simt":
        achieved = m["flops"] / (per_launch_ms * 1e-3) / 1e12
        peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        r = {"kernel": name, "bound": "alu", "achieved": achieved, "peak": peak,
             "unit": "TFLOP/s", "peak_kind": "fp32 FFMA, 152 SMs x 128 lanes x 2 x max SM clock"}
    else:
        achieved = m["bytes"] / (per_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        r = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": peak,
             "unit": "GB/s", "peak_kind": "HBM copy (of " + peaks["source"] + ")"}
    r["frac"] = r["achieved"] / r["peak"]
    r["ms_per_launch"] = per_launch_ms
    r["traffic"] = measured_traffic(w.name, name, w.problems) if w is not None else None
    return r


def roofline_all(kernels: dict, model: dict, peaks: dict, w, region_ms: float) -> dict:
    """Every kernel's time per launch with its fraction of the HBM roof (and
    of the tensor roof for the Gram)."""
    out = {}
    for k, v in kernels.items():
        if k not in model or not v["launches"]:
            continue
        per = v["ms"] / v["launches"] * 1e-3
        m = model[k]
        entry = {"ms_per_launch": per * 1e3, "traffic": measured_traffic(w.name, k, w.problems)}
        if "bytes" in m:
            entry["hbm_frac"] = m["bytes"] / per / 1e9 / peaks["hbm_gbs"]
        if k == "gram_tc":
            entry["tensor_frac"] = m["flops"] / per / 1e12 / tensor_peak(peaks, region_ms)[0]
            entry["tensor_frac_of_burst"] = m["flops"] / per / 1e12 / peaks["bf16_tflops"]
        out[k] = entry
    return out


# ------------------------------------------------------------ CPU oracle --

def cpu_oracle_sample(w: wl.Workload, K, Q, seconds: float = 15.0, max_problems: int = 4096):
    """Times the oracle (as it stands) on a bounded sample of the workload's
    problems on all host cores; returns a cpu_baseline dict in tokens/s."""
    import oracle
    cores = oracle.default_threads()
    # calibrate on a few problems, then size the sample to ~`seconds`
    n0 = min(max(cores, 4), K.shape[0])
    Kh = K[:n0, :w.n_cached].cpu()
    Qh = Q[:n0].cpu()
    t0 = time.perf_counter()
    oracle.score(Kh, Qh, w.n_obs, w.lam, w.beta, w.tau, nthreads=cores)
    dt = time.perf_counter() - t0
    per_problem = dt / n0
    n = int(min(max_problems, K.shape[0], max(n0, seconds / max(per_problem, 1e-9))))
    Kh = K[:n, :w.n_cached].cpu()
    Qh = Q[:n].cpu()
    t0 = time.perf_counter()
    sc = oracle.score(Kh, Qh, w.n_obs, w.lam, w.beta, w.tau, nthreads=cores)
    oracle.select(sc["Z"], w.n_obs, w.budget)
    dt = time.perf_counter() - t0
    # the same on one core, on a sample of about a tenth of the time
    n1 = int(min(n, max(1, 0.1 * seconds / max(per_problem * cores, 1e-9))))
    t0 = time.perf_counter()
    sc1 = oracle.score(Kh[:n1], Qh[:n1], w.n_obs, w.lam, w.beta, w.tau, nthreads=1)
    oracle.select(sc1["Z"], w.n_obs, w.budget)
    dt1 = time.perf_counter() - t0
    return {"value": n * w.n_cached / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.problems} problems of {w.name} (N={w.n_cached}, d={w.head_dim}),"
                      f" scores + selection in fp64, {dt:.1f} s",
            "seconds": dt, "problems": n,
            "one_core": {"value": n1 * w.n_cached / dt1, "unit": UNIT, "problems": n1,
                         "seconds": dt1}}


# ------------------------------------------------------------------ arms --

def run_reference(args, w):
    """The oracle as the reference arm: each step scores and selects a
    bounded sample of the workload's problems on the host cores."""
    import oracle
    world, rank, _ = _dist()
    if rank != 0:
        return
    cores = oracle.default_threads()
    P = min(w.problems, args.ref_problems or max(cores, 16))
    K, V, Q = wl.make_inputs(w, device="cpu", problems=P)
    Kh = K[:, :w.n_cached].double().numpy()
    Qh = Q.double().numpy()
    oracle.score(Kh[:1], Qh[:1], w.n_obs, w.lam, w.beta, w.tau, nthreads=1)  # warm-up
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sc = oracle.score(Kh, Qh, w.n_obs, w.lam, w.beta, w.tau, nthreads=cores)
        oracle.select(sc["Z"], w.n_obs, w.budget)
    dt = time.perf_counter() - t0
    value = args.steps * P * w.n_cached / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, sample_problems=P),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{P} of {w.problems} problems per step (scores + selection)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, **extra):
    c = {"workload": w.name, "layers": w.layers, "batch": w.batch, "kv_heads": w.kv_heads,
         "gqa": w.gqa, "head_dim": w.head_dim, "problems": w.problems, "n_cached": w.n_cached,
         "budget": w.budget, "n_obs": w.n_obs, "lambda": w.lam, "beta": w.beta, "tau": w.tau,
         "l2": "no flush: K+V inputs exceed the 129 MB L2"}
    c.update(extra)
    return c


def _sentences(args, w, dev):
    """Synthetic sentence inputs at the workload's size (model width of the
    Llama-8B configuration), or None without --sentences."""
    if not args.sentences:
        return None
    si = wl.make_sentences(w.batch, w.kv_heads, w.layers, w.n_cached, wl.HIDDEN_LLAMA8B,
                           device=dev)
    reps = rkv.rkv_sentence_reps(si.hidden, si.token_seg, si.max_sentences)
    return rkv.Sentences(reps, si.count, si.seg_id, si.heads, wl.SENT_TAU)


def _schedule(args, w, dev):
    """The ForesightKV-style schedule of --recent-window / --pool-extra /
    --temperature, with seeded uniforms for a sampled pool, or None."""
    if not args.recent_window:
        return None
    L = args.recent_window
    C, k = w.n_cached - L, w.budget - L
    u = None
    if args.pool_extra > 0:
        g = torch.Generator(device=dev).manual_seed(w.seed + 17)
        u = torch.rand((w.problems, C), generator=g, device=dev)
    return rkv.Schedule(L, min(C, k + args.pool_extra), args.temperature, u)


def _step_fn(w, K, V, Q, out_K, out_V, idx, ws, stream, softmax=False, window=1,
             sentences=None, schedule=None):
    """One compression step of workload `w` (with a scoring variant if asked)."""
    if softmax or window != 1 or sentences is not None or schedule is not None:
        def step():
            rkv.rkv_compress_ex(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                                redundancy_softmax=softmax, pool_window=window,
                                sentences=sentences, schedule=schedule, out_K=out_K,
                                out_V=out_V, out_idx=idx, workspace=ws, stream=stream)
    else:
        def step():
            rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                             out_K=out_K, out_V=out_V, out_idx=idx, workspace=ws, stream=stream)
    return step


def _busy(intervals):
    """Union of [start, end) intervals: (total length, merged list)."""
    merged = []
    for a, b in sorted(intervals):
        if merged and a <= merged[-1][1]:
            merged[-1][1] = max(merged[-1][1], b)
        else:
            merged.append([a, b])
    return sum(b - a for a, b in merged), merged


def trace_step(step) -> dict:
    """One more step with the library's launch trace on (global-timer stamps
    around every launch, one clock for both SM partitions): each launch's
    lane and interval, each lane's busy time, and how long the tensor
    partition (importance, Gram) and the other one (selection + copy) were
    busy at the same time."""
    torch.cuda.synchronize()
    rkv.rkv_trace_enable(True)
    step()
    recs = rkv.rkv_trace_read()
    rkv.rkv_trace_enable(False)
    if not recs:
        return {}
    t0 = min(r[2] for r in recs)
    span = (max(r[3] for r in recs) - t0) * 1e-6
    lanes = {}
    for name, lane, a, b in recs:
        lanes.setdefault(lane, []).append(((a - t0) * 1e-6, (b - t0) * 1e-6))
    out = {"span_ms": span, "lanes": {}, "launches": [
        [name, lane, round((a - t0) * 1e-3, 1), round((b - t0) * 1e-3, 1)]
        for name, lane, a, b in recs]}
    names = {0: "caller stream (whole device)", 1: "tensor partition", 2: "hbm partition"}
    merged = {}
    for lane, iv in sorted(lanes.items()):
        busy, merged[lane] = _busy(iv)
        out["lanes"][names.get(lane, str(lane))] = {"launches": len(iv), "busy_ms": busy}
    both = 0.0
    for a, b in merged.get(1, []):
        for c, d in merged.get(2, []):
            both += max(0.0, min(b, d) - max(a, c))
    out["tensor_and_hbm_busy_together_ms"] = both
    out["launches_columns"] = ["kernel", "lane", "start_us", "end_us"]
    return out


def _time_steps(step, steps, warmup, ws, stream, local, world):
    """W untimed steps, then K steps between CUDA events on the launching
    stream with a barrier and a synchronize on both sides and the clocks
    sampled meanwhile.  The per-kernel split comes from K more steps after
    the timed region, each launch between CUDA events on its own stream (the
    events cost the grouped schedule ~0.1 ms a step, so they stay out of the
    timed region).  Returns (elapsed ms, per-kernel totals, clocks)."""
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    if rkv.rkv_get_device_status(ws) != 0:
        raise RuntimeError("a kernel reported a device error during warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        _barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
    elapsed = start.elapsed_time(stop)
    rkv.rkv_timing_read(reset=True)
    rkv.rkv_timing_enable(True)
    for _ in range(steps):
        step()
    rkv.rkv_timing_enable(False)
    torch.cuda.synchronize()
    timing = rkv.rkv_timing_read(reset=True)
    kernels = {k: {"ms": v[0], "launches": v[1]} for k, v in timing.items() if v[1] > 0}
    if rkv.rkv_get_device_status(ws) != 0:
        raise RuntimeError("a kernel reported a device error in the timed region")
    return elapsed, kernels, clocks.summary()


# lambda / beta / tau swept one at a time around the page's setting, and the
# scoring variants (beta above 63 would switch to the CUDA-core Gram)
SWEEP = ([{"lam": v} for v in (0.0, 0.5, 1.0)] + [{"beta": v} for v in (0, 1, 8, 63)]
         + [{"tau": v} for v in (0.5, 0.7, 0.8, 0.95, 0.99)]
         + [{"softmax": True}, {"window": 7}, {"softmax": True, "window": 7}])


def run_sweep(args, w):
    """One JSON line per setting of SWEEP on the workload (device-timed step
    and per-kernel split; no end-to-end or CPU legs)."""
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rkv.load()
    K, V, Q = wl.make_inputs(w, device=dev, seed=w.seed + rank)
    out_K, out_V = torch.empty_like(K), torch.empty_like(V)
    idx = torch.empty((w.problems, w.budget), dtype=torch.int32, device=dev)
    ws = rkv.alloc_workspace(K, w.gqa, w.n_cached, w.n_obs)
    stream = torch.cuda.current_stream()
    for setting in [{}] + SWEEP:
        ws_ = w.scaled(**{k: v for k, v in setting.items() if k in ("lam", "beta", "tau")})
        step = _step_fn(ws_, K, V, Q, out_K, out_V, idx, ws, stream,
                        setting.get("softmax", False), setting.get("window", 1))
        elapsed, kernels, clocks = _time_steps(step, args.steps, args.warmup, ws, stream, local,
                                               world)
        line = {"sweep": {"lambda": ws_.lam, "beta": ws_.beta, "tau": ws_.tau,
                          "redundancy_softmax": setting.get("softmax", False),
                          "pool_window": setting.get("window", 1)},
                "workload": w.name, "steps": args.steps, "ms_per_step": elapsed / args.steps,
                "value": args.steps * w.problems * w.n_cached / (elapsed * 1e-3), "unit": UNIT,
                "kernels_ms_per_step": {k: v["ms"] / args.steps for k, v in kernels.items()},
                "clocks": clocks}
        if rank == 0:
            print(json.dumps(line), flush=True)


def run_paged(args, w):
    """The step on a paged cache (rkv_paged_compress, in place): the
    workload's K, V scattered into [num_blocks, H, bs, d] pools through a
    shuffled block table.  Each round compacts the pools and clears the
    table's freed entries, so the pristine pools and table are restored
    between timed rounds (outside the events; the 9.7 GB copy also flushes
    L2) and the K rounds' event times are summed."""
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rkv.load()
    bs = args.block_size
    S, H, N, d = w.layers * w.batch, w.kv_heads, w.n_cached, w.head_dim
    nb = -(-N // bs)
    num_blocks = S * nb
    g = torch.Generator().manual_seed(w.seed)
    table0 = torch.randperm(num_blocks, generator=g).reshape(S, nb).to(torch.int32).to(dev)
    K, V, Q = wl.make_inputs(w, device=dev, seed=w.seed + rank)
    pools = []
    for X in (K, V):
        pool = torch.zeros((num_blocks, H, bs, d), dtype=X.dtype, device=dev)
        Xl = X[:, :N].reshape(S, H, N, d)
        if nb * bs > N:
            Xl = torch.cat([Xl, torch.zeros((S, H, nb * bs - N, d), dtype=X.dtype, device=dev)], 2)
        pool[table0.long()] = Xl.reshape(S, H, nb, bs, d).permute(0, 2, 1, 3, 4)
        pools.append(pool)
    del K, V
    K0, V0 = pools
    K_pool, V_pool, table = K0.clone(), V0.clone(), table0.clone()
    n_free = rkv.rkv_paged_freed_per_seq(K_pool, table, N, w.budget)
    idx = torch.empty((S * H, w.budget), dtype=torch.int32, device=dev)
    freed = torch.empty((S, n_free), dtype=torch.int32, device=dev)
    ws = torch.zeros(rkv.rkv_paged_workspace_size(K_pool, table, w.gqa, N, w.n_obs, w.beta),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sent = _sentences(args, w, dev)
    seg0 = sent.seg_id.clone() if sent is not None else None

    def restore():
        K_pool.copy_(K0)
        V_pool.copy_(V0)
        table.copy_(table0)
        if sent is not None:
            sent.seg_id.copy_(seg0)

    def step():
        rkv.rkv_paged_compress(K_pool, V_pool, Q, table, N, w.budget, w.n_obs, w.lam, w.beta,
                               w.tau, redundancy_softmax=args.redundancy_softmax,
                               pool_window=args.pool_window, sentences=sent, out_idx=idx,
                               out_freed=freed, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        restore()
        step()
    torch.cuda.synchronize()
    if rkv.rkv_get_device_status(ws) != 0:
        raise RuntimeError("a kernel reported a device error during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    rkv.rkv_timing_read(reset=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        torch.cuda.synchronize()
        for a, b in evs:
            restore()
            a.record(stream)
            rkv.rkv_timing_enable(True)
            step()
            rkv.rkv_timing_enable(False)
            b.record(stream)
        torch.cuda.synchronize()
    elapsed = sum(a.elapsed_time(b) for a, b in evs)
    timing = rkv.rkv_timing_read(reset=True)
    kernels = {k: {"ms": v[0], "launches": v[1]} for k, v in timing.items() if v[1] > 0}
    if rkv.rkv_get_device_status(ws) != 0:
        raise RuntimeError("a kernel reported a device error in the timed region")
    # rows the in-place compaction moves: from each problem's first evicted
    # position on (the identity prefix stays where it is)
    ar = torch.arange(w.budget, device=dev, dtype=torch.int32)
    first = torch.where(idx != ar, ar, w.budget).min(dim=1).values
    moved_rows = int((w.budget - first).sum())
    es = 2 if w.dtype == "bf16" else 4
    P = S * H
    model = {
        "key_stats_paged": {"bytes": 2 * P * N * d * es + 2 * P * N * 4},
        "compact_paged": {"bytes": P * (N - w.n_obs) * 4 + P * w.budget * 4
                          + 4 * moved_rows * d * es},
    }
    peaks = _peaks()
    roof = {}
    for k, v in kernels.items():
        per = v["ms"] / v["launches"] * 1e-3
        e = {"ms_per_launch": per * 1e3,
             "traffic": measured_traffic(w.name + "_paged", k, P) if bs == 128 else None}
        if k in model:
            e["hbm_frac"] = model[k]["bytes"] / per / 1e9 / peaks["hbm_gbs"]
        if k == "gram_tc":
            e["tensor_frac"] = P * N * (N - 1) * d / per / 1e12 / peaks["bf16_tflops_sustained"]
        roof[k] = e
    line = {
        "mode": "paged", "metric": METRIC, "value": args.steps * P * N / (elapsed * 1e-3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": elapsed / args.steps, "higher_is_better": True, "dtype": w.dtype,
        "data": "synthetic",
        "config": _config(w, block_size=bs, num_seqs=S, num_blocks=num_blocks,
                          blocks_freed_per_seq=n_free, moved_rows_per_problem=moved_rows / P,
                          variant={"redundancy_softmax": args.redundancy_softmax,
                                   "pool_window": args.pool_window,
                                   "sentences": sent is not None},
                          l2="pools restored between rounds (9.7 GB copy, flushes L2)"),
        "kernels_ms_per_step": {k: v["ms"] / args.steps for k, v in kernels.items()},
        "roofline_all": roof,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args, w):
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rkv.load()
    if args.schedule == "one-launch":
        rkv.rkv_set_overlap(rkv.RKV_SCHEDULE_ONE_LAUNCH)
    K, V, Q = wl.make_inputs(w, device=dev, seed=w.seed + rank)
    out_K = torch.empty_like(K)
    out_V = torch.empty_like(V)
    idx = torch.empty((w.problems, w.budget), dtype=torch.int32, device=dev)
    ws = rkv.alloc_workspace(K, w.gqa, w.n_cached, w.n_obs)
    stream = torch.cuda.current_stream()
    sent = _sentences(args, w, dev)
    sch = _schedule(args, w, dev)
    step = _step_fn(w, K, V, Q, out_K, out_V, idx, ws, stream, args.redundancy_softmax,
                    args.pool_window, sent, sch)
    elapsed, kernels, clock_summary = _time_steps(step, args.steps, args.warmup, ws, stream,
                                                  local, world)
    launches = sum(v["launches"] for v in kernels.values())

    units = args.steps * w.problems * w.n_cached
    t_max, u_sum = aggregate(elapsed, units, world)
    peaks = _peaks()
    model = work_model(w)
    line = {
        "metric": METRIC, "value": u_sum / (t_max * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": _config(w, mode="out-of-place (outputs in separate buffers)",
                          parallelism=f"replicas x{world}, no collective"),
        "steps_per_s": world * args.steps / (t_max * 1e-3),
        "evicted_tokens_per_s": world * args.steps * w.problems * (w.n_cached - w.budget)
        / (t_max * 1e-3),
        "gpu_launches": launches,
        "kernels_ms_per_step": {k: v["ms"] / args.steps for k, v in kernels.items()},
        "clocks": clock_summary,
    }
    if args.redundancy_softmax or args.pool_window != 1 or sent is not None or sch is not None:
        line["config"]["variant"] = {"redundancy_softmax": args.redundancy_softmax,
                                     "pool_window": args.pool_window}
        if sch is not None:
            line["config"]["variant"]["schedule"] = {
                "recent_window": sch.recent_window, "pool_size": sch.pool_size,
                "temperature": sch.temperature, "sampled": sch.uniforms is not None}
        if sent is not None:
            line["config"]["variant"]["sentences"] = {
                "sequences": sent.reps.shape[0], "max_sentences": sent.reps.shape[1],
                "hidden": sent.reps.shape[2], "tau": sent.tau}
    # The step's default schedule scores groups of problems on one SM
    # partition while the previous group is compacted on the other, so its
    # kernels share the device and overlap in time.  Each kernel's roofline
    # is taken from the one-launch-per-stage schedule instead, where every
    # kernel has the whole device to itself, timed the same way.
    grouped = kernels.get("gram_tc", {}).get("launches", 0) > args.steps
    line["schedule"] = {
        "kind": "two SM partitions (importance + Gram | select + copy), groups overlapped"
        if grouped else "one launch per stage over the whole device",
        "groups_per_step": kernels.get("gram_tc", {}).get("launches", 0) // max(1, args.steps)}
    r_elapsed, r_kernels = elapsed, kernels
    if grouped:
        rkv.rkv_set_overlap(rkv.RKV_SCHEDULE_ONE_LAUNCH)
        try:
            r_elapsed, r_kernels, _ = _time_steps(step, args.steps, args.warmup, ws, stream,
                                                  local, world)
        finally:
            rkv.rkv_set_overlap(*rkv.DEFAULT_OVERLAP)

        line["schedule"]["one_launch_ms_per_step"] = r_elapsed / args.steps
        line["schedule"]["one_launch_kernels_ms_per_step"] = {
            k: v["ms"] / args.steps for k, v in r_kernels.items()}
    if grouped:
        line["trace"] = trace_step(step)
    line["roofline"] = roofline(r_kernels, model, peaks, args.steps, w, region_ms=r_elapsed)
    line["roofline"]["schedule"] = "one launch per stage (kernel alone on the whole device)"
    # all kernels' fractions, for the record
    line["roofline_all"] = roofline_all(r_kernels, model, peaks, w, r_elapsed)

    if not args.no_e2e:
        line["e2e"] = e2e(args, w, K, V, Q, out_K, out_V, idx, ws, stream, world, sent)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, K, Q, seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e(args, w, K, V, Q, out_K, out_V, idx, ws, stream, world, sent=None):
    """Same step through the public API with host buffers: every step copies
    K, V, Q_obs in from pinned host memory and the compacted K, V (the kept
    rows) and idx out.  Steps are pipelined over two device buffer sets: the
    host->device copy of step k+1 and the device->host copy of step k-1 run on
    their own streams while step k computes (events order each slot's reuse).
    The timed region spans the first copy-in to the last copy-out."""
    B = w.budget
    hK = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
    hV = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
    hQ = torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True)
    hK.copy_(K)
    hV.copy_(V)
    hQ.copy_(Q)
    oK = torch.empty((K.shape[0], B, K.shape[2]), dtype=K.dtype, pin_memory=True)
    oV = torch.empty_like(oK, pin_memory=True)
    oI = torch.empty(idx.shape, dtype=idx.dtype, pin_memory=True)
    # the kept rows land in outputs of `budget` rows per problem, so that they
    # come back as one contiguous copy
    slots = [(K, V, Q, torch.empty_like(oK, device=K.device), torch.empty_like(oV, device=K.device),
              idx),
             (torch.empty_like(K), torch.empty_like(V), torch.empty_like(Q),
              torch.empty_like(oK, device=K.device), torch.empty_like(oV, device=K.device),
              torch.empty_like(idx))]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    done_compute = [None, None]
    done_d2h = [None, None]

    def step(k):
        sl = k % 2
        dK, dV, dQ, dOK, dOV, dI = slots[sl]
        e_in = ev()
        with torch.cuda.stream(h2d_s):
            if done_compute[sl] is not None:
                h2d_s.wait_event(done_compute[sl])  # slot's inputs consumed
            dK.copy_(hK, non_blocking=True)
            dV.copy_(hV, non_blocking=True)
            dQ.copy_(hQ, non_blocking=True)
            e_in.record(h2d_s)
        stream.wait_event(e_in)
        if done_d2h[sl] is not None:
            stream.wait_event(done_d2h[sl])  # slot's outputs copied out
        rkv.rkv_compress_ex(dK, dV, dQ, w.n_cached, B, w.n_obs, w.lam, w.beta, w.tau,
                            redundancy_softmax=args.redundancy_softmax,
                            pool_window=args.pool_window, sentences=sent, out_K=dOK, out_V=dOV,
                            out_idx=dI, workspace=ws, stream=stream)
        e_c = ev()
        e_c.record(stream)
        done_compute[sl] = e_c
        e_out = ev()
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(e_c)
            oK.copy_(dOK, non_blocking=True)
            oV.copy_(dOV, non_blocking=True)
            oI.copy_(dI, non_blocking=True)
            e_out.record(d2h_s)
        done_d2h[sl] = e_out

    steps = max(1, min(args.steps, args.e2e_steps))
    for k in range(2):
        step(k)
    torch.cuda.synchronize()
    done_compute[:] = [None, None]
    done_d2h[:] = [None, None]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    s0.record(stream)
    h2d_s.wait_event(s0)
    d2h_s.wait_event(s0)
    last = None
    for k in range(steps):
        step(k)
    stream.wait_event(done_d2h[(steps - 1) % 2])
    if steps > 1:
        stream.wait_event(done_d2h[(steps - 2) % 2])
    s1.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    del last
    t_max, u_sum = aggregate(s0.elapsed_time(s1), steps * w.problems * w.n_cached, world)
    h2d = hK.numel() * hK.element_size() + hV.numel() * hV.element_size() + \
        hQ.numel() * hQ.element_size()
    d2h = oK.numel() * oK.element_size() * 2 + oI.numel() * oI.element_size()
    return {"value": u_sum / (t_max * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": t_max / steps,
            "pipelined": "2 buffer sets; copy-in, compute, copy-out on three streams",
            "outputs": "budget rows per problem (contiguous copy-out)"}


def run_stream(args, w):
    """The sustained decode stream: every `buffer` generated tokens the new
    keys/values are appended, and when the cache exceeds the budget one
    in-place rkv_compress call compacts every (layer, sequence, head) problem
    back to the budget.  Only the compression calls are timed (CUDA events
    on the launching stream); the amortised cost is their total time over all
    generated tokens (sequences x tokens)."""
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rkv.load()
    P = w.problems
    src = wl.StreamSource(w, device=dev, seed=w.seed + rank)
    cap = w.budget + w.buffer
    K = torch.zeros(P, cap, w.head_dim, dtype=w.torch_dtype, device=dev)
    V = torch.zeros_like(K)
    idx = torch.empty((P, w.budget), dtype=torch.int32, device=dev)
    ws = rkv.alloc_workspace(K, w.gqa, cap, w.n_obs)
    stream = torch.cuda.current_stream()
    n, rounds, total_ms, launches = 0, 0, 0.0, 0
    work = {}  # algorithmic bytes / flops of every kernel, summed over the rounds
    rkv.rkv_timing_read(reset=True)
    with ClockSampler(local) as clocks:
        while src.t < w.gen_tokens:
            kc, vc = src.next_chunk()
            K[:, n:n + w.buffer] = kc
            V[:, n:n + w.buffer] = vc
            n += w.buffer
            if n <= w.budget:
                continue
            Q = src.queries(K[:, n - 1])
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            rkv.rkv_timing_enable(True)
            rkv.rkv_compress(K, V, Q, n, w.budget, w.n_obs, w.lam, w.beta, w.tau, out_K=K,
                             out_V=V, out_idx=idx, workspace=ws, stream=stream)
            rkv.rkv_timing_enable(False)
            s1.record(stream)
            s1.synchronize()
            total_ms += s0.elapsed_time(s1)
            rounds += 1
            for k, m in work_model(w.scaled(n_cached=n)).items():
                acc = work.setdefault(k, {})
                for unit, v in m.items():
                    acc[unit] = acc.get(unit, 0.0) + v
            n = w.budget
    timing = rkv.rkv_timing_read(reset=True)
    launches = sum(v[1] for v in timing.values())
    if rkv.rkv_get_device_status(ws) != 0:
        raise RuntimeError("a kernel reported a device error in the stream")
    gen = w.batch * w.gen_tokens  # generated tokens over all sequences
    line = {
        "metric": "amortised compression cost per generated token (decode stream)",
        "value": total_ms * 1e3 / gen, "unit": "us/token", "higher_is_better": False,
        "n_gpus": 1, "steps": rounds, "warmup": 0, "ms_per_step": total_ms / rounds,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": _config(w, mode="in place", gen_tokens=w.gen_tokens, buffer=w.buffer,
                          compress_at=f"N={w.budget + w.buffer} after the first at "
                                      f"{(w.budget // w.buffer + 1) * w.buffer}"),
        "compressed_tokens_per_s": P * (w.budget + w.buffer) * rounds / (total_ms * 1e-3),
        "gpu_launches": launches,
        "kernels_ms_total": {k: v[0] for k, v in timing.items() if v[1]},
        "clocks": clocks.summary(),
    }
    # rooflines over the whole stream: each kernel's summed algorithmic work
    # over its summed time (the work model is per round, so with `launches`
    # set to 1 the per-launch figures are the stream's totals)
    kernels = {k: {"ms": v[0], "launches": 1} for k, v in timing.items() if v[1]}
    peaks = _peaks()
    line["roofline"] = roofline(kernels, work, peaks, rounds, w, region_ms=total_ms)
    line["roofline"]["traffic"] = None
    line["roofline_all"] = roofline_all(kernels, work, peaks, w, total_ms)
    for e in line["roofline_all"].values():
        e["ms_total"] = e.pop("ms_per_launch")
        e["traffic"] = None
    print(json.dumps(line), flush=True)


def run_all_configs(args):
    """One JSON line per workload of the table (tiny, Llama-8B layer, Llama-8B
    full step, Qwen-14B step, decode stream), each with its rooflines; the
    end-to-end and CPU legs are left to the single-workload runs."""
    args.no_e2e = True
    args.no_cpu_baseline = True
    for w in wl.WORKLOADS:
        if w.gen_tokens:
            run_stream(args, w)
        else:
            run_ours(args, w)
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama8b_full", choices=list(wl.BY_NAME))
    ap.add_argument("--config", type=int, default=None, choices=range(len(wl.WORKLOADS)),
                    help="the workload by its position in the table (0 tiny .. 4 stream)")
    ap.add_argument("--seed", type=int, default=None,
                    help="seed of the synthetic inputs (default: the workload's own)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-problems", type=int, default=0)
    ap.add_argument("--problems", type=int, default=0,
                    help="override the problem count (smaller copies for profiling; "
                         "such a run is not the workload's bench line)")
    ap.add_argument("--redundancy-softmax", action="store_true",
                    help="scoring variant: softmax of the redundancy over the candidates")
    ap.add_argument("--pool-window", type=int, default=1,
                    help="scoring variant: odd max-pooling window on the importance")
    ap.add_argument("--paged", action="store_true",
                    help="time the step on a paged cache (block pools + block table)")
    ap.add_argument("--block-size", type=int, default=16, help="rows per block with --paged")
    ap.add_argument("--sentences", action="store_true",
                    help="scoring variant: sentence-level penalty on synthetic sentences")
    ap.add_argument("--recent-window", type=int, default=0,
                    help="schedule: keep the newest L rows (ForesightKV-style), 0 = off")
    ap.add_argument("--pool-extra", type=int, default=0,
                    help="schedule: pool = kept + this many, sampled by Gumbel keys")
    ap.add_argument("--temperature", type=float, default=0.05,
                    help="schedule: sampling temperature")
    ap.add_argument("--sweep", action="store_true",
                    help="time the step over a lambda/beta/tau/variant sweep, one line each")
    ap.add_argument("--all-configs", action="store_true",
                    help="one line per workload (tiny .. stream), with rooflines")
    ap.add_argument("--schedule", default="grouped", choices=["grouped", "one-launch"],
                    help="the library's step schedule: groups of problems on two SM "
                         "partitions (its default) or one launch per stage")
    args = ap.parse_args()
    if args.all_configs and args.impl == "ours":
        run_all_configs(args)
        return
    w = wl.WORKLOADS[args.config] if args.config is not None else wl.BY_NAME[args.workload]
    if args.seed is not None:
        w = w.scaled(seed=args.seed)
    if args.problems:
        # a scaled copy: sequences of the workload's heads where the count
        # allows (blocks of a paged pool hold all heads of a sequence)
        H = w.kv_heads if args.problems % w.kv_heads == 0 else 1
        w = w.scaled(layers=1, batch=args.problems // H, kv_heads=H)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.sweep:
        run_sweep(args, w)
    elif args.paged:
        run_paged(args, w)
    elif w.gen_tokens:
        run_stream(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
