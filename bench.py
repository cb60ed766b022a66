"""Benchmark of the binned-summation hot path on GB300.

One step = one pass of every hot-path row over its full-size synthetic input:
  binned sum, K=3:            float32 N(0,1) 100M; float64 wide-range 100M
  binned cumulative sum, K=3: the same two arrays (out of place)
  segmented binned sum, K=3:  [4096, 4096] float32 rows
  float32 variance kernel:    [4096, 4096] float32, axis 1, ddof 1
The value is elements processed per second over the whole step
(GElements/s); per-row device times, the roofline of the dominant kernel, an
end-to-end run through the C ABI with host buffers, comparison baselines and
the CPU oracle's rate are reported on the same JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_SUM = 100_000_000
ROWS = COLS = 4096
METRIC = "GElements/s and % HBM roofline: ADN sum/cumsum 100M fp32/fp64 K=3; var [4096²]"
WORKLOAD = ("adn sum+cumsum 1e8 f32 N(0,1) & 1e8 f64 wide-range (K=3) + segmented sum and "
            "stable_var_f32 [4096,4096] axis1 ddof1")
# algorithmic bytes per element of each row (input read once, output written once)
ROWS_SPEC = [
    # name, elements, bytes/element
    ("var_f32_4096x4096", ROWS * COLS, 4),
    ("sum_f32_1e8", N_SUM, 4),
    ("segsum_f32_4096x4096", ROWS * COLS, 4),
    ("cumsum_f32_1e8", N_SUM, 8),
    ("sum_f64_1e8", N_SUM, 8),
    ("cumsum_f64_1e8", N_SUM, 16),
]


def set_vector_length(n: int) -> None:
    """Use n-element vectors for the 1e8-element rows (smaller profiling
    captures); the row names keep their labels."""
    global N_SUM, ROWS_SPEC
    N_SUM = n
    ROWS_SPEC = [(name, (n if name.endswith("1e8") else cnt), bpe) for name, cnt, bpe in ROWS_SPEC]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ours
def run_ours(args):
    import numpy as np
    import torch

    from compensated_bit_reproducible_gb300 import api, inputs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    api.lib()
    api.validate_environment()
    seed_off = 100 * rank
    h32 = inputs.normal_f32(N_SUM, seed=1 + seed_off)
    h64 = inputs.wide_f64(N_SUM, seed=2 + seed_off)
    hA = inputs.offset_rows(ROWS, COLS, seed=3 + seed_off)
    x32 = torch.from_numpy(h32).to(dev)
    x64 = torch.from_numpy(h64).to(dev)
    A = torch.from_numpy(hA).to(dev)
    c32 = torch.empty_like(x32)
    c64 = torch.empty_like(x64)
    s32 = torch.empty(1, dtype=torch.float32, device=dev)
    s64 = torch.empty(1, dtype=torch.float64, device=dev)
    vout = torch.empty(ROWS, dtype=torch.float32, device=dev)
    vmean = torch.empty(ROWS, dtype=torch.float32, device=dev)
    segout = torch.empty(ROWS, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    calls = {
        "var_f32_4096x4096": lambda: api.stable_var(A, axis=1, ddof=1, out=vout, mean_out=vmean),
        "sum_f32_1e8": lambda: api.repro_sum_async(x32, s32, args.k),
        "segsum_f32_4096x4096": lambda: api.repro_segsum(A, axis=1, K=3, out=segout),
        "cumsum_f32_1e8": lambda: api.repro_cumsum(x32, out=c32, K=args.k),
        "sum_f64_1e8": lambda: api.repro_sum_async(x64, s64, args.k),
        "cumsum_f64_1e8": lambda: api.repro_cumsum(x64, out=c64, K=args.k),
    }
    # kernels per call: the double sum is the fixed-index first pass plus its
    # second pass (idle unless the first missed); a cumulative sum is totals,
    # scan and replay plus four gated fallback kernels (no call launches a
    # memset)
    launches_per_row = {"var_f32_4096x4096": 1, "sum_f32_1e8": 1, "segsum_f32_4096x4096": 1,
                        "cumsum_f32_1e8": 7, "sum_f64_1e8": 2, "cumsum_f64_1e8": 7}

    active = [r for r in ROWS_SPEC if not args.rows or r[0] in args.rows.split(",")]

    def step(evs=None):
        for name, _, _ in active:
            if evs is not None:
                evs[name][0].append(torch.cuda.Event(enable_timing=True))
                evs[name][0][-1].record(stream)
            calls[name]()
            if evs is not None:
                evs[name][1].append(torch.cuda.Event(enable_timing=True))
                evs[name][1][-1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    clocks = ClockSampler(local)
    clocks.start()
    evs = {name: ([], []) for name, _, _ in active}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step(evs)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, ws)
    ms_step = ms_total / args.steps
    elems_step = sum(n for _, n, _ in active)
    value = elems_step * ws / (ms_step * 1e-3) / 1e9
    hbm, peak_kind = load_peaks()
    rows = {}
    for name, n, bpe in active:
        durs = [a.elapsed_time(b) for a, b in zip(*evs[name])]
        ms = sum(durs) / len(durs)
        rows[name] = {"ms": round(ms, 4), "gelem_s": round(n / (ms * 1e-3) / 1e9, 2),
                      "gb_s": round(n * bpe / (ms * 1e-3) / 1e9, 1),
                      "hbm_frac": round(n * bpe / (ms * 1e-3) / 1e9 / hbm, 4)}
    dom = max(rows, key=lambda k: rows[k]["ms"])
    dom_n, dom_bpe = [(n, b) for nm, n, b in active if nm == dom][0]
    achieved = dom_n * dom_bpe / (rows[dom]["ms"] * 1e-3) / 1e9
    traffic = load_traffic(dom)

    # end to end through the C ABI: pinned host buffers in, results out
    e2e = cpu = comparisons = None
    if not args.skip_extras:
        e2e = run_e2e(args, api, torch, h32, h64, hA, dev, stream)
        if rank == 0 and not args.no_cpu_baseline:
            cpu = cpu_baseline(args.cpu_seconds)
        comparisons = run_comparisons(api, torch, x32, x64, A, stream)
    gpu_launches = args.steps * sum(launches_per_row[name] for name, _, _ in active)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "GElements/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32+f64 inputs, exact int64/int128 binned lanes",
        "data": "synthetic (seeded numpy generators, shapes and distributions of the pages' workloads)",
        "config": {"workload": WORKLOAD if N_SUM == 100_000_000 else WORKLOAD.replace("1e8", "%d" % N_SUM),
                   "K": args.k,
                   "elements_per_step_per_gpu": elems_step,
                   "l2": "every input is larger than L2 or follows >= 400 MB of other traffic in the step",
                   "parallelism": "independent replicas" if ws > 1 else "single GPU"},
        "rows": rows,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic},
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "cpu_baseline": cpu,
        "comparisons": comparisons,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def load_traffic(kernel_row: str):
    """DRAM bytes per call of a row from the committed ncu summary
    (profiles/traffic_per_call.md), or None when not captured for the
    current kernels."""
    p = os.path.join(ROOT, "profiles", "traffic_per_call.md")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) == 3 and cells[0] == kernel_row and cells[2] == "yes":
                try:
                    return int(cells[1])
                except ValueError:
                    return None
    return None


def run_e2e(args, api, torch, h32, h64, hA, dev, stream):
    """Same step through the C ABI from pinned host buffers: every input is
    copied host->device once and every result device->host inside the timed
    region.  Each 1e8-element vector goes over the link in chunks (the
    library's binned states carry the sums across them):
    - chunk 0's cumulative sum is a plain call, chunk j's continues from the
      state of chunks 0..j-1 (repro_cumsum_from_state), and the chunk is
      then deposited into that state; the state's value is the vector's sum.
      Binned states merge exactly, so every output has the bits of the
      one-call cumulative sum and sum (checked below, outside the timed
      region);
    - input copies run on one stream, in the order the calls use them, and
      result copies on another, each after an event on the compute stream,
      so a chunk's results go back while later chunks come in.
    The host link (about 210 GB/s in, 190 GB/s out, measured with pinned
    copies) bounds this number, not the kernels."""
    p32 = torch.from_numpy(h32).pin_memory()
    p64 = torch.from_numpy(h64).pin_memory()
    pA = torch.from_numpy(hA).pin_memory()
    oc32 = torch.empty(N_SUM, dtype=torch.float32).pin_memory()
    oc64 = torch.empty(N_SUM, dtype=torch.float64).pin_memory()
    ov = torch.empty(ROWS, dtype=torch.float32).pin_memory()
    om = torch.empty(ROWS, dtype=torch.float32).pin_memory()
    oseg = torch.empty(ROWS, dtype=torch.float32).pin_memory()
    os32 = torch.empty(1, dtype=torch.float32).pin_memory()
    os64 = torch.empty(1, dtype=torch.float64).pin_memory()
    d32 = torch.empty(N_SUM, dtype=torch.float32, device=dev)
    d64 = torch.empty(N_SUM, dtype=torch.float64, device=dev)
    c32 = torch.empty(N_SUM, dtype=torch.float32, device=dev)
    c64 = torch.empty(N_SUM, dtype=torch.float64, device=dev)
    dA = torch.empty(ROWS, COLS, dtype=torch.float32, device=dev)
    s32 = torch.empty(1, dtype=torch.float32, device=dev)
    s64 = torch.empty(1, dtype=torch.float64, device=dev)
    seg = torch.empty(ROWS, dtype=torch.float32, device=dev)
    var = torch.empty(ROWS, dtype=torch.float32, device=dev)
    mean = torch.empty(ROWS, dtype=torch.float32, device=dev)
    st32 = api.state_new(torch.float32, 3, device=dev, stream=stream)
    st64 = api.state_new(torch.float64, 3, device=dev, stream=stream)
    copy_stream = torch.cuda.Stream(device=dev)
    h2d_stream = torch.cuda.Stream(device=dev)
    bounds = chunk_bounds(N_SUM, max(1, args.e2e_chunks))

    # events made once (each is recorded at most once per step, and a step
    # ends with a device synchronisation)
    ev_pool = [torch.cuda.Event() for _ in range(4 * len(bounds) + 8)]
    ev_next = [0]

    def event():
        ev = ev_pool[ev_next[0]]
        ev_next[0] += 1
        return ev

    def back(dst, src):
        # device->host on the copy stream once `src` is complete
        ev = event()
        ev.record(stream)
        copy_stream.wait_event(ev)
        with torch.cuda.stream(copy_stream):
            dst.copy_(src, non_blocking=True)

    def send(dst, src):
        with torch.cuda.stream(h2d_stream):
            dst.copy_(src, non_blocking=True)
            ev = event()
            ev.record(h2d_stream)
        return ev

    def vector(d, c, oc, st, s, so, evs):
        # on the compute stream: every chunk's cumulative sum, then the sum
        api.state_init(st, d.dtype, 3)
        for j, (a, b) in enumerate(bounds):
            stream.wait_event(evs[j])
            if j == 0:
                api.repro_cumsum(d[a:b], out=c[a:b], K=3)
            else:
                api.repro_cumsum_from_state(d[a:b], st, K=3, out=c[a:b])
            back(oc[a:b], c[a:b])
            api.state_deposit(st, d[a:b], K=3)
        api.state_finalize(st, d.dtype, 3, out=s)
        back(so, s)

    def one():
        # inputs in the order the calls use them: the double vector first, so
        # that its 800 MB of cumulative sums go back while the rest comes in
        ev_next[0] = 0
        e64 = [send(d64[a:b], p64[a:b]) for a, b in bounds]
        eA = send(dA, pA)
        e32 = [send(d32[a:b], p32[a:b]) for a, b in bounds]
        with torch.cuda.stream(stream):
            vector(d64, c64, oc64, st64, s64, os64, e64)
            stream.wait_event(eA)
            api.stable_var(dA, axis=1, ddof=1, out=var, mean_out=mean)
            back(ov, var)
            back(om, mean)
            api.repro_segsum(dA, axis=1, K=3, out=seg)
            back(oseg, seg)
            vector(d32, c32, oc32, st32, s32, os32, e32)
        torch.cuda.synchronize()

    # untimed steps first, as many as the resident loop's warm-up (at least
    # three): in runs with a single one, the slow steps came among the first
    # four timed ones
    for _ in range(max(3, args.warmup)):
        one()
    n = max(1, args.e2e_steps)
    times = []
    # no garbage collection inside the timed steps (as timeit does)
    gc.collect()
    gc_on = gc.isenabled()
    gc.disable()
    try:
        for _ in range(n):
            t = time.perf_counter()
            one()
            times.append(time.perf_counter() - t)
    finally:
        if gc_on:
            gc.enable()
    dt = sum(times) / n
    check_e2e(api, torch, dev, stream, (d32, d64, dA), (oc32, oc64, os32, os64, ov, om, oseg))
    elems = sum(nn for _, nn, _ in ROWS_SPEC)
    h2d = 4 * N_SUM + 8 * N_SUM + 4 * ROWS * COLS
    d2h = 4 * N_SUM + 8 * N_SUM + 4 + 8 + 3 * 4 * ROWS
    # the host link in this run: pinned copies of 1 GiB each way, best of 3
    link = measure_link(torch, dev)
    return {"value": round(elems / dt / 1e9, 3), "unit": "GElements/s", "ms_per_step": round(dt * 1e3, 3),
            "ms_per_step_min": round(min(times) * 1e3, 3), "ms_per_step_max": round(max(times) * 1e3, 3),
            "ms_per_step_median": round(sorted(times)[len(times) // 2] * 1e3, 3),
            "ms_steps": [round(t * 1e3, 3) for t in times],
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n, "chunks": len(bounds),
            "bits_equal_to_resident_calls": True,
            "link_gbs": link,
            "link_bound_ms": round(max(h2d / link["h2d"], d2h / link["d2h"]) / 1e6, 3),
            "link_bound_ms_duplex": round(max(h2d / link["h2d_duplex"], d2h / link["d2h_duplex"]) / 1e6, 3),
            "host_api": run_host_api(api, torch, h32, h64)}


def chunk_bounds(n: int, nch: int):
    """[start, end) of nch nearly equal chunks of an n-element vector:
    multiples of 64 elements, so every chunk starts 256-byte aligned."""
    step = -(-n // nch)
    step = -(-step // 64) * 64
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def check_e2e(api, torch, dev, stream, inputs, outs):
    """The end-to-end leg's host results against the one-call device results
    on the same (device-resident) inputs, bit for bit; raises on any
    difference."""
    d32, d64, dA = inputs
    oc32, oc64, os32, os64, ov, om, oseg = outs
    with torch.cuda.stream(stream):
        want = {
            "cumsum_f32": (oc32, api.repro_cumsum(d32, K=3)),
            "cumsum_f64": (oc64, api.repro_cumsum(d64, K=3)),
            "sum_f32": (os32, api.repro_sum_async(d32, torch.empty(1, dtype=torch.float32, device=dev), 3)),
            "sum_f64": (os64, api.repro_sum_async(d64, torch.empty(1, dtype=torch.float64, device=dev), 3)),
            "segsum": (oseg, api.repro_segsum(dA, axis=1, K=3)),
        }
        v, m = api.stable_var(dA, axis=1, ddof=1)
        want["var"], want["mean"] = (ov, v), (om, m)
    torch.cuda.synchronize()
    for name, (got, ref) in want.items():
        it = torch.int64 if got.dtype == torch.float64 else torch.int32
        if not torch.equal(got.view(it), ref.cpu().view(it)):
            raise RuntimeError("end-to-end %s differs from the one-call device result" % name)


def measure_link(torch, dev):
    """Pinned host<->device copy rates (GB/s) of 1 GiB, best of three: each
    direction alone, and both at once."""
    nb = 1 << 30
    h = torch.empty(nb, dtype=torch.uint8).pin_memory()
    d = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = 1e9
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e-3)
        out[name] = round(nb / best / 1e9, 1)
    # both directions at once, each on its own stream (the end-to-end leg's
    # copies overlap like this)
    h2 = torch.empty(nb, dtype=torch.uint8).pin_memory()
    d2 = torch.empty(nb, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    best_in = best_out = 1e9
    for _ in range(3):
        torch.cuda.synchronize()
        go = torch.cuda.Event()
        go.record()
        evs = []
        for st, dst, src in ((s_in, d, h), (s_out, h2, d2)):
            st.wait_event(go)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            with torch.cuda.stream(st):
                dst.copy_(src, non_blocking=True)
            b.record(st)
            evs.append((a, b))
        torch.cuda.synchronize()
        best_in = min(best_in, evs[0][0].elapsed_time(evs[0][1]) * 1e-3)
        best_out = min(best_out, evs[1][0].elapsed_time(evs[1][1]) * 1e-3)
    out["h2d_duplex"] = round(nb / best_in / 1e9, 1)
    out["d2h_duplex"] = round(nb / best_out / 1e9, 1)
    del h, d, h2, d2
    return out


def run_host_api(api, torch, h32, h64, reps=3):
    """The library's own host-memory path: the synchronous calls given plain
    (pageable) host arrays, which copy the input in (and, for the cumulative
    sums, the output back) inside the call.  Mean wall time per call, after
    one untimed call."""
    res = {}
    x32, x64 = torch.from_numpy(h32), torch.from_numpy(h64)
    o32, o64 = torch.empty_like(x32), torch.empty_like(x64)
    calls = {"sum_f32_1e8": lambda: api.repro_sum(x32, 3), "sum_f64_1e8": lambda: api.repro_sum(x64, 3),
             "cumsum_f32_1e8": lambda: api.repro_cumsum(x32, out=o32, K=3),
             "cumsum_f64_1e8": lambda: api.repro_cumsum(x64, out=o64, K=3)}
    for name, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            fn()
        dt = (time.perf_counter() - t) / reps
        res[name] = {"ms": round(dt * 1e3, 3), "gelem_s": round(N_SUM / dt / 1e9, 3)}
    return res


def run_comparisons(api, torch, x32, x64, A, stream):
    """Context only: non-reproducible and comparison reductions on the same
    inputs (device time per call, CUDA events)."""
    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        # a device-side wait of about 2 ms first, so that every call is
        # queued before the first event: the timed region is device time
        # only, even for calls shorter than their host-side launch
        torch.cuda._sleep(4_000_000)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    A64 = A.double()
    c64k6 = torch.empty_like(x64)
    # inputs that leave the fast paths: magnitudes ascending (the cumulative
    # sum's index settles late), and one value far above the sampled bins (the
    # double sum's index guess misses)
    asc = x64.abs().sort().values * torch.sign(x64)
    outl = x64.clone()
    outl[-1] = 3e200
    AC = A.view(torch.complex64)   # [4096, 2048] complex pairs of the same floats
    st32 = api.state_new(torch.float32, 3)
    st64 = api.state_new(torch.float64, 3)
    r32 = torch.empty(1, dtype=torch.float32, device=x32.device)
    r64 = torch.empty(1, dtype=torch.float64, device=x64.device)

    def chunked(x, st, r, parts=8):
        # the binned-state path: init, eight deposits, finalize
        api.state_init(st, x.dtype, 3, stream)
        for c in torch.chunk(x, parts):
            api.state_deposit(st, c, 3, stream)
        api.state_finalize(st, x.dtype, 3, r, stream)

    out = {}
    for name, fn, n in (
        ("sum_f64_k6_1e8", lambda: api.repro_sum_async(x64, r64, 6), N_SUM),
        ("cumsum_f64_k6_1e8", lambda: api.repro_cumsum(x64, out=c64k6, K=6), N_SUM),
        ("cumsum_f64_k4_1e8", lambda: api.repro_cumsum(x64, out=c64k6, K=4), N_SUM),
        ("adn_cumsum_f64_1e8", lambda: api.repro_cumsum(x64, out=c64k6, K=3), N_SUM),
        ("cumsum_f64_ascending_1e8", lambda: api.repro_cumsum(asc, out=c64k6, K=3), N_SUM),
        ("sum_f64_one_outlier_1e8", lambda: api.repro_sum_async(outl, r64, 3), N_SUM),
        ("state_8_chunks_f32_1e8", lambda: chunked(x32, st32, r32), N_SUM),
        ("state_8_chunks_f64_1e8", lambda: chunked(x64, st64, r64), N_SUM),
        # the hot-path calls again, timed the same way as the others here
        ("adn_sum_f32_1e8", lambda: api.repro_sum_async(x32, r32, 3), N_SUM),
        ("adn_sum_f64_1e8", lambda: api.repro_sum_async(x64, r64, 3), N_SUM),
        ("stable_var_f32_4096x4096", lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False), ROWS * COLS),
        ("naive_sum_f32_1e8", lambda: api.compare_sum(x32, "naive"), N_SUM),
        ("pairwise_sum_f32_1e8", lambda: api.compare_sum(x32, "pairwise"), N_SUM),
        ("torch_sum_f32_1e8", lambda: torch.sum(x32), N_SUM),
        ("naive_sum_f64_1e8", lambda: api.compare_sum(x64, "naive"), N_SUM),
        ("torch_sum_f64_1e8", lambda: torch.sum(x64), N_SUM),
        ("torch_cumsum_f32_1e8", lambda: torch.cumsum(x32, 0), N_SUM),
        ("torch_cumsum_f64_1e8", lambda: torch.cumsum(x64, 0), N_SUM),
        ("twoterm_var_f32_4096x4096", lambda: api.twoterm_var(A, axis=1, ddof=1), ROWS * COLS),
        ("var_variant2_plain_no_twoterm_f32_4096x4096",
         lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False, variant=2), ROWS * COLS),
        ("var_variant3_plain_f32_4096x4096",
         lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False, variant=3), ROWS * COLS),
        ("var_variant4_reference_twosum_f32_4096x4096",
         lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False, variant=4), ROWS * COLS),
        ("var_variant5_no_twoterm_f32_4096x4096",
         lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False, variant=5), ROWS * COLS),
        ("var_variant6_kahan_f32_4096x4096",
         lambda: api.stable_var(A, axis=1, ddof=1, with_mean=False, variant=6), ROWS * COLS),
        ("var_f64_4096x4096", lambda: api.stable_var(A64, axis=1, ddof=1, with_mean=False), ROWS * COLS),
        ("var_c64_4096x2048", lambda: api.stable_var(AC, axis=1, ddof=1, with_mean=False), ROWS * COLS // 2),
        ("torch_var_f32_4096x4096", lambda: torch.var(A, dim=1), ROWS * COLS),
    ):
        ms = timed(fn)
        out[name] = {"ms": round(ms, 4), "gelem_s": round(n / (ms * 1e-3) / 1e9, 2)}
    del asc, outl
    return out


# ------------------------------------------------------------ oracle (CPU)
_SAMPLES = {}


def oracle_samples():
    """Bounded samples of the step's inputs for the CPU oracle: prefixes of
    the same seeded arrays (generated once per process)."""
    if not _SAMPLES:
        from compensated_bit_reproducible_gb300 import inputs
        n = 2_000_000
        _SAMPLES["a32"] = inputs.normal_f32(N_SUM, seed=1)[:n].copy()
        _SAMPLES["a64"] = inputs.wide_f64(N_SUM, seed=2)[:n].copy()
        _SAMPLES["A"] = inputs.offset_rows(ROWS, COLS, seed=3)[:128].copy()
    return _SAMPLES


def oracle_rates(seconds: float):
    """Oracle throughput per hot-path row on bounded samples of the workload
    (single thread).  Returns ({row: elements/s}, {row: sample})."""
    import oracle

    oracle.build()
    smp = oracle_samples()
    a32, a64, A = smp["a32"], smp["a64"], smp["A"]
    budget = max(0.05, seconds / 6.0)
    rates = {}
    samples = {}

    def measure(name, fn, unit_elems, max_reps=64):
        reps, el, t0 = 0, 0, time.perf_counter()
        while reps < max_reps:
            fn()
            reps += 1
            el += unit_elems
            if time.perf_counter() - t0 >= budget:
                break
        dt = time.perf_counter() - t0
        rates[name] = el / dt
        samples[name] = "%d x %d elements" % (reps, unit_elems)

    n = a32.size
    measure("sum_f32_1e8", lambda: oracle.adn_sum(a32, 3, "fp"), n)
    measure("sum_f64_1e8", lambda: oracle.adn_sum(a64, 3, "fp"), n)
    m = 200_000
    measure("cumsum_f32_1e8", lambda: oracle.adn_cumsum(a32[:m], 3), m)
    measure("cumsum_f64_1e8", lambda: oracle.adn_cumsum(a64[:m], 3), m)
    measure("var_f32_4096x4096", lambda: oracle.var_kernel(A, 1, 1), A.size)
    measure("segsum_f32_4096x4096", lambda: oracle.segsum(A[:32], 1, 3), 32 * COLS)
    return rates, samples


def cpu_baseline(seconds: float):
    rates, samples = oracle_rates(seconds)
    t_step = sum(n / rates[name] for name, n, _ in ROWS_SPEC)
    elems = sum(n for _, n, _ in ROWS_SPEC)
    return {"value": round(elems / t_step / 1e9, 6), "unit": "GElements/s", "cores": 1, "kind": "oracle",
            "sample": "per row: " + "; ".join("%s %s" % (k, v) for k, v in samples.items()) +
                      " (step time extrapolated from each row's rate)",
            "rows_gelem_s": {k: round(v / 1e9, 6) for k, v in rates.items()}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    t = []
    for _ in range(args.warmup):
        oracle_rates(args.cpu_seconds / 3)
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rates, samples = oracle_rates(args.cpu_seconds / 3)
        t.append((rates, samples, time.perf_counter() - t0))
    # each step: the oracle's rate on bounded samples -> whole-step rate
    vals = []
    for rates, _, _ in t:
        t_step = sum(n / rates[name] for name, n, _ in ROWS_SPEC)
        vals.append(sum(n for _, n, _ in ROWS_SPEC) / t_step / 1e9)
    v = statistics.mean(vals)
    ms = statistics.mean(x[2] for x in t) * 1e3
    line = {"metric": METRIC, "value": round(v, 6), "unit": "GElements/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32+f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "K": 3},
            "cpu_baseline": {"value": round(v, 6), "unit": "GElements/s", "cores": 1, "kind": "oracle",
                             "sample": "per step, bounded samples of each row: " +
                                       "; ".join("%s %s" % kv for kv in t[-1][1].items())},
            "e2e": {"value": round(v, 6), "unit": "GElements/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ distributed
def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def init_dist(ws, backend=None):
    if ws > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)


SMALL_N_SIZES = (1, 64, 1024, 2048, 2049, 4096, 4097, 16384, 16385)


def run_small_n(reps: int = 201):
    """Call latency at small sizes, measured like the pages' small-N tables:
    three warm-up calls, then `reps` synchronous calls alternating baseline
    and ADN, median host wall time per call (internal allocation and
    synchronisation included).  Sum: `repro_sum` (result on the host) against
    `torch.sum(x).item()`; cumulative sum (K = 3): `repro_cumsum` plus a
    stream synchronisation against `torch.cumsum` plus one.  Prints one JSON
    object (not the benchmark line)."""
    import numpy as np
    import torch
    from compensated_bit_reproducible_gb300 import api, inputs
    dev = torch.device("cuda:0")
    api.validate_environment()
    table = {}
    for name, dt in (("f32", torch.float32), ("f64", torch.float64)):
        for n in SMALL_N_SIZES:
            xh = inputs.normal_f32(n, seed=n) if name == "f32" else inputs.wide_f64(n, seed=n)
            x = torch.from_numpy(xh).to(dev)
            o1 = torch.empty_like(x)
            o2 = torch.empty_like(x)

            def adn_sum():
                api.repro_sum(x, 3)

            def base_sum():
                torch.sum(x).item()

            def adn_cs():
                api.repro_cumsum(x, out=o1, K=3)
                torch.cuda.synchronize()

            def base_cs():
                torch.cumsum(x, 0, out=o2)
                torch.cuda.synchronize()

            row = {}
            for op, (fa, fb) in (("sum", (adn_sum, base_sum)), ("cumsum", (adn_cs, base_cs))):
                for _ in range(3):
                    fa()
                    fb()
                ta, tb = [], []
                for _ in range(reps):
                    t0 = time.perf_counter_ns()
                    fb()
                    tb.append(time.perf_counter_ns() - t0)
                    t0 = time.perf_counter_ns()
                    fa()
                    ta.append(time.perf_counter_ns() - t0)
                a = float(np.median(ta)) / 1e3
                b = float(np.median(tb)) / 1e3
                row[op] = {"adn_us": round(a, 2), "baseline_us": round(b, 2), "adn_over_baseline": round(a / b, 3)}
            table["%s_%d" % (name, n)] = row
    print(json.dumps({"small_n_latency": table, "reps": reps, "K": 3,
                      "baselines": {"sum": "torch.sum(x).item()", "cumsum": "torch.cumsum + synchronize"}}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="chunks per 1e8-element vector in the end-to-end leg")
    ap.add_argument("--k", type=int, default=3,
                    help="fold count of the sum and cumulative-sum rows (for profiling other K; the metric is "
                         "quoted at K = 3)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", default="", help="comma list of rows to run (profiling); default: all")
    ap.add_argument("--skip-extras", action="store_true",
                    help="skip the end-to-end, CPU-baseline and comparison legs (profiling)")
    ap.add_argument("--n", type=int, default=0,
                    help="vector length of the 1e8-element rows (profiling on a smaller case); default 1e8")
    ap.add_argument("--small-n", action="store_true",
                    help="print the small-size call latencies (not the benchmark line) and exit")
    args = ap.parse_args(argv)
    if args.small_n:
        run_small_n()
        return
    if args.n:
        set_vector_length(args.n)
    ws, _, _ = dist_env()
    if args.impl == "reference":
        run_reference(args)
        return
    init_dist(ws)
    run_ours(args)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
