"""Benchmark: DeepSelect row-wise top-k on GB300, effective input HBM bandwidth.

Workload (the DSA-indexer shape): 64 rows x 131,072 bf16 scores, i.i.d. N(0,1), row
stride 131,072 elements (256 KiB, a multiple of 1024 bytes), k=512, B=B2=4096.  One step
is one ds_topk call over the whole batch (every step of the method runs in the CUDA
kernels).  value = rows*N*2 bytes per step / device time per step, in decimal GB/s,
summed over ranks (each rank runs its own copy: rows are independent, weak scaling).

Timing: W warm-up steps, then exactly K steps captured in CUDA graphs and replayed on one
stream, bracketed by a barrier and torch.cuda.synchronize(), timed with CUDA events on
that stream.  Inputs rotate over R device copies whose total exceeds 4x the L2, so each
step reads its input from HBM.  SM clocks are sampled with nvidia-smi during the timed
region.  Each call of `value` reads its input only after the previous kernel on the stream
has completed (the library's default: the input may be that kernel's output).
`input_ready` times the same calls with the option stating that each input was complete
before the previous call started, which lets consecutive calls overlap.

e2e: the same metric through the public API with host buffers: every step copies the
step's input from pinned host memory (on a copy stream, into one of two device buffers,
so the next step's upload overlaps this step's call), runs ds_topk, and reads the
results back; the timed region runs from the first upload to the last read-back.

cold_call: one call alone, the stream idle and the L2 flushed just before it, CUDA events
around that call (median of 5): what a caller pays for a single isolated call.

--impl reference: the oracle (the CPU transcription of the method, oracle/) timed on
this host's cores on a bounded sample of the same workload.

--workload {indexer,sampler,longctx,row65536} and --k run the same measurement on the
method's other workload shapes (sampler: 256 x 129280 fp32 logits; longctx: 4 x 1M bf16;
row65536: one fp32 row); the default, and the headline, is the indexer shape at k=512.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective input HBM GB/s (rows·N·bytes/time) at k=512; % of GB300 HBM peak"
ROWS, N, K_TOP, B, B2 = 64, 131072, 512, 4096, 4096
# --workload: the headline shape (indexer, the default) and the other shapes of the
# method's workloads, each with its rows per GPU, default k and data seed
SHAPES = {
    "indexer": ("indexer_bf16", 64, 512, 2001),
    "sampler": ("sampler_f32", 256, 512, 3001),
    "longctx": ("longctx_bf16", 4, 512, 4001),
    "row65536": ("row65536_f32", 1, 512, 1001),
}


class Shape:
    """One workload of the bench: the synthetic rows, k, and the names the JSON line uses."""

    def __init__(self, name: str, k: int | None, rank: int = 0):
        import synth
        fn, rows, k0, seed = SHAPES[name]
        self.name = name
        self.k = k or k0
        self.w = getattr(synth, fn)(seed=seed + rank, rows=rows)
        w = self.w
        self.rows, self.N, self.stride, self.B, self.B2 = w.rows, w.N, w.stride, w.B, w.B2
        self.bf16 = w.dtype == synth.BF16
        self.dtype = w.dtype
        self.es = 2 if self.bf16 else 4
        self.dname = "bf16" if self.bf16 else "fp32"
        self.step_bytes = self.rows * self.N * self.es
        self.desc = (f"{fn}: {self.rows} rows x {self.N} {self.dname} ({w.desc}), stride {self.stride}, "
                     f"k={self.k}, B={self.B}, B2={self.B2}")
        if name == "indexer" and self.k == K_TOP:
            self.desc = WORKLOAD

    def host_array(self):
        return self.w.x.view(np.int16) if self.bf16 else self.w.x
SEED = 0x5EED
WORKLOAD = f"indexer_bf16: {ROWS} rows x {N} bf16 N(0,1), stride {N}, k={K_TOP}, B={B}, B2={B2}"
FALLBACK_HBM_GBS = 6800.0


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_selection_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def _profile(label: str, sh) -> dict | None:
    """The ncu capture written by capture_profile.py for this kernel, workload and k, if
    one exists (profiles/<kernel>_<workload>_k<k>.json)."""
    path = os.path.join(ROOT, "profiles", f"{label}_{sh.name}_k{sh.k}.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def _traffic_from_profile(label: str, sh):
    """DRAM bytes per launch from the last capture of this kernel on this workload, if the
    kernel sources have not changed since (else None)."""
    prof = _profile(label, sh)
    if not prof or prof.get("source_digest") != _source_digest():
        return None
    return prof.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _cpu_oracle(seconds: float, sh: "Shape", threads: int | None = None):
    """The oracle's DeepSelect transcription over the workload's rows on this host's
    cores, repeated for about `seconds`."""
    import oracle
    w = sh.w
    th = threads or oracle.max_threads()
    oracle.deepselect(w.x[:4], w.dtype, sh.k, sh.B, sh.B2, SEED, N=w.N, threads=th)   # build / warm
    t0 = time.perf_counter()
    runs = 0
    while True:
        oracle.deepselect(w.x, w.dtype, sh.k, sh.B, sh.B2, SEED + runs, N=w.N, threads=th)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = runs * w.input_bytes / el / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": th, "kind": "oracle",
            "sample": f"oracle DeepSelect transcription (C, OpenMP over rows) on the full {sh.rows}x{sh.N} "
                      f"{sh.dname} batch, {runs} runs in {el:.1f} s"}



# The method's other workload shapes, timed in the same run (each its own inputs, rotated
# over device copies totalling more than 4x the L2): (label, synth generator, kwargs, k).
OTHER_SHAPES = [
    ("sampler_f32 256x129280", "sampler_f32", {}, k) for k in (1, 64, 512, 4096)
] + [
    (f"longctx_bf16 4x1048576 {kind}", "longctx_bf16", {"kind": kind}, k)
    for kind in ("iid", "ascending", "levels") for k in (512, 2048)
] + [
    ("row65536_f32 1x65536", "row65536_f32", {}, 512),
    ("huge_f32 1x268435456", "huge_f32", {}, 32),
    ("huge_f32 1x268435456", "huge_f32", {}, 4096),
]


def time_shapes(dev, ds, l2, peak, regions=7, budget_ms=3.0):
    """us per call and effective input GB/s of default ds_topk calls on every other
    workload shape: CUDA graphs of back-to-back calls on one stream, CUDA events around
    each replay, the median of `regions` replays."""
    import torch
    import synth
    out = []
    cache = {}
    stream = torch.cuda.Stream(dev)
    for label, fn, kw, k in OTHER_SHAPES:
        key = (fn, tuple(sorted(kw.items())))
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            w = getattr(synth, fn)(**kw)
            host = torch.from_numpy(w.x.view(np.int16) if w.dtype == synth.BF16 else w.x)
            nbytes = w.rows * w.stride * host.element_size()
            R = max(1, -(-4 * l2 // nbytes))
            x0 = host.to(dev)
            cache[key] = (w, [x0] + [x0.clone() for _ in range(R - 1)])
        w, xs = cache[key]
        R = len(xs)
        es = 2 if w.dtype == synth.BF16 else 4
        vals = torch.empty((w.rows, k), dtype=xs[0].dtype, device=dev)
        idx = torch.empty((w.rows, k), dtype=torch.int32, device=dev)
        plan = ds.ds_get_plan(w.dtype, w.rows, w.N, k, w.B, w.B2)
        step_bytes = w.rows * w.N * es

        def call(i):
            st = ds.ds_topk(xs[i % R].data_ptr(), w.dtype, w.rows, w.N, w.stride, k, w.B, w.B2, SEED,
                            vals.data_ptr(), idx.data_ptr(), stream.cuda_stream)
            if st != 0:
                raise ds.DSError(st)

        with torch.cuda.stream(stream):
            call(0)
        stream.synchronize()
        est_us = max(step_bytes / (peak * 1e3) * 2.0, 5.0)
        G = max(R, min(4000, int(budget_ms * 1e3 / est_us)), 2)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(G):
                    call(i)
            g.replay()
        stream.synchronize()
        ts = []
        for _ in range(regions):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / G)
        status = ds.ds_get_device_status(stream.cuda_stream)
        us = statistics.median(ts)
        gbs = step_bytes / (us * 1e-6) / 1e9
        out.append({"workload": label, "k": k, "B": w.B, "B2": w.B2, "us_per_call": round(us, 3),
                    "us_min": round(min(ts), 3), "us_max": round(max(ts), 3), "value": round(gbs, 1),
                    "unit": "GB/s", "hbm_frac_of_peak": round(gbs / peak, 4),
                    "plan": {"parts": plan["parts"], "cluster": plan["cluster"],
                             "merge_launch": plan["merge_launch"]},
                    "calls_per_graph": G, "input_copies": R, "device_status": status})
        del g
    cache.clear()
    torch.cuda.empty_cache()
    out.append(_time_sampling(dev, ds, l2, peak, regions))
    return out


def _time_sampling(dev, ds, l2, peak, regions, k=512, temperature=1.0):
    """The sampler's use of top-k end to end on the device: ds_topk_sample on the sampler
    shape (sorted top-k, softmax of the k logits, one draw per row from given uniforms)."""
    import torch
    import synth
    w = synth.sampler_f32()
    x0 = torch.from_numpy(w.x).to(dev)
    R = max(1, -(-4 * l2 // x0.numel() // 4))
    xs = [x0] + [x0.clone() for _ in range(R - 1)]
    u = torch.rand(w.rows, generator=torch.Generator().manual_seed(7)).to(dev)
    vals = torch.empty((w.rows, k), dtype=torch.float32, device=dev)
    idx = torch.empty((w.rows, k), dtype=torch.int32, device=dev)
    tok = torch.empty(w.rows, dtype=torch.int32, device=dev)
    prob = torch.empty(w.rows, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def call(i):
        st = ds.ds_topk_sample(xs[i % R].data_ptr(), w.dtype, w.rows, w.N, w.stride, k, w.B, w.B2, SEED, temperature,
                               u.data_ptr(), vals.data_ptr(), idx.data_ptr(), tok.data_ptr(), prob.data_ptr(),
                               stream.cuda_stream)
        if st != 0:
            raise ds.DSError(st)

    with torch.cuda.stream(stream):
        call(0)
    stream.synchronize()
    G = max(R, 40)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                call(i)
        g.replay()
    stream.synchronize()
    ts = []
    for _ in range(regions):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / G)
    us = statistics.median(ts)
    step_bytes = w.rows * w.N * 4
    gbs = step_bytes / (us * 1e-6) / 1e9
    res = {"workload": f"sampler_f32 256x129280 top-k sampling (sorted top-k, softmax, one draw per row; "
                       f"temperature {temperature})", "k": k, "B": w.B, "B2": w.B2, "us_per_call": round(us, 3),
           "us_min": round(min(ts), 3), "us_max": round(max(ts), 3), "value": round(gbs, 1), "unit": "GB/s",
           "hbm_frac_of_peak": round(gbs / peak, 4), "calls_per_graph": G, "input_copies": R,
           "device_status": ds.ds_get_device_status(stream.cuda_stream),
           "launches_per_call": 3}
    del g, xs
    torch.cuda.empty_cache()
    return res

def _cpu_sort(seconds: float, sh: "Shape", threads: int | None = None):
    """The oracle's full stable sort (the definition of the result) over the workload's
    rows on this host's cores, repeated for about `seconds`."""
    import oracle
    w = sh.w
    th = threads or oracle.max_threads()
    bits = w.x.view(np.uint16) if sh.bf16 else w.x.view(np.uint32)
    rows = max(1, min(w.rows, 2 * th))
    sample = np.ascontiguousarray(bits[:rows, :w.N])
    oracle.topk_sort(sample[:1], w.dtype, sh.k, threads=1)   # build / warm
    t0 = time.perf_counter()
    runs = 0
    while True:
        oracle.topk_sort(sample, w.dtype, sh.k, threads=th)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    gbs = runs * rows * w.N * sh.es / el / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": th, "kind": "oracle",
            "sample": f"oracle full stable sort per row (C, OpenMP over rows) on {rows} of the {sh.rows} rows x "
                      f"{sh.N} {sh.dname}, {runs} runs in {el:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm: each step runs the oracle's DeepSelect
    transcription on a sample of the workload (a prefix of its rows, or of one row),
    sized so that the whole run stays within about two minutes of CPU time."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    sh = Shape(args.workload, args.k)
    w = sh.w
    ROWS_, N_ = sh.rows, sh.N
    th = oracle.max_threads()
    steps = max(1, args.steps)
    x = np.ascontiguousarray(w.x[:, :N_])
    t0 = time.perf_counter()
    oracle.deepselect(x, w.dtype, sh.k, sh.B, sh.B2, SEED, threads=th)
    t_full = time.perf_counter() - t0
    budget = 120.0
    rows_ps, n_ps = ROWS_, N_
    if steps * t_full > budget:
        rows_ps = max(1, int(ROWS_ * budget / (steps * t_full)))
        if rows_ps == 1:
            t_row = t_full * th / ROWS_
            n_ps = int(min(N_, max(2 * sh.B, N_ * budget / (steps * max(t_row, 1e-9)))))
    sample = np.ascontiguousarray(x[:rows_ps, :n_ps])
    k_ps = min(sh.k, n_ps)
    use_th = min(th, rows_ps)
    for i in range(args.warmup):
        oracle.deepselect(sample, w.dtype, k_ps, sh.B, sh.B2, SEED + i, threads=use_th)
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.deepselect(sample, w.dtype, k_ps, sh.B, sh.B2, SEED + i, threads=use_th)
    el = time.perf_counter() - t0
    gbs = steps * rows_ps * n_ps * sh.es / el / 1e9
    desc = (f"{rows_ps} row(s) x {n_ps} of the {ROWS_}x{N_} {sh.dname} batch per step, oracle DeepSelect "
            f"transcription")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": el / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": sh.dname, "data": "synthetic",
        "config": {"workload": sh.desc, "sample_per_step": desc},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": use_th, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    import synth
    import top_selection_gb300 as ds
    from top_selection_gb300 import build as tbuild
    from top_selection_gb300.sharding import max_over_ranks, row_range

    ws, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or ws == 1:
        tbuild.build()
    if dist:
        dist.barrier()
    ds.load()

    # weak scaling: rank r owns global rows [lo, hi) of a ROWS*ws batch (its own copy of
    # the workload shape, drawn with its own seed); no data-path collective
    sh = Shape(args.workload, args.k, rank)
    ROWS, N, K_TOP, B, B2, STRIDE, DT = sh.rows, sh.N, sh.k, sh.B, sh.B2, sh.stride, sh.dtype
    vdt = torch.int16 if sh.bf16 else torch.float32
    host = torch.from_numpy(sh.host_array())
    x0 = host.to(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 132 * 1024 * 1024) or 132 * 1024 * 1024
    step_bytes = sh.step_bytes
    R = max(8, -(-4 * l2 // step_bytes))
    xs = [x0.clone() for _ in range(R)]
    outs = [(torch.empty((ROWS, K_TOP), dtype=vdt, device=dev),
             torch.empty((ROWS, K_TOP), dtype=torch.int32, device=dev)) for _ in range(R)]
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    plan = ds.ds_get_plan(DT, ROWS, N, K_TOP, B, B2)
    launches_per_step = 2 if plan["merge_launch"] else 1

    def call(i, ready=False):
        x = xs[i % R]
        v, ix = outs[i % R]
        if ready:
            st = ds.ds_topk_ex(x.data_ptr(), DT, ROWS, N, STRIDE, K_TOP, B, B2, SEED, v.data_ptr(),
                               ix.data_ptr(), input_ready=True, stream=sptr)
        else:
            st = ds.ds_topk(x.data_ptr(), DT, ROWS, N, STRIDE, K_TOP, B, B2, SEED, v.data_ptr(),
                            ix.data_ptr(), sptr)
        if st != 0:
            raise ds.DSError(st)

    # first calls outside capture (attributes, any workspace)
    with torch.cuda.stream(stream):
        for i in range(R):
            call(i)
    stream.synchronize()
    if ds.ds_get_device_status(sptr) != 0:
        raise RuntimeError("device status after first calls")

    G = min(args.graph_len, max(1, args.steps))

    def make_graph(n, ready):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(i, ready)
        return g

    def timed_ms(ready):
        """W warm-up calls, then the timed region -- exactly K calls on the stream, CUDA
        events around it, barrier + synchronize on both sides -- repeated `regions` times.
        Returns the per-region times (ms); the median is reported, with the spread."""
        g_full = make_graph(G, ready)
        rem = args.steps % G
        g_rem = make_graph(rem, ready) if rem else None
        g_warm = make_graph(max(3, args.warmup), ready)
        with torch.cuda.stream(stream):
            g_warm.replay()
        stream.synchronize()
        out = []
        for _ in range(args.regions):
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            if dist:
                dist.barrier()
            torch.cuda.synchronize(dev)
            with torch.cuda.stream(stream):
                ev0.record(stream)
                for _ in range(args.steps // G):
                    g_full.replay()
                if g_rem is not None:
                    g_rem.replay()
                ev1.record(stream)
            torch.cuda.synchronize(dev)
            if dist:
                dist.barrier()
            out.append(ev0.elapsed_time(ev1))
        return out

    sampler = ClockSampler(local if ws > 1 else (dev.index or 0))
    sampler.start()
    # the public call as is: each call reads its input only after the previous kernel
    # on the stream has completed (the input may be that kernel's output)
    ms_regions = timed_ms(False)
    ms = statistics.median(ms_regions)
    # the same calls stating that their inputs were complete before the previous call
    # started (true here: the inputs are written once, before any timed call)
    ms_ready = statistics.median(timed_ms(True))
    clocks = sampler.stop()
    status = ds.ds_get_device_status(sptr)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    t_max = max_over_ranks(ms, device=dev)
    ms_per_step = t_max / args.steps
    value = ws * step_bytes * args.steps / (t_max * 1e-3) / 1e9
    t_ready = max_over_ranks(ms_ready, device=dev)
    input_ready = {"value": round(ws * step_bytes * args.steps / (t_ready * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "ms_per_step": t_ready / args.steps,
                   "call": "ds_topk_ex with options.input_ready = 1 (inputs complete before the previous "
                           "call started, so each call's loads overlap the previous call's tail)"}

    # roofline of the split-row kernel (the one kernel of a step): algorithmic bytes per
    # launch / average launch time
    alg_bytes = step_bytes + ROWS * K_TOP * (sh.es + 4)
    peak, peak_kind = _peak()
    achieved = alg_bytes / (ms / args.steps * 1e-3) / 1e9
    # the split-row kernel runs 256 threads per CTA (also for one part per row), the
    # one-CTA-per-row kernel 288
    kbase = "ds_split_kernel" if plan["threads"] == 256 else "ds_scan_kernel"
    kname = kbase + ("<uint16_t>" if sh.bf16 else "<uint32_t>")
    klabel = kbase + ("_u16" if sh.bf16 else "_u32")
    traffic = _traffic_from_profile(klabel, sh)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "traffic_over_algorithmic": round(traffic / alg_bytes, 4) if traffic else None,
                "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)", "kernel": kname}
    prof = _profile(klabel, sh)
    if prof and prof.get("per_launch"):
        durs = sorted(p["duration_us"] for p in prof["per_launch"] if p.get("duration_us"))
        roofline["ncu_launch_us"] = durs[len(durs) // 2] if durs else None
        roofline["ncu_capture_current"] = prof.get("source_digest") == _source_digest()
        roofline["ncu_note"] = ("ncu times one launch alone with caches flushed; back to back on a stream a "
                                "call's prologue overlaps the previous call, so ms_per_step is shorter")
    if plan["merge_launch"]:
        roofline["note"] = "each step also runs ds_merge_kernel (rows over several clusters)"

    # e2e through the public API with host buffers: every step uploads its input from
    # pinned host memory on a copy stream (two device buffers, so step i+1's upload runs
    # while step i computes), runs topk on the compute stream and reads the results back
    pinned = host.pin_memory()
    xe = [torch.empty_like(x0) for _ in range(2)]
    ve = torch.empty((ROWS, K_TOP), dtype=vdt, device=dev)
    ie = torch.empty((ROWS, K_TOP), dtype=torch.int32, device=dev)
    hv = torch.empty((ROWS, K_TOP), dtype=vdt).pin_memory()
    hi = torch.empty((ROWS, K_TOP), dtype=torch.int32).pin_memory()
    e_steps = args.e2e_steps
    copy_s = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps_run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(copy_s):
                if i >= 2:
                    copy_s.wait_event(ev_used[b])  # the call that read this buffer is done
                xe[b].copy_(pinned, non_blocking=True)
                ev_in[b].record(copy_s)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[b])
                ds.topk(xe[b], K_TOP, B, B2, seed=SEED, N=N, out=(ve, ie), stream=sptr)
                ev_used[b].record(stream)
                hv.copy_(ve, non_blocking=True)
                hi.copy_(ie, non_blocking=True)

    e2e_steps_run(3)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(copy_s)               # the first upload starts the timed region
    stream.wait_event(e0)
    e2e_steps_run(e_steps)
    with torch.cuda.stream(stream):
        e1.record(stream)           # after the last read-back
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(e0.elapsed_time(e1), device=dev)
    # the box's raw pinned host-to-device copy rate for one step's input, alone on the copy
    # stream: the bound of the e2e number above
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(copy_s):
        xe[0].copy_(pinned, non_blocking=True)
        h0.record(copy_s)
        for _ in range(10):
            xe[0].copy_(pinned, non_blocking=True)
        h1.record(copy_s)
    torch.cuda.synchronize(dev)
    h2d_gbs = 10 * pinned.numel() * pinned.element_size() / (h0.elapsed_time(h1) * 1e-3) / 1e9
    e2e = {"value": round(ws * step_bytes * e_steps / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_pinned_copy_gbs": round(h2d_gbs, 1),
           "h2d_bytes_per_step": ROWS * STRIDE * sh.es, "d2h_bytes_per_step": ROWS * K_TOP * (sh.es + 4),
           "steps": e_steps}

    # one call alone: the stream idle, L2 flushed by writing a buffer of twice its size just
    # before, CUDA events around the single call (median of 5) -- launch, prologue and the
    # input's first bytes are all on this clock, with no previous call to overlap
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    cold = []
    for i in range(5):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.fill_(i)
            c0.record(stream)
            call(i)
            c1.record(stream)
        stream.synchronize()
        cold.append(c0.elapsed_time(c1))
    cold_ms = max_over_ranks(statistics.median(cold), device=dev)
    del flush
    cold_call = {"us": round(cold_ms * 1e3, 3), "value": round(ws * step_bytes / (cold_ms * 1e-3) / 1e9, 2),
                 "unit": "GB/s", "call": "one ds_topk call alone after an L2 flush, CUDA events around it "
                                         "(median of 5)"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    shapes = time_shapes(dev, ds, l2, peak, regions=args.regions // 2 + 1) if (ws == 1 and args.shapes) else None
    cpu = _cpu_oracle(args.cpu_seconds, sh) if (ws == 1 and args.cpu_seconds > 0) else None
    cpu_sort = _cpu_sort(args.cpu_seconds, sh) if (ws == 1 and args.cpu_seconds > 0) else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": sh.dname, "data": "synthetic",
        "config": {"workload": sh.desc, "global_batch_rows": ROWS * ws, "parallelism": f"rows replicated x{ws}",
                   "l2": f"inputs rotated over {R} device copies ({R * step_bytes / 1e6:.0f} MB > 4x L2 "
                         f"{l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA graphs of {G} calls, CUDA events on the launching stream; the "
                             f"{args.steps}-call timed region is run {args.regions} times, median reported",
                   "plan": plan},
        "timing_spread": {"regions": len(ms_regions), "region_ms_median": ms,
                          "region_ms_min": min(ms_regions), "region_ms_max": max(ms_regions),
                          "us_per_step_x_sm_ghz": (round(ms / args.steps * 1e3 * clocks["sm_mhz"] / 1e3, 4)
                                                   if clocks.get("sm_mhz") else None)},
        "hbm_frac_of_peak": round(value / ws / peak, 4),
        "roofline": roofline,
        "input_ready": input_ready,
        "cold_call": cold_call,
        "cpu_baseline": cpu,
        "cpu_baseline_full_sort": cpu_sort,
        "e2e": e2e,
        "shapes": shapes,
        "clocks": clocks,
        "gpu_launches": args.steps * launches_per_step,
        "device": torch.cuda.get_device_name(dev),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--regions", type=int, default=15,
                    help="the K-step timed region is repeated this many times; the median is reported")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--graph-len", type=int, default=2000)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", choices=sorted(SHAPES), default="indexer",
                    help="the indexer shape is the headline; the others are the method's other workloads")
    ap.add_argument("--k", type=int, default=0, help="k (default: the workload's)")
    ap.add_argument("--no-shapes", dest="shapes", action="store_false",
                    help="skip timing the other workload shapes (reported under 'shapes')")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
