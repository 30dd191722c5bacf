"""Benchmark of the strided tile layout copy on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..8] [--elem-bytes W] [--kernel auto|vec_copy|
                    warp_permute|warp_shuffle|tile_transpose|smem_transpose|tma_copy]
                    [--loop "[(extent, thread_stride, slot_stride), ...]"]
                    [--in-place | --unit-run]
                    [--graph] [--copy-ceiling] [--e2e-steps E] [--no-cpu-baseline]
                    [--flush read|write] [--no-per-config] [--per-config-only 3,4:1,...]

A step is one lc_layout_copy over the whole workload (one kernel launch);
inputs are synthetic, seeded and resident in HBM; workloads smaller than
twice the L2 get an L2 flush between steps (by default a read of twice the
L2 size, so no dirty line of the flush drains into the timed launch; --flush
write fills the buffer instead).  Prints ONE JSON line on rank 0.  The default
run (workload 2 on one GPU) adds `per_config`: workloads 1, 3, 4 (1- to
16-byte words) and 5 measured the same way, each with its kernel, GB/s,
roofline fraction, a 4096-point oracle check and its clocks.
The default workload is the scale-factor transpose batch: 2^20 tiles of
(pipe=2, high=1, 4, 32) fp32, strides (128,128,32,1) -> (128,128,1,4).
Workloads: 1 one 32x32 fp32 transpose; 2 the default; 3 a 16384^2 bf16
transpose; 4 an 8192^2 transpose of W-byte words; 5 a (256,32,128,128) bf16
permute (0,2,1,3); 6 an 8191 x 8193 transpose of W-byte words (strides off
the 16-byte grid); 7 the window sum of three over 2^28 float32 outputs;
8 workload 5's permute as 256 tiles moved under an explicit loop layout
(lc_layout_copy_loop; --loop replaces the workload's override).  With
workload 2, --in-place permutes the buffer in place (destination = source,
the aliasing the warp permute allows) and --unit-run moves the same units
through lc_warp_unit_run (the op between shared-memory buffers, staged from
and back to HBM).

--impl reference times the CPU oracle (the plain C word loop) on the host
cores over a bounded sample of the same workload; it never touches a GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "effective GB/s (read+write) and % of GB300 HBM peak per layout permute"
UNIT = "GB/s"
DEFAULT_WORKLOAD = 2
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    p.add_argument("--elem-bytes", type=int, default=None)
    p.add_argument("--kernel", default="auto")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--copy-ceiling", action="store_true",
                   help="also time a plain device copy of the same byte count (same L2 policy)")
    p.add_argument("--graph", action="store_true",
                   help="replay the K timed launches from one CUDA graph (launch-bound copies)")
    p.add_argument("--loop", default=None,
                   help="loop layout for workload 8, a Python literal list of (extent, thread_stride, slot_stride)")
    p.add_argument("--in-place", action="store_true",
                   help="workload 2 permuted in place (destination = source buffer)")
    p.add_argument("--unit-run", action="store_true",
                   help="workload 2's units through lc_warp_unit_run (shared-memory buffers)")
    p.add_argument("--flush", default="read", choices=["read", "write"],
                   help="how L2 is evicted between timed launches of workloads under twice its size")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the other workloads' measurements added to the default line")
    p.add_argument("--per-config-only", default=None,
                   help="comma list of workloads (4:W for workload 4 with W-byte words) for per_config")
    p.add_argument("--n-tiles", type=int, default=None,
                   help="override the tile count (a smaller case of the same kernel, e.g. for ncu)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# helpers shared with the tests (rank aggregation, peaks, workload description)
# ---------------------------------------------------------------------------

def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def workload_bytes(cfg) -> int:
    """Algorithmic bytes of one step: every logical word read once, written once."""
    return 2 * workloads.logical_elems(cfg) * cfg["elem_bytes"]


def describe(cfg) -> str:
    s, d = cfg["src"], cfg["dst"]
    return "%s: %d tile(s) of shape %s, %d-byte words, strides %s -> %s" % (
        cfg["name"], cfg["n_tiles"], s["shape"], cfg["elem_bytes"], s["stride"], d["stride"])


def _code_only(text: bytes) -> bytes:
    """Source text without comments, runs of spaces collapsed and blank lines
    dropped (line breaks kept for the preprocessor): a comment edit leaves a
    kernel's hash alone.  No string literal in the hashed sources holds a
    comment marker."""
    s = re.sub(r"/\*.*?\*/", " ", text.decode(), flags=re.S)
    s = re.sub(r"//[^\n]*", "", s)
    lines = (re.sub(r"[ \t]+", " ", ln).strip() for ln in s.split("\n"))
    return "\n".join(ln for ln in lines if ln).encode()


def kernel_sources_sha(kernel_name: str) -> str:
    """Hash of the code (comments excluded) of a kernel class's sources."""
    warp = ["k_warp.cu", "k_warp.cuh"] + ["k_warp_w%d.cu" % w for w in (1, 2, 4, 8, 16)]
    files = {"warp_permute": warp, "warp_unit_shared": warp, "tile_transpose": ["k_tile.cu", "bulk_store.cuh"],
             "vec_copy": ["k_vec.cu"], "smem_transpose": ["k_smem.cu"],
             "tma_copy": ["k_tma_copy.cu", "bulk_store.cuh"], "window_sum": ["k_stencil.cu"],
             "loop_copy": ["k_loop.cu"], "warp_shuffle": ["k_shuffle.cu"],
             "smem_staged": ["k_staged.cu"]}.get(kernel_name, [])
    paths = [os.path.join(ROOT, "movement_primitives_gb300", "csrc", f) for f in files + ["ptx.cuh", "device_common.cuh"]]
    if kernel_name in ("warp_permute", "warp_unit_shared", "smem_staged"):  # device functions in the public header
        paths.append(os.path.join(ROOT, "include", "layout_copy_device.cuh"))
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as fh:
            h.update(_code_only(fh.read()))
    return h.hexdigest()[:16]


def profiled_traffic(kernel_name: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel_name, workload_name))
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_per_launch_bytes:\s*(\d+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_sources_sha(kernel_name):
        return None
    return int(m.group(1))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", self.gpu_id, "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def snapshot(self):
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=" + self.FIELDS,
                                  "--format=csv,noheader,nounits", "-i", self.gpu_id],
                                 capture_output=True, text=True, timeout=10).stdout
            self.lines += [l.strip() for l in out.splitlines() if l.strip()]
        except (OSError, subprocess.TimeoutExpired):
            pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        sm, smax, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(self.REASONS, parts[3:]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[device_index] if vis else str(device_index)


class L2Flush:
    """Evicts L2 between timed launches, outside their event pairs.

    ``read`` (the default) reduces a buffer of twice the L2 size to one
    8-byte value: L2 is left holding clean lines of that buffer, so the next
    timed launch neither hits its own previous lines nor pays for the flush's
    write-back.  ``write`` fills the buffer instead, which leaves L2 full of
    dirty lines whose write-back overlaps the next launch.
    """

    def __init__(self, dev, kind: str = "read"):
        import torch
        self.kind = kind
        self.buf = torch.zeros(2 * workloads.HBM_L2_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self, k: int) -> None:
        if self.kind == "read":
            self.buf.sum()
        else:
            self.buf.fill_(k & 0xFF)

    def describe(self) -> str:
        mib = 2 * workloads.HBM_L2_BYTES >> 20
        if self.kind == "read":
            return "L2 flushed between steps by reading a %d MiB buffer (a reduction to 8 bytes) " \
                   "outside the timed launches; value from per-launch CUDA events" % mib
        return "L2 flushed between steps by writing a %d MiB buffer outside the timed launches; " \
               "value from per-launch CUDA events" % mib


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sampled(cfg, fraction: float):
    """The same workload restricted to a leading fraction of its tiles, or of
    its outermost non-unit mode when it has a single tile."""
    c = dict(cfg)
    if cfg["n_tiles"] > 1:
        c["n_tiles"] = max(1, int(cfg["n_tiles"] * fraction))
        return c
    shape = list(cfg["src"]["shape"])
    k = next(i for i, e in enumerate(shape) if e > 1)
    shape[k] = max(1, int(shape[k] * fraction))
    c["src"] = dict(cfg["src"], shape=tuple(shape))
    c["dst"] = dict(cfg["dst"], shape=tuple(shape))
    return c


def run_oracle(cfg, src_np, dst_np, cores: int) -> float:
    """One oracle pass over `cfg` split across `cores` threads; returns seconds."""
    import oracle
    tasks = []
    if cfg["n_tiles"] >= cores:
        step = -(-cfg["n_tiles"] // cores)
        for b in range(0, cfg["n_tiles"], step):
            tasks.append((cfg, (b, min(cfg["n_tiles"], b + step))))
    else:
        # split the outermost non-unit mode into slabs, each its own copy
        shape = list(cfg["src"]["shape"])
        k = next((i for i, e in enumerate(shape) if e > 1), 0)
        n = shape[k]
        step = max(1, -(-n // cores))
        for b in range(0, n, step):
            sub = dict(cfg)
            sh = list(shape)
            sh[k] = min(n, b + step) - b
            sub["src"] = dict(cfg["src"], shape=tuple(sh),
                              offset=cfg["src"]["offset"] + b * cfg["src"]["stride"][k],
                              tile_stride=cfg["src"]["tile_stride"] or workloads.footprint_elems(cfg["src"], 1))
            sub["dst"] = dict(cfg["dst"], shape=tuple(sh),
                              offset=cfg["dst"]["offset"] + b * cfg["dst"]["stride"][k],
                              tile_stride=cfg["dst"]["tile_stride"] or workloads.footprint_elems(cfg["dst"], 1))
            tasks.append((sub, None))

    def one(task):
        c, rng = task
        oracle.copy(src_np, c["src"], dst_np, c["dst"], c["elem_bytes"], c["n_tiles"], tile_range=rng)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(one, tasks))
    return time.perf_counter() - t0


def calibrate(cfg, src_np, dst_np, cores, seconds):
    """Sample for about `seconds` of oracle work here: (fraction of the
    workload, passes over it).  Probes with growing samples until one takes a
    measurable time; a workload that the host moves faster than that is
    repeated whole."""
    frac = 1.0 / 4096
    while True:
        t = run_oracle(sampled(cfg, frac), src_np, dst_np, cores)
        if t >= 0.25 or frac >= 1.0:
            break
        frac = min(1.0, frac * 8)
    want = frac * seconds / max(t, 1e-6)
    if want <= 1.0:
        return want, 1
    return 1.0, max(1, min(200, int(round(want))))


def cpu_baseline(cfg, src_np, seconds: float):
    """The oracle, as it stands, on this host's cores over a bounded sample."""
    import numpy as np
    cores = host_cores()
    dst = np.empty(workloads.footprint_elems(cfg["dst"], cfg["n_tiles"]) * cfg["elem_bytes"], np.uint8)
    frac, passes = calibrate(cfg, src_np, dst, cores, seconds)
    sample = sampled(cfg, frac)
    t = sum(run_oracle(sample, src_np, dst, cores) for _ in range(passes))
    gbs = passes * workload_bytes(sample) / t / 1e9
    # the same oracle on one thread, over a sample of a quarter of the time
    frac1, passes1 = calibrate(cfg, src_np, dst, 1, seconds / 4)
    sample1 = sampled(cfg, frac1)
    t1 = sum(run_oracle(sample1, src_np, dst, 1) for _ in range(passes1))
    gbs1 = passes1 * workload_bytes(sample1) / t1 / 1e9
    return dict(value=round(gbs, 3), unit=UNIT, cores=cores, kind="oracle",
                sample="%d pass(es) over %.4f of the workload (%d logical words each), %.2f s on %d threads"
                       % (passes, frac, workloads.logical_elems(sample), t, cores),
                single_thread={"value": round(gbs1, 3), "unit": UNIT,
                               "sample": "%d pass(es) over %.4f of the workload, %.2f s on 1 thread"
                                         % (passes1, frac1, t1)})


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    import numpy as np
    cfg = workloads.config(args.workload, args.elem_bytes)
    src = workloads.make_src(cfg).numpy()
    dst = np.empty(workloads.footprint_elems(cfg["dst"], cfg["n_tiles"]) * cfg["elem_bytes"], np.uint8)
    cores = host_cores()
    budget = 120.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    frac, _ = calibrate(cfg, src, dst, cores, budget)
    sample = sampled(cfg, frac)
    for _ in range(args.warmup):
        run_oracle(sample, src, dst, cores)
    times = [run_oracle(sample, src, dst, cores) for _ in range(args.steps)]
    total = sum(times)
    value = workload_bytes(sample) * args.steps / total / 1e9
    desc = "%.5f of the workload per step (%d logical words) on %d threads" % (
        frac, workloads.logical_elems(sample), cores)
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(cfg), "data": "synthetic",
            "config": {"workload": describe(cfg), "sample": desc},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def dtype_name(cfg) -> str:
    return {"uniform_f32": "f32", "normal_bf16": "bf16"}.get(
        cfg["kind"], {1: "u8", 2: "u16", 4: "u32", 8: "u64", 16: "u128"}[cfg["elem_bytes"]])


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    __graft_entry__.build()
    import movement_primitives_gb300 as lc

    cfg = workloads.config(args.workload, args.elem_bytes)
    if args.n_tiles:
        cfg["n_tiles"] = args.n_tiles
    mode = "in_place" if args.in_place else "unit_run" if args.unit_run else None
    check_args(args)
    if mode:
        cfg["name"] += "_" + mode
        args.e2e_steps = 0  # the host-buffer entry point has no such variant
    step_bytes = workload_bytes(cfg)
    src_h = workloads.make_src(cfg)
    src = src_h.to(dev)
    dst = workloads.make_dst(cfg, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    loop = cfg.get("loop")
    unit = None
    if mode == "unit_run":
        # workload 2's tiles are two (4, 32) units back to back on both sides
        unit, _info = lc.warp_unit_plan(dict(shape=(4, 32), stride=(32, 1)), dict(shape=(4, 32), stride=(1, 4)),
                                        cfg["elem_bytes"])
        n_units = cfg["n_tiles"] * 2
    if loop is not None and args.loop:
        import ast
        loop = [tuple(m) for m in ast.literal_eval(args.loop)]
    if loop is not None:
        kernel_name = "loop_copy"
    elif unit is not None:
        kernel_name = "warp_unit_shared"
    else:
        kernel_name = lc.plan(cfg["src"], cfg["dst"], cfg["elem_bytes"], cfg["n_tiles"], args.kernel)["kernel_name"]

    def launch(stream_handle, out=None):
        out = dst if out is None else out
        if unit is not None:
            lc.warp_unit_run(src, out, unit, cfg["elem_bytes"], n_units, stream=stream_handle)
        elif mode == "in_place":
            lc.layout_copy_ptr(out.data_ptr(), cfg["src"], out.data_ptr(), cfg["dst"], cfg["elem_bytes"],
                               cfg["n_tiles"], kernel=args.kernel, stream=stream_handle)
        elif loop is not None:
            lc.layout_copy_loop_ptr(src.data_ptr(), cfg["src"], dst.data_ptr(), cfg["dst"], cfg["elem_bytes"],
                                    loop, cfg["n_tiles"], 0, stream_handle)
        else:
            lc.layout_copy_ptr(src.data_ptr(), cfg["src"], out.data_ptr(), cfg["dst"], cfg["elem_bytes"],
                               cfg["n_tiles"], kernel=args.kernel, stream=stream_handle)

    if mode == "in_place":
        # one in-place step on a copy of the source is checked below; the
        # timed steps keep permuting the same buffer (same work every step)
        del dst
        dst = src.clone()
        launch(sh, dst)
        torch.cuda.synchronize()
        checked = dst.clone()
        dst = src

    def step():
        launch(sh)

    for _ in range(max(3, args.warmup)):
        step()
    st, detail = lc.last_device_error(sh)
    if st != 0:
        raise RuntimeError("device error word %#x during warm-up" % detail)
    # spot check against the oracle's offsets (the tests do the full parity)
    import oracle
    n = workloads.logical_elems(cfg)
    pts = np.random.default_rng(0).integers(0, n, 4096)
    so, do = oracle.offsets_of(cfg["src"], cfg["dst"], cfg["n_tiles"], pts)
    w = cfg["elem_bytes"]
    sv = src_h.to(dev).view(-1, w) if mode == "in_place" else src.view(-1, w)
    dv = (checked if mode == "in_place" else dst).view(-1, w)
    if not torch.equal(sv[torch.from_numpy(so).to(dev)], dv[torch.from_numpy(do).to(dev)]):
        raise RuntimeError("spot check against the oracle failed")

    sampler = ClockSampler(gpu_id_for(dev.index)) if rank == 0 else None
    per_side = step_bytes // 2
    flush = per_side < 2 * workloads.HBM_L2_BYTES and not args.graph
    flusher = L2Flush(dev, args.flush) if flush else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = None
    if args.graph:
        cap = torch.cuda.Stream()  # graphs are captured on a side stream
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(args.steps):
                launch(cap.cuda_stream)
        stream.wait_stream(cap)
        graph.replay()
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(args.steps):
            if flush:
                flusher(k)  # evicts the previous step's lines from L2
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
    t1.record(stream)
    if sampler:
        sampler.snapshot()  # while the queued launches run
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    st, detail = lc.last_device_error(sh)
    if st != 0:
        raise RuntimeError("device error word %#x in the timed region" % detail)
    launch_median_ms = None
    if graph is not None:
        launch_ms = t0.elapsed_time(t1) / args.steps
        timed_ms = t0.elapsed_time(t1)
    else:
        launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        launch_median_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        # with L2 flushes in between, the job time is the launches' own time
        timed_ms = sum(a.elapsed_time(b) for a, b in ev) if flush else t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(timed_ms, dev)

    # end to end through the C-ABI host-buffer call: pinned host source in,
    # pinned host destination out; uploads, permutes and downloads pipelined
    # by the library over chunks of tiles, all inside the timed region
    e2e = None
    if args.e2e_steps > 0 and loop is not None:
        # no host-buffer form of the loop copy: pinned upload, the copy, pinned
        # download, in order on the stream, every step
        src_pin = src_h.pin_memory()
        dst_pin = torch.empty(dst.numel(), dtype=torch.uint8).pin_memory()
        for it in range(args.e2e_steps + 2):
            if it == 2:
                barrier()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            src.copy_(src_pin, non_blocking=True)
            launch(sh)
            dst_pin.copy_(dst, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev)
        if not torch.equal(dst_pin[:1 << 20], dst[:1 << 20].cpu()):
            raise RuntimeError("end-to-end result differs from the device result")
        e2e = {"value": round(world * step_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": src.numel() * src.element_size(),
               "d2h_bytes_per_step": dst.numel() * dst.element_size(),
               "path": "pinned upload, lc_layout_copy_loop, pinned download (one stream, not pipelined)"}
    elif args.e2e_steps > 0:
        # two public host-buffer paths, each timed over the same steps; the
        # line reports the faster and lists both
        src_pin = src_h.pin_memory()
        dst_pin = torch.empty(dst.numel(), dtype=torch.uint8).pin_memory()
        staging = torch.empty(max(256, lc.host_staging_bytes(cfg["src"], cfg["dst"], cfg["elem_bytes"],
                                                             cfg["n_tiles"])), dtype=torch.uint8, device=dev)

        def staged():
            lc.layout_copy_host(src_pin, cfg["src"], dst_pin, cfg["dst"], n_tiles=cfg["n_tiles"],
                                elem_bytes=cfg["elem_bytes"], staging=staging, stream=stream)

        def mapped():
            lc.layout_copy_mapped(src_pin, cfg["src"], dst_pin, cfg["dst"], n_tiles=cfg["n_tiles"],
                                  elem_bytes=cfg["elem_bytes"], stream=stream)

        paths = []
        for name, call in (("lc_layout_copy_host (pinned host buffers, staged on the device, transfers and "
                            "permutes pipelined over tile chunks)", staged),
                           ("lc_layout_copy_mapped (pinned host buffers read and written by the copy kernels "
                            "over the CPU-GPU link, no staging)", mapped)):
            dst_pin.fill_(0)
            for it in range(args.e2e_steps + 2):
                if it == 2:
                    barrier()
                    torch.cuda.synchronize()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev)
            if not torch.equal(dst_pin[:1 << 20], dst[:1 << 20].cpu()) or \
                    not torch.equal(dst_pin[-(1 << 20):], dst[-(1 << 20):].cpu()):
                raise RuntimeError("end-to-end result differs from the device result (%s)" % name)
            paths.append({"path": name, "value": round(world * step_bytes / (e2e_ms / 1e3) / 1e9, 2)})
        best = max(paths, key=lambda x: x["value"])
        e2e = {"value": best["value"], "unit": UNIT,
               "h2d_bytes_per_step": src.numel() * src.element_size(),
               "d2h_bytes_per_step": dst.numel() * dst.element_size(),
               "path": best["path"], "paths": paths}
        del staging

    copy_ceiling = None
    if args.copy_ceiling:
        # a contiguous device-to-device copy of the same bytes: the practical
        # ceiling for a workload of this size (launch and ramp costs included)
        nbytes = step_bytes // 2
        a_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        b_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(5):
            b_buf.copy_(a_buf)
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(args.steps, 200))]
        torch.cuda.synchronize()
        for k, (e0c, e1c) in enumerate(cev):
            if flush:
                flusher(k)
            e0c.record(stream)
            b_buf.copy_(a_buf)
            e1c.record(stream)
        torch.cuda.synchronize()
        cms = statistics.mean(x.elapsed_time(y) for x, y in cev)
        copy_ceiling = round(step_bytes / (cms / 1e3) / 1e9, 2)
        del a_buf, b_buf

    peak, peak_kind = measured_peak()
    achieved = step_bytes / (launch_ms / 1e3) / 1e9
    traffic = profiled_traffic(kernel_name, cfg["name"])
    per_config = None
    if (rank == 0 and world == 1 and not args.no_per_config and mode is None and loop is None
            and args.workload == DEFAULT_WORKLOAD and not args.n_tiles and args.kernel == "auto"):
        per_config = {}
        for c_id, c_w in parse_per_config(args.per_config_only):
            other = workloads.config(c_id, c_w)
            per_config[other["name"]] = measure_workload(other, dev, lc, stream, args.flush, peak)
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline(cfg, src_h.numpy(), args.cpu_seconds)
        value = world * step_bytes * args.steps / (elapsed_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 5),
            "launch_ms_median": round(launch_median_ms, 5) if launch_median_ms is not None else None,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(cfg), "data": "synthetic",
            "config": {"workload": describe(cfg), "kernel": kernel_name,
                       "loop_layout": loop, "mode": mode,
                       "bytes_per_step": step_bytes,
                       "l2": (flusher.describe() if flush
                              else "inputs larger than L2 (%d MiB per side), no flush" % (step_bytes // 2 >> 20)),
                       "timing": "one CUDA graph of K launches" if args.graph else "K launches from the host",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                         if peak_kind == "measured" else peak_kind},
            "clocks": clocks,
            "gpu_launches": args.steps,
            "copy_ceiling_gbs": copy_ceiling,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# The other workloads of the metric ("per layout permute"), measured after the
# default one and reported beside it: (workload, element bytes).
PER_CONFIG = [(1, None), (3, None), (4, 1), (4, 2), (4, 4), (4, 8), (4, 16), (5, None)]


def parse_per_config(text):
    if not text:
        return PER_CONFIG
    out = []
    for item in text.split(","):
        cfg, _, w = item.partition(":")
        out.append((int(cfg), int(w) if w else None))
    return out


def measure_workload(cfg, dev, lc, stream, flush_kind, peak, min_ms=250.0):
    """One workload at full size: planner's kernel, per-launch CUDA-event
    times (L2 evicted between launches when a side is under twice its size),
    a 4096-point check of the result against the oracle's offsets, and the
    clocks seen while the launches ran."""
    import numpy as np
    import torch

    import oracle
    src_h = workloads.make_src(cfg)
    src = src_h.to(dev)
    del src_h
    dst = workloads.make_dst(cfg, device=dev)
    sh = stream.cuda_stream
    w, nt = cfg["elem_bytes"], cfg["n_tiles"]
    kernel_name = lc.plan(cfg["src"], cfg["dst"], w, nt)["kernel_name"]

    def launch():
        lc.layout_copy_ptr(src.data_ptr(), cfg["src"], dst.data_ptr(), cfg["dst"], w, nt, stream=sh)

    for _ in range(3):
        launch()
    st, detail = lc.last_device_error(sh)
    if st != 0:
        raise RuntimeError("device error word %#x during warm-up of %s" % (detail, cfg["name"]))
    n = workloads.logical_elems(cfg)
    pts = np.random.default_rng(cfg["cfg"]).integers(0, n, 4096)
    so, do = oracle.offsets_of(cfg["src"], cfg["dst"], nt, pts)
    sv, dv = src.view(-1, w), dst.view(-1, w)
    checked = torch.equal(sv[torch.from_numpy(so).to(dev)], dv[torch.from_numpy(do).to(dev)])
    if not checked:
        raise RuntimeError("spot check against the oracle failed on %s" % cfg["name"])

    step_bytes = workload_bytes(cfg)
    flush = step_bytes // 2 < 2 * workloads.HBM_L2_BYTES
    flushers = {k: L2Flush(dev, k) for k in (("read", "write") if flush else ())}

    def timed(steps, flusher, op=launch):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for k in range(steps):
            if flusher is not None:
                flusher(k)
            ev[k][0].record(stream)
            op()
            ev[k][1].record(stream)
        return ev

    probe = timed(5, flushers.get(flush_kind))
    torch.cuda.synchronize()
    est = statistics.median(a.elapsed_time(b) for a, b in probe)
    steps = int(min(2000, max(50, min_ms / max(est, 1e-3))))
    sampler = ClockSampler(gpu_id_for(dev.index))
    sampler.start()
    ev = timed(steps, flushers.get(flush_kind))
    sampler.snapshot()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    other = None
    if flush:
        other_kind = "write" if flush_kind == "read" else "read"
        ev2 = timed(min(steps, 200), flushers[other_kind])
        torch.cuda.synchronize()
        other = {"flush": other_kind,
                 "gbs": round(step_bytes / (statistics.mean(a.elapsed_time(b) for a, b in ev2) / 1e3) / 1e9, 2)}
    st, detail = lc.last_device_error(sh)
    if st != 0:
        raise RuntimeError("device error word %#x while timing %s" % (detail, cfg["name"]))
    mean_ms = statistics.mean(times)
    gbs = step_bytes / (mean_ms / 1e3) / 1e9
    out = {"workload": describe(cfg), "kernel": kernel_name, "bytes_per_launch": step_bytes,
           "launches": steps, "launch_us_mean": round(1e3 * mean_ms, 3),
           "launch_us_median": round(1e3 * statistics.median(times), 3),
           "gbs": round(gbs, 2), "pct_of_peak": round(100.0 * gbs / peak, 2),
           "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "traffic": profiled_traffic(kernel_name, cfg["name"])},
           "l2": flushers[flush_kind].describe() if flush
           else "inputs larger than L2 (%d MiB per side), no flush" % (step_bytes // 2 >> 20),
           "other_flush": other,
           "spot_check": "4096 random logical points equal at the oracle's offsets",
           "clocks": clocks}
    if step_bytes < (1 << 20):
        # latency-bound: the floor any launch pays under the same protocol
        # (flush, events), from the smallest device operation there is
        tiny = torch.zeros(1, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            fl = timed(min(steps, 500), flushers.get(flush_kind), op=lambda: tiny.fill_(1))
        torch.cuda.synchronize()
        floor_us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in fl)
        out["latency"] = {"launch_floor_us": round(floor_us, 3),
                          "floor_op": "a one-element device fill, launched and timed the same way",
                          "kernel_over_floor_us": round(out["launch_us_median"] - floor_us, 3)}
    del src, dst, flushers
    torch.cuda.empty_cache()
    return out


def run_window_sum(args):
    """Workload 7: b[i] = a[i] + a[i+1] + a[i+2] over 2^28 float32 outputs."""
    import numpy as np
    import torch

    import __graft_entry__
    from oracle import stencil
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    import movement_primitives_gb300 as lc
    cfg = workloads.config(7)
    n, win = cfg["n_out"], cfg["window"]
    a_h = workloads.make_bytes(n + win - 1, 4, cfg["kind"], cfg["seed"]).view(torch.float32)
    if args.impl == "reference":
        cores = host_cores()
        m = min(n, 1 << 26)
        t0 = time.perf_counter()
        passes = 0
        while time.perf_counter() - t0 < args.cpu_seconds / 2 or passes == 0:
            stencil.window_sum_f32(a_h.numpy()[:m + win - 1], m, win)
            passes += 1
        t = time.perf_counter() - t0
        value = passes * (2 * m + win - 1) * 4 / t / 1e9
        print(json.dumps({"metric": METRIC, "value": round(value, 3), "unit": UNIT, "impl": "reference",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                          "data": "synthetic", "config": {"workload": cfg["name"]},
                          "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": "%d pass(es) over %d outputs" % (passes, m)},
                          "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    a = a_h.to(dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    step_bytes = (2 * n + win - 1) * 4
    for _ in range(max(3, args.warmup)):
        lc.window_sum(a, out, win, stream=stream)
    m = 1 << 20
    if not np.array_equal(out[:m].cpu().numpy(), stencil.window_sum_f32(a_h.numpy()[:m + win - 1], m, win)):
        raise RuntimeError("spot check against the oracle failed")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(gpu_id_for(0))
    torch.cuda.synchronize()
    sampler.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        lc.window_sum(a, out, win, stream=stream)
        ev[k][1].record(stream)
    t1.record(stream)
    sampler.snapshot()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    elapsed = t0.elapsed_time(t1)
    launch_ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    peak, peak_kind = measured_peak()
    value = step_bytes * args.steps / (elapsed / 1e3) / 1e9
    achieved = step_bytes / (launch_ms / 1e3) / 1e9
    e2e = None
    if args.e2e_steps > 0:
        a_pin, o_pin = a_h.pin_memory(), torch.empty(n, dtype=torch.float32).pin_memory()
        for it in range(args.e2e_steps + 1):
            if it == 1:
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            a.copy_(a_pin, non_blocking=True)
            lc.window_sum(a, out, win, stream=stream)
            o_pin.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        e2e = {"value": round(step_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": (n + win - 1) * 4, "d2h_bytes_per_step": n * 4,
               "path": "pinned copies around lc_window_sum_f32 on one stream"}
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "%s: %d outputs, window %d" % (cfg["name"], n, win), "kernel": "window_sum",
                       "bytes_per_step": step_bytes, "l2": "inputs larger than L2, no flush"},
            "pct_of_peak": round(100.0 * value / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": profiled_traffic("window_sum", cfg["name"]),
                         "peak_kind": peak_kind},
            "clocks": clocks, "gpu_launches": args.steps, "e2e": e2e, "cpu_baseline": None}
    print(json.dumps(line), flush=True)
    return 0


def check_args(args) -> None:
    """Refuses flag combinations that name no workload."""
    if (args.in_place or args.unit_run) and (args.workload != 2 or (args.in_place and args.unit_run)):
        raise SystemExit("--in-place or --unit-run (one of them) applies to workload 2")
    if args.loop and args.workload != 8:
        raise SystemExit("--loop applies to workload 8")


def main(argv=None):
    args = parse_args(argv)
    check_args(args)
    if args.workload == 7:
        return run_window_sum(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
