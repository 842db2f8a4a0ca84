"""Benchmark of the MX block-quantization hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. mx9_pack of an fp32 [16384, 8192] N(0,1) tensor;
  2. mxq_quantize_2d_dual on the MoE-grouped bf16 [65536, 7168] tensor
     (64 K-groups, offs[-1] = 57344, 8192-row uncovered tail);
  3. mx9_unpack of the packed parts of step 1 back to fp32.
The warm-up replays a one-step CUDA graph; the timed region replays, once, a
graph of the K steps (three kernel nodes each, programmatic dependent launch
between consecutive kernels) between one pair of events.  Throughput = algorithmic bytes of the step
(4.0625 B per element for the dual cast; 5.125 B per element for each MX9
pass on fp32) / device time.  Inputs are larger than the 129 MB L2, so no
flush is needed between steps.  Per-kernel figures come from separate passes
after the timed region, and the `configs` key holds the graph-replay rates of
every other workload (the 128x128 case, the MX9 outlier tensor, the specials
tensor, the throughput sweep with the three-pass speedup, the packed forms).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on the
host cores instead, on bounded samples of the same workload.  `--sweep` prints
one extra line per packed-tensor geometry, timed under CUDA-graph replay.

Multi-GPU (torchrun): every rank quantizes its own tensors (independent work,
no collective on the data path); the timing is the max over ranks and `value`
aggregates all ranks' bytes (weak scaling).
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

METRIC = "dual-axis MXFP8 quantize HBM GB/s (% of GB300 peak); MX9 pack/unpack GB/s"
DUAL_M, DUAL_N = 65536, 7168
MX9_ROWS, MX9_COLS = 16384, 8192
B_DUAL = 4.0625          # bytes per element: 2 in + 1 + 1 + 1/32 + 1/32 out
B_MX9_F32 = 5.125        # bytes per element: 4 (fp32) + 1 (q) + 1/16 + 1/16
WORKLOAD = (f"MoE-grouped dual-axis MXFP8 bf16[{DUAL_M},{DUAL_N}] 64 groups offs[-1]=57344 "
            f"+ MX9 pack/unpack fp32[{MX9_ROWS},{MX9_COLS}]")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "mxq_dual_moe_65536x7168.md")


def step_bytes() -> dict:
    return {"mxq_dual": B_DUAL * DUAL_M * DUAL_N,
            "mx9_pack": B_MX9_F32 * MX9_ROWS * MX9_COLS,
            "mx9_unpack": B_MX9_F32 * MX9_ROWS * MX9_COLS}


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("mxq_dual.cu", "mxq_device.cuh"):
        with open(os.path.join(ROOT, "mx_block_quantization_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dual kernel from the committed ncu summary,
    or None when there is none or the kernel source changed since."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")
    BUSY_PCT = 50.0  # samples below this utilization are idle moments, left out of the median

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mxq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, total = [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        try:
            rows = open(self.path).read().strip().splitlines()
        except OSError:
            rows = []
        for row in rows:
            parts = [p.strip() for p in row.split(",")]
            if len(parts) < 9:
                continue
            try:
                clk, clk_max = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            total += 1
            # a throttle reason counts whenever it shows; the clock median only
            # over samples taken while the GPU was busy (utilization, when given)
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
            try:
                busy = float(parts[9]) >= self.BUSY_PCT if len(parts) > 9 else True
            except ValueError:
                busy = True
            if busy:
                sm.append(clk)
                smax.append(clk_max)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "samples_all": total, "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------
def dist_init():
    import torch
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
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank moved bytes_per_step per step; the job
    took the slowest rank's time (weak scaling)."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


# ---------------------------------------------------------------------------
# CPU oracle timings (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------
def oracle_sample_inputs(rank_seed: int):
    """Host inputs for the oracle samples: the full workloads' generators, cut
    to windows (tiles and 16-element blocks are independent)."""
    from mx_block_quantization_gb300 import workloads as W
    xd = W.normal_bf16((1024, DUAL_N), seed=rank_seed, scale=0.02)   # first rows of the MoE tensor
    offs = W.moe_group_offsets(seed=rank_seed + 1)
    offs_win = np.minimum(offs, 1024).astype(np.int32)                # groups clipped to the window
    xm = W.normal_f32((512, MX9_COLS), seed=rank_seed)
    return xd, offs_win, xm


def _oracle_sample_loop(budget_s: float, inputs) -> tuple[float, int, float]:
    """Repeat the oracle over one sample for about budget_s: (bytes, reps, seconds)."""
    import oracle
    xd, offs, xm = inputs
    done_bytes, reps, t0 = 0.0, 0, time.perf_counter()
    while True:
        oracle.mxfp8_dual(xd, offs)
        q, e, p = oracle.mx9_pack(xm)
        oracle.mx9_unpack(q, e, p, "f32", *xm.shape)
        done_bytes += B_DUAL * xd.size + 2 * B_MX9_F32 * xm.size
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            return done_bytes, reps, time.perf_counter() - t0


def time_oracle(budget_s: float, rank_seed: int = 0) -> dict:
    """The oracle on one host thread for about budget_s, then on every host core
    at once (one independent sample per thread; the C oracle runs with the
    interpreter lock released) for about budget_s / 2; GB/s of algorithmic
    bytes."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    inputs = oracle_sample_inputs(rank_seed)
    done_bytes, reps, dt = _oracle_sample_loop(budget_s, inputs)
    what = (f"dual bf16[1024,{DUAL_N}] window of the MoE tensor with its groups clipped + "
            f"MX9 pack/unpack fp32[512,{MX9_COLS}]")
    line = {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} x ({what}), single thread, {dt:.1f} s"}
    threads = os.cpu_count() or 1
    per_thread = [oracle_sample_inputs(rank_seed + 1 + i) for i in range(threads)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(lambda inp: _oracle_sample_loop(budget_s / 2, inp), per_thread))
    wall = time.perf_counter() - t0
    line["all_cores"] = {"value": sum(r[0] for r in res) / wall / 1e9, "unit": "GB/s",
                         "cores": threads,
                         "sample": (f"{sum(r[1] for r in res)} x ({what}) over {threads} threads, "
                                    f"one seed each, {wall:.1f} s wall")}
    return line


def run_reference(args):
    # rank 0 alone times the oracle; other ranks exit without work
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if rank != 0:
        return 0
    import oracle
    from mx_block_quantization_gb300 import workloads as W
    oracle.build()
    # each step: one 128x1024 tile-row window of the MoE tensor + MX9 on fp32[8, 8192]
    xd = W.normal_bf16((128, 1024), seed=0, scale=0.02)
    offs = np.array([128], np.int32)
    xm = W.normal_f32((8, MX9_COLS), seed=0)
    step_b = B_DUAL * xd.size + 2 * B_MX9_F32 * xm.size

    def one():
        oracle.mxfp8_dual(xd, offs)
        q, e, p = oracle.mx9_pack(xm)
        oracle.mx9_unpack(q, e, p, "f32", *xm.shape)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    gbs = step_b * args.steps / dt / 1e9
    sample = (f"per step: dual bf16[128,1024] window of the MoE tensor + MX9 pack/unpack "
              f"fp32[8,{MX9_COLS}], single thread")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def graph_census(g):
    """Kernel nodes and programmatic (PDL) edges of a captured graph, read with
    the driver API; None when the graph or the driver entry points are not
    reachable (the replay-time check below still applies)."""
    import ctypes
    try:
        raw = g.raw_cuda_graph()
        cu = ctypes.CDLL("libcuda.so.1")
    except (AttributeError, RuntimeError, OSError):
        return None
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    n = sz(0)
    if cu.cuGraphGetNodes(vp(raw), None, ctypes.byref(n)) != 0:
        return None
    nodes = (vp * max(n.value, 1))()
    if cu.cuGraphGetNodes(vp(raw), nodes, ctypes.byref(n)) != 0:
        return None
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        if cu.cuGraphNodeGetType(vp(nodes[i]), ctypes.byref(t)) != 0:
            return None
        kernels += int(t.value == 0)  # CU_GRAPH_NODE_TYPE_KERNEL
    out = {"nodes": n.value, "kernel_nodes": kernels, "programmatic_edges": None}
    ne = sz(0)
    f = getattr(cu, "cuGraphGetEdges_v2", None)
    if f is not None and f(vp(raw), None, None, None, ctypes.byref(ne)) == 0 and ne.value:
        frm, to = (vp * ne.value)(), (vp * ne.value)()
        data = (ctypes.c_uint8 * (8 * ne.value))()  # CUgraphEdgeData: from_port, to_port, type, 5 reserved
        if f(vp(raw), frm, to, data, ctypes.byref(ne)) == 0:
            out["programmatic_edges"] = sum(1 for i in range(ne.value) if data[8 * i + 2] != 0)
    return out


def capture_graph(torch, stream, launch):
    """Capture `launch()` (work enqueued on `stream`) into a CUDA graph; return
    the graph and its census (graph_census)."""
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        launch()
    census = graph_census(g)
    if hasattr(g, "instantiate"):
        try:
            g.instantiate()
        except RuntimeError:
            pass  # already instantiated at capture end
    return g, census


def upload_graph(g, stream) -> bool:
    """Upload an instantiated graph to the device ahead of its first replay
    (driver API cuGraphUpload); False when the handle or entry point is not
    reachable."""
    import ctypes
    try:
        exe = g.raw_cuda_graph_exec()
        cu = ctypes.CDLL("libcuda.so.1")
        return cu.cuGraphUpload(ctypes.c_void_p(exe), ctypes.c_void_p(stream.cuda_stream)) == 0
    except (AttributeError, RuntimeError, OSError):
        return False


def in_step_breakdown(torch, dev, stream, launches, steps=20, reps=3):
    """Per-kernel durations inside the graph-replayed step with the
    programmatic overlap between kernels left intact: a graph of `steps` steps
    in which every kernel node also feeds an event-record node on a side
    branch (off the kernel chain), so that each event marks the completion of
    its kernel.  A kernel's in-step duration is the time from the previous
    kernel's completion to its own; the first kernel of each replay (timed from
    the graph's start) is left out.  Returns ({name: [us, ...]}, mean step us)."""
    side = torch.cuda.Stream(dev)
    names = [n for n, _ in launches]
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in launches] for _ in range(steps)]
    ev0 = torch.cuda.Event(enable_timing=True, external=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ev0.record(stream)
        for k in range(steps):
            for j, (_, f) in enumerate(launches):
                f()
                fork = torch.cuda.Event()
                fork.record(stream)
                side.wait_event(fork)
                ev[k][j].record(side)
        stream.wait_stream(side)
    per = {n: [] for n in names}
    step_us = []
    for rep in range(reps + 1):
        g.replay()
        torch.cuda.synchronize(dev)
        if rep == 0:
            continue  # warm replay
        prev = None
        for k in range(steps):
            for j, n in enumerate(names):
                if prev is not None:
                    per[n].append(prev.elapsed_time(ev[k][j]) * 1e3)
                prev = ev[k][j]
        step_us.append(ev[0][-1].elapsed_time(ev[steps - 1][-1]) * 1e3 / (steps - 1))
    return per, float(np.mean(step_us))


def run_gpu(args):
    import ctypes

    import torch

    import mx_block_quantization_gb300 as mxq
    from mx_block_quantization_gb300 import workloads as W
    from mx_block_quantization_gb300.build import build_library

    rank, world, local = dist_init()
    build_library()
    dev = torch.device("cuda", local)
    cap = torch.cuda.Stream(dev)          # the step's kernels are captured on this stream
    cur = torch.cuda.current_stream(dev)  # graphs replay on the current stream
    seed = rank  # each rank quantizes its own tensors

    # ---- inputs (host-generated, seeded) and outputs, resident in HBM
    xd_h, offs_h = W.moe_grouped(seed=seed)
    xm_h = W.normal_f32((MX9_ROWS, MX9_COLS), seed=seed)
    x = torch.from_numpy(xd_h.view(np.int16)).view(torch.bfloat16).to(dev)
    offs = torch.from_numpy(offs_h).to(dev)
    xm = torch.from_numpy(xm_h).to(dev)
    kw = dict(dtype=torch.uint8, device=dev)
    M, N = DUAL_M, DUAL_N
    dual_out = mxq.DualOutputs(torch.empty((M, N), **kw), torch.empty((M * N // 32,), **kw),
                               torch.empty((N, M), **kw), torch.empty((M * N // 32,), **kw))
    nb = MX9_ROWS * MX9_COLS // 16
    q = torch.empty((nb, 16), dtype=torch.int8, device=dev)
    e = torch.empty((nb,), dtype=torch.uint8, device=dev)
    p = torch.empty((nb, 1), dtype=torch.uint8, device=dev)
    y = torch.empty((MX9_ROWS, MX9_COLS), dtype=torch.float32, device=dev)

    # The graph holds the same C-ABI calls as the Python binding makes, with
    # pre-marshalled arguments; one eager step through the checked binding
    # first validates every argument.
    L = mxq.lib()
    vp = ctypes.c_void_p
    hs = vp(cap.cuda_stream)
    # Step order: the pack, the dual cast, the unpack of the pack's output.  The
    # three are independent but for the unpack, and the three orders measured
    # within 0.15% of one another; a kernel pays for the dirty L2 lines that its
    # predecessor leaves, and in this order the dual cast, which moves 58% of
    # the step's bytes, follows the read-heavy pack.
    kernels = [
        ("mx9_pack", L.mx9_pack,
         (vp(xm.data_ptr()), mxq.F32, MX9_ROWS, MX9_COLS, vp(q.data_ptr()), vp(e.data_ptr()),
          vp(p.data_ptr()), hs)),
        ("mxq_dual", L.mxq_quantize_2d_dual,
         (vp(x.data_ptr()), M, N, vp(offs.data_ptr()), offs.numel(), *(vp(t.data_ptr()) for t in dual_out), hs)),
        ("mx9_unpack", L.mx9_unpack,
         (vp(q.data_ptr()), vp(e.data_ptr()), vp(p.data_ptr()), vp(y.data_ptr()), mxq.F32,
          MX9_ROWS, MX9_COLS, hs)),
    ]

    def launcher(name, fn, a):
        def launch():
            rc = fn(*a)
            if rc:
                raise mxq.MxqError(rc, name)
        return launch

    launches = [(name, launcher(name, fn, a)) for name, fn, a in kernels]

    def launch_step():
        for _, f in launches:
            f()

    with torch.cuda.stream(cap):
        mxq.mx9_pack(xm, out=(q, e, p), stream=cap)
        mxq.quantize_2d_dual(x, offs, out=dual_out, stream=cap)
        mxq.mx9_unpack(q, e, p, torch.float32, (MX9_ROWS, MX9_COLS), out=y, stream=cap)
    torch.cuda.synchronize(dev)
    # the warm-up replays a one-step graph; the timed region replays, once, a
    # graph of the K steps, so that consecutive steps also follow each other
    # with programmatic dependent launch
    step_graph, census1 = capture_graph(torch, cap, launch_step)

    def launch_k_steps():
        for _ in range(args.steps):
            launch_step()

    timed_graph, census = capture_graph(torch, cap, launch_k_steps)
    for c, k in ((census1, 1), (census, args.steps)):
        if c is not None:
            assert c["kernel_nodes"] == len(launches) * k, f"graph of {k} steps: {c}"

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step_graph.replay()
    uploaded = upload_graph(timed_graph, cur)  # so that the timed replay does not pay for it
    torch.cuda.synchronize(dev)
    assert mxq.device_status(clear=True) == 0

    # ---- timed region: the K-step graph, no events inside
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start.record(cur)
    timed_graph.replay()
    t_end.record(cur)
    torch.cuda.synchronize(dev)
    barrier(world)
    assert mxq.device_status(clear=True) == 0
    sb = step_bytes()
    bytes_per_step = sum(sb.values())
    own_ms = t_start.elapsed_time(t_end)
    peak, peak_kind = measured_peak()
    # a replay that did no work would be far faster than the copy rate allows
    assert own_ms > 0.5 * args.steps * bytes_per_step / (peak * 1e9) * 1e3, "empty step graph"
    total_ms = max_over_ranks(own_ms, world)
    value = aggregate_gbs(bytes_per_step, args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps

    # ---- per-kernel figures, from separate passes after the timed region
    per, step_us_inst = in_step_breakdown(torch, dev, cap, launches)
    breakdown = {}
    for name, f in launches:
        avg = float(np.mean(per[name]))
        gbs = sb[name] / (avg / 1e6) / 1e9
        iso = graph_time(torch, dev, lambda s, f=f: f(), per_graph=20, replays=5, stream=cap)
        iso_gbs = sb[name] / (iso / 1e6) / 1e9
        breakdown[name] = {"avg_us": avg, "gbs": gbs, "frac_of_measured": gbs / peak,
                           "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
                           "algorithmic_bytes": sb[name],
                           "isolated": {"us": iso, "gbs": iso_gbs, "frac_of_measured": iso_gbs / peak}}
    assert mxq.device_status(clear=True) == 0
    achieved = breakdown["mxq_dual"]["gbs"]
    roofline = {"bound": "hbm", "kernel": "mxq_tile_kernel<kDual>", "achieved": achieved, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(), "algorithmic_bytes": sb["mxq_dual"],
                "timing": ("in-step duration (previous kernel's completion to this one's) from CUDA "
                           "events recorded by side-branch nodes of a 20-step graph of the same step, "
                           "replayed 3 times after the timed region; the programmatic overlap between "
                           "kernels is kept")}
    graph_info = {"steps_per_graph": args.steps, "replays_timed": 1, "uploaded_before_timing": uploaded,
                  "kernel_nodes": None if census is None else census["kernel_nodes"],
                  "programmatic_edges": None if census is None else census["programmatic_edges"],
                  "instrumented_step_us": step_us_inst}

    configs = None
    if rank == 0 and not args.no_configs:
        configs = measure_configs(mxq, torch, dev, peak)
    # the clock record spans the warm-up, the timed region, the per-kernel
    # passes and the configs (the timed region alone is a few ms at small K)
    clocks = sampler.stop()
    clocks["window"] = "warm-up through the per-workload figures; busy samples only"

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, mxq, torch, dev, cur, xd_h, offs, xm_h, dual_out, (q, e, p), y, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                           "l2": "inputs larger than L2 (129 MB); no flush",
                           "timing": "one replay of a CUDA graph holding the K steps (3 kernel "
                                     "nodes each, programmatic dependent launch between them), "
                                     "one event pair around it",
                           "frac_of_nominal_8tbs": value / world / NOMINAL_HBM_GBS},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": len(launches) * args.steps, "clocks": clocks,
                "graph": graph_info, "breakdown": breakdown, "configs": configs}
        print(json.dumps(line), flush=True)
    if args.sweep:
        run_sweep(mxq, torch, dev, rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _dual_outputs(mxq, torch, dev, M, N):
    kw = dict(dtype=torch.uint8, device=dev)
    return mxq.DualOutputs(torch.empty((M, N), **kw), torch.empty((M * N // 32,), **kw),
                           torch.empty((N, M), **kw), torch.empty((M * N // 32,), **kw))


def measure_configs(mxq, torch, dev, peak):
    """Graph-replay throughput of every workload besides the step's (20
    launches per graph, median of 5 replays): the 128x128 case, the MX9
    4096x4096 outlier tensor, the 8192x8192 specials tensor, the throughput
    sweep (fused cast, its three-pass composition and the speedup, MX9 fp32
    and bf16) and the packed MX9/MX6 tensor along both axes at 16384x8192."""
    from mx_block_quantization_gb300 import workloads as W

    def rate(us, nbytes):
        gbs = nbytes / (us / 1e6) / 1e9
        return {"us": round(us, 3), "gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4)}

    def t(launch):
        return graph_time(torch, dev, launch, per_graph=20, replays=5)

    def bf16_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    res = {"peak_gbs": peak, "timing": "CUDA-graph replay, 20 launches per graph, median of 5"}
    xb, offs1 = W.dual_small()
    x, o = bf16_dev(xb), torch.from_numpy(offs1).to(dev)
    out = _dual_outputs(mxq, torch, dev, 128, 128)
    res["dual_128x128_one_group"] = {
        **rate(t(lambda s: mxq.quantize_2d_dual(x, o, out=out, stream=s)), B_DUAL * 128 * 128),
        "note": "66.6 KB per launch: launch-bound, L2-resident"}
    xf = torch.from_numpy(W.mx9_outliers()).to(dev)
    for dt, tdt, bpe in (("f32", torch.float32, B_MX9_F32), ("bf16", torch.bfloat16, 3.125)):
        xin = xf.to(tdt)
        q, e, p = mxq.mx9_pack(xin)
        yy = torch.empty_like(xin)
        nbytes = bpe * xin.numel()
        res[f"mx9_outliers_4096x4096_{dt}"] = {
            "pack": rate(t(lambda s: mxq.mx9_pack(xin, out=(q, e, p), stream=s)), nbytes),
            "unpack": rate(t(lambda s: mxq.mx9_unpack(q, e, p, tdt, tuple(xin.shape), out=yy, stream=s)),
                           nbytes),
            "l2_resident": nbytes < 129e6}
    del xf, xin, q, e, p, yy
    xs = bf16_dev(W.dual_specials())
    out = _dual_outputs(mxq, torch, dev, 8192, 8192)
    res["dual_specials_8192x8192_dense"] = rate(t(lambda s: mxq.quantize_2d_dual(xs, out=out, stream=s)),
                                                B_DUAL * 8192 * 8192)
    del xs, out
    sweep, speedups = {}, []
    gen = torch.Generator(device=dev)
    for (M, N) in W.SWEEP_SHAPES:
        gen.manual_seed(0)
        xf = torch.randn((M, N), generator=gen, device=dev, dtype=torch.float32)
        xb16 = xf.to(torch.bfloat16)
        out = _dual_outputs(mxq, torch, dev, M, N)
        ws = torch.empty((M * N // 32,), dtype=torch.uint8, device=dev)
        fused = t(lambda s: mxq.quantize_2d_dual(xb16, out=out, stream=s))
        three = t(lambda s: mxq.quantize_2d_dual_3pass(xb16, workspace=ws, out=out, stream=s))
        row = {"dual": rate(fused, B_DUAL * M * N), "dual_3pass": rate(three, B_DUAL * M * N),
               "fused_speedup_vs_3pass": round(three / fused, 3),
               "l2_resident": B_DUAL * M * N < 129e6}
        speedups.append(three / fused)
        del out, ws
        for dt, xin, bpe in (("f32", xf, B_MX9_F32), ("bf16", xb16, 3.125)):
            q, e, p = mxq.mx9_pack(xin)
            yy = torch.empty_like(xin)
            row[f"mx9_pack_{dt}"] = rate(t(lambda s: mxq.mx9_pack(xin, out=(q, e, p), stream=s)), bpe * M * N)
            row[f"mx9_unpack_{dt}"] = rate(t(lambda s: mxq.mx9_unpack(
                q, e, p, xin.dtype, (M, N), out=yy, stream=s)), bpe * M * N)
            del q, e, p, yy
        sweep[f"{M}x{N}"] = row
        del xf, xb16
        torch.cuda.empty_cache()
    res["sweep"] = sweep
    res["fused_speedup_geomean"] = round(float(np.exp(np.mean(np.log(speedups)))), 3)
    res["fused_speedup_pages"] = "2.6x geomean, 2.0x at the largest shape (GB200, 2062 MHz)"
    M, N = 16384, 8192
    gen.manual_seed(1)
    xf = torch.randn((M, N), generator=gen, device=dev, dtype=torch.float32)
    packed = {}
    for dt, xin, esz in (("f32", xf, 4), ("bf16", xf.to(torch.bfloat16), 2)):
        yy = torch.empty_like(xin)
        for fmt, fname in ((mxq.FMT_MX9, "mx9"), (mxq.FMT_MX6, "mx6")):
            nbytes = (esz + mxq.RECORD_BYTES[fmt] / 16) * M * N
            for axis, aname in ((1, "rows"), (0, "cols")):
                rec = mxq.mx_pack_packed(xin, fmt, axis)
                packed[f"{fname}_{aname}_{dt}"] = {
                    "pack": rate(t(lambda s: mxq.mx_pack_packed(xin, fmt, axis, out=rec, stream=s)), nbytes),
                    "unpack": rate(t(lambda s: mxq.mx_unpack_packed(rec, fmt, yy, axis, stream=s)), nbytes)}
                del rec
        del yy
    res[f"packed_{M}x{N}"] = packed
    del xf
    torch.cuda.empty_cache()
    return res


def run_e2e(args, mxq, torch, dev, stream, xd_h, offs, xm_h, dual_out, mx9_parts, y, world):
    """The same step through the public API with pinned host buffers, as a
    pipelined stream of batches: every step copies its inputs host->device,
    runs the three calls and copies every output device->host, all inside the
    timed region.  Two device buffer sets and three streams (H2D, compute,
    D2H) ordered by events let step k+1's upload and step k-1's download run
    while step k computes."""
    x_h = torch.from_numpy(xd_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    xm_hp = torch.from_numpy(xm_h).pin_memory()
    q0, e0, p0 = mx9_parts

    def device_slot():
        kw = dict(dtype=torch.uint8, device=dev)
        M, N = x_h.shape
        return {"x": torch.empty_like(x_h, device=dev), "xm": torch.empty_like(xm_hp, device=dev),
                "dual": mxq.DualOutputs(torch.empty((M, N), **kw), torch.empty((M * N // 32,), **kw),
                                        torch.empty((N, M), **kw), torch.empty((M * N // 32,), **kw)),
                "mx9": (torch.empty_like(q0), torch.empty_like(e0), torch.empty_like(p0)),
                "y": torch.empty_like(y)}

    slots = [device_slot(), device_slot()]
    for sl in slots:
        sl["outs"] = list(sl["dual"]) + list(sl["mx9"]) + [sl["y"]]
        sl["host"] = [torch.empty_like(t, device="cpu").pin_memory() for t in sl["outs"]]
        sl["h2d_done"] = torch.cuda.Event()
        sl["comp_done"] = torch.cuda.Event()
        sl["d2h_done"] = torch.cuda.Event()
    s_h2d, s_comp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))

    def step(k):
        sl = slots[k % 2]
        with torch.cuda.stream(s_h2d):
            if k >= 2:
                s_h2d.wait_event(sl["comp_done"])     # inputs of step k-2 consumed
            sl["x"].copy_(x_h, non_blocking=True)
            sl["xm"].copy_(xm_hp, non_blocking=True)
            sl["h2d_done"].record(s_h2d)
        s_comp.wait_event(sl["h2d_done"])
        if k >= 2:
            s_comp.wait_event(sl["d2h_done"])         # outputs of step k-2 downloaded
        q, e, p = sl["mx9"]
        mxq.mx9_pack(sl["xm"], out=(q, e, p), stream=s_comp)
        mxq.quantize_2d_dual(sl["x"], offs, out=sl["dual"], stream=s_comp)
        mxq.mx9_unpack(q, e, p, torch.float32, tuple(sl["xm"].shape), out=sl["y"], stream=s_comp)
        sl["comp_done"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(sl["comp_done"])
            for h, d in zip(sl["host"], sl["outs"]):
                h.copy_(d, non_blocking=True)
            sl["d2h_done"].record(s_d2h)

    for k in range(2):
        step(k)
    torch.cuda.synchronize(dev)
    steps = args.e2e_steps
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_h2d)
    s_comp.wait_event(t0)
    s_d2h.wait_event(t0)
    for k in range(steps):
        step(k)
    s_d2h.wait_event(slots[(steps - 1) % 2]["d2h_done"])
    t1.record(s_d2h)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    h2d = x_h.numel() * 2 + xm_hp.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in slots[0]["host"])
    return {"value": aggregate_gbs(sum(step_bytes().values()), steps, world, ms), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "pipelining": "2 buffer sets; H2D, compute and D2H streams overlap across steps"}


def run_sweep(mxq, torch, dev, rank):
    """With --sweep: the packed tensor in its other geometries (blocks along
    columns, and blocked rows at a pitch of cols + 64, the input a strided
    view) at a mid and a large shape, one line each, under graph replay."""
    peak, kind = measured_peak()
    for M, N in ((16384, 8192), (32768, 16384)):
        run_sweep_packed(mxq, torch, dev, rank, M, N, peak, kind)


def run_sweep_packed(mxq, torch, dev, rank, M, N, peak, kind):
    from mx_block_quantization_gb300 import workloads as W

    line = {"sweep_packed_geometries": [M, N], "peak_gbs": peak, "peak_kind": kind}
    for dt, tdt, esz in (("f32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        wide = torch.from_numpy(W.normal_f32((M, N + 64), seed=0)).to(dev).to(tdt)
        ywide = torch.empty_like(wide)
        for layout, xin, yout, axis in (("axis0", wide[:, :N].contiguous(), None, 0),
                                        ("pitched_rows", wide[:, :N], ywide[:, :N], 1)):
            yy = torch.empty_like(xin) if yout is None else yout
            for fmt, name in ((mxq.FMT_MX9, "mx9"), (mxq.FMT_MX6, "mx6")):
                rec = mxq.mx_pack_packed(xin, fmt, axis)
                pbytes = (esz + mxq.RECORD_BYTES[fmt] / 16) * M * N
                for op, launch in (("pack", lambda s: mxq.mx_pack_packed(xin, fmt, axis, out=rec, stream=s)),
                                   ("unpack", lambda s: mxq.mx_unpack_packed(rec, fmt, yy, axis, stream=s))):
                    gbs = pbytes / (graph_time(torch, dev, launch) / 1e6) / 1e9
                    line[f"{name}_{layout}_{op}_{dt}"] = {"gbs": gbs, "frac_of_measured": gbs / peak}
                del rec
        del wide, ywide
    if rank == 0:
        print(json.dumps(line), flush=True)
    torch.cuda.empty_cache()


def graph_time(torch, dev, launch, per_graph=20, replays=10, stream=None):
    """Median per-launch time (us) of `launch(stream)` captured per_graph times
    into one CUDA graph; the graph must contain kernel work (timed replay > 0)."""
    s = torch.cuda.Stream(dev) if stream is None else stream
    with torch.cuda.stream(s):
        launch(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            launch(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(replays):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        g.replay()
        b.record(cur)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b) * 1e3 / per_graph)
    med = statistics.median(times)
    assert med > 0.5, "graph replay took no time: nothing was captured"
    return med


def run_case(args):
    """Launch one kernel `--warmup` times on one shape (for profiler captures)."""
    import torch

    import mx_block_quantization_gb300 as mxq
    from mx_block_quantization_gb300 import workloads as W
    from mx_block_quantization_gb300.build import build_library

    build_library()
    M, N = (int(v) for v in args.shape.lower().split("x"))
    dev = torch.device("cuda", 0)
    if args.case in ("dual", "dual3"):
        # dual3: the three-pass composition (1x32 cast, 32x1 cast, K-groups swizzle)
        offs = None
        if args.groups:
            offs = torch.from_numpy(W.moe_group_offsets(args.groups, M // 128 - M // 1024)).to(dev)
        x = torch.from_numpy(W.normal_bf16((M, N), seed=0, scale=0.02).view(np.int16)).view(
            torch.bfloat16).to(dev)
        out = mxq.quantize_2d_dual(x, offs)
        ws = torch.empty(M * N // 32, dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            if args.case == "dual":
                mxq.quantize_2d_dual(x, offs, out=out)
            else:
                mxq.quantize_2d_dual_3pass(x, offs, workspace=ws, out=out)
    elif args.case == "mma":
        # the tensor-core consumer check on the cast of an [M, N] tensor: q_row
        # and s_row against themselves (K = N)
        x = torch.from_numpy(W.normal_bf16((M, N), seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
        out = mxq.quantize_2d_dual(x)
        d = torch.empty((M, M), dtype=torch.float32, device=dev)
        for _ in range(args.warmup):
            mxq.mxfp8_scaled_mm(out.q_row, out.s_row, out.q_row, out.s_row, out=d)
    elif args.case.startswith("rec_"):
        # the single packed tensor of MX9 (--fmt 9) or MX6 (--fmt 6) records, rows blocked
        tdt = torch.float32 if args.case.endswith("f32") else torch.bfloat16
        wide = torch.from_numpy(W.normal_f32((M, N + args.pad), seed=0)).to(dev).to(tdt)
        xm = wide[:, :N]                       # rows args.pad elements longer than the tensor
        rec = mxq.mx_pack_packed(xm, args.fmt, args.axis)
        y = torch.empty_like(wide)[:, :N]
        for _ in range(args.warmup):
            if args.case.startswith("rec_pack"):
                mxq.mx_pack_packed(xm, args.fmt, args.axis, out=rec)
            else:
                mxq.mx_unpack_packed(rec, args.fmt, y, args.axis)
    else:
        tdt = torch.float32 if args.case.endswith("f32") else torch.bfloat16
        xm = torch.from_numpy(W.normal_f32((M, N), seed=0)).to(dev).to(tdt)
        q, e, p = mxq.mx9_pack(xm)
        for _ in range(args.warmup):
            if args.case.startswith("pack"):
                mxq.mx9_pack(xm, out=(q, e, p))
            else:
                mxq.mx9_unpack(q, e, p, tdt, (M, N))
    torch.cuda.synchronize()
    assert mxq.device_status(clear=True) == 0
    print(json.dumps({"case": args.case, "shape": [M, N], "launches": args.warmup,
                      **({"fmt": args.fmt, "axis": args.axis, "pad": args.pad} if args.case.startswith("rec_") else {})}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload graph-replay figures of the JSON line's configs key")
    ap.add_argument("--sweep", action="store_true",
                    help="also print one line per packed-tensor geometry (graph replay)")
    ap.add_argument("--case", choices=["dual", "dual3", "mma", "pack_f32", "pack_bf16", "unpack_f32", "unpack_bf16",
                                       "rec_pack_f32", "rec_pack_bf16", "rec_unpack_f32",
                                       "rec_unpack_bf16"],
                    help="only launch this kernel --warmup times on --shape (profiling)")
    ap.add_argument("--shape", default="16384x7168")
    ap.add_argument("--fmt", type=int, choices=[9, 6], default=9,
                    help="with --case rec_*: MX9 or MX6 records")
    ap.add_argument("--axis", type=int, choices=[0, 1], default=1,
                    help="with --case rec_*: blocks along columns (0) or rows (1)")
    ap.add_argument("--pad", type=int, default=0,
                    help="with --case rec_*: row pitch = columns + PAD elements")
    ap.add_argument("--groups", type=int, default=0,
                    help="with --case dual: that many K-groups and a 1/8 uncovered tail")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
