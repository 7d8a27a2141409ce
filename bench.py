"""Benchmark: ICP registration of the 100k <-> 100k synthetic scene on GB300.

One step = one full registration of the resident source against the resident
target tree (Morton ordering of the source, every fused correspondence pass,
every host solve, the stopping rule, the final error pass).  The target's
tree is built once per target (host) and uploaded once; `e2e` repeats the
whole job from host buffers -- tree build, upload, source upload, registration
-- through the C ABI every step.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the
same workload instead.

Launch: python bench.py [--gpus 1] [--steps K] [--warmup W]
        python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...
(N > 1: independent replicas, one per GPU, no data exchange: weak scaling.)
"""
from __future__ import annotations

import os

# the CPU oracle (baseline leg) is timed single-threaded
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NN queries/s and ICP iterations/s at 100k↔100k pts; % of HBM/L2 roofline"
UNIT = "ICP iterations/s"
WORKLOAD = ("scene 100k<->100k: ground plane 40x40 m + 20 boxes + 10 cylinders, N(0,0.01 m) noise, "
            "offset <=15 deg / <=1 m; leaf 12, max_iter 50, max correspondence 1.0 m, eps 1e-5 m^2")

# Algorithmic work per query, counted by the oracle's reference search
# (python -m oracle.yardstick; near child first, plane pruning only, no
# radius seeding, no box tests): 16 B source record + 8 B per node entered +
# 16 B per reference point measured, averaged over every query of the 51
# passes of this registration (35.85 nodes, 101.24 points per query), and
# 8 float32 operations per point measured.
ICP_BYTES_PER_QUERY = 1922.64
ICP_FP32_FLOPS_PER_QUERY = 8 * 101.24
# The same count for the 1M x 1M Gaussian-mixture nearest-neighbour query
# (leaf 16): 16 B query + 8 B result + 8 B per node + 16 B per point.
# (25.16 nodes, 49.99 points per query on average)
GMM_BYTES_PER_QUERY = 1025.07
GMM_FP32_FLOPS_PER_QUERY = 8 * 49.99

# Measured traffic of the fused pass kernel comes from the ncu summary below;
# its figures belong to the kernel source whose hash it records and are
# reported as null when the source has changed since.
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "icp_pass_kernel_traffic_scene100k.md")
KERNEL_SOURCES = [os.path.join(ROOT, "icp_nearest_neighbour_gb300", "csrc", f)
                  for f in ("kernels.cu", "kernels.cuh")]

SLOWDOWN_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


# ------------------------------------------------------------------ ranks

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(elapsed_s: float, units: float, group=None):
    """(max elapsed over ranks, sum of units over ranks); identity without a
    process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ours

def flush_l2(buf):
    buf.add_(1)


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """DRAM and L2 bytes per launch of the fused pass from the committed ncu
    summary, if it belongs to the current kernel source; else None."""
    try:
        with open(TRAFFIC_PROFILE) as f:
            text = f.read()
    except OSError:
        return None, "no traffic capture committed"
    vals = {}
    for line in text.splitlines():
        if line.startswith("traffic:"):
            for tok in line.split()[1:]:
                k, _, v = tok.partition("=")
                vals[k] = v
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None, "capture is stale: the kernel source changed since (hash differs)"
    try:
        return {"dram_bytes": float(vals["dram_bytes_per_launch"]),
                "l2_bytes": float(vals["lts_bytes_per_launch"])}, \
            f"ncu capture in {os.path.relpath(TRAFFIC_PROFILE, ROOT)} (kernel source hash matches)"
    except (KeyError, ValueError):
        return None, "traffic capture unreadable"


def workload_config(case, depth, n_nodes, iters_per_step, passes_per_step, ws):
    """The benchmark's workload description, the same for both arms."""
    return {
        "workload": WORKLOAD,
        "n_target": len(case.target), "n_source": len(case.source), "leaf_size": case.leaf_size,
        "max_iter": case.max_iter, "eps": case.eps, "max_corr_dist": case.max_corr_dist[0],
        "tree_depth": depth, "tree_nodes": n_nodes,
        "iters_per_step": iters_per_step, "passes_per_step": passes_per_step,
        "l2": "GPU arm: flushed between steps (2x L2 written); the working set stays cache-resident "
              "within a step",
        "parallelism": f"replicas x{ws}",
    }


def run_ours(args):
    import torch
    import icp_nearest_neighbour_gb300 as nn
    import workloads

    ws, rank, local = dist_env()
    # --no-prelaunch: every pass an ordinary launch (bit-identical results),
    # for profilers that serialise kernel launches
    pre = not args.no_prelaunch
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    nn.load()

    case = workloads.scene_case()
    dmax = case.max_corr_dist[0]
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.zeros(2 * l2 // 4, dtype=torch.float32, device="cuda")

    # once per target: host build + upload (timed separately, reported)
    t0 = time.perf_counter()
    tree = nn.kdtree_build(case.target, case.leaf_size)
    build_ms = (time.perf_counter() - t0) * 1e3
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    nn.kdtree_upload(tree)
    upload_ms = (time.perf_counter() - t0) * 1e3
    info = nn.kdtree_info(tree)
    src = torch.from_numpy(case.source).cuda()
    n = len(case.source)

    def step(timing, ordinary=False):
        # the library's default path: one persistent kernel per registration
        # (--no-prelaunch: ordinary launches).  timing: per-pass device times,
        # from the persistent kernel's own clock, or CUDA events around each
        # ordinary launch.
        return nn.icp_align(tree, src, case.max_iter, case.eps, dmax, timing=timing,
                            prelaunch=pre and not ordinary, warn_overlap=False, stream=stream)

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()

    # ---- device-resident timed region
    barrier()
    torch.cuda.synchronize()
    launches0 = nn.launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    results, kresults, dresults = [], [], []
    with ClockSampler(torch.cuda.current_device()) as clk:
        wall0 = time.perf_counter()
        for k in range(args.steps):
            flush_l2(flush)
            ev[k][0].record(stream)
            results.append(step(False))
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        launches = nn.launch_count() - launches0
        # the same registrations with per-pass device times
        for k in range(args.steps):
            flush_l2(flush)
            dresults.append(step(True))
        torch.cuda.synchronize()
        # and once more as ordinary launches, each pass bracketed by CUDA
        # events on its stream (the per-pass kernel's own duration)
        for k in range(args.steps):
            flush_l2(flush)
            ev_k[k][0].record(stream)
            kresults.append(step(True, ordinary=True))
            ev_k[k][1].record(stream)
        torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = sum(step_ms) / 1e3
    iters = sum(r["iters"] for r in results)
    passes = sum(r["iters"] + 1 for r in results)
    kernel_ms = [rec["kernel_ms"] for r in kresults for rec in r["trace"]]
    device_pass_ms = [rec["kernel_ms"] for r in dresults for rec in r["trace"] if rec["kernel_ms"] > 0]
    plain_s = sum(a.elapsed_time(b) for a, b in ev_k) / 1e3
    plain_iters = sum(r["iters"] for r in kresults)
    t_max, iters_all = reduce_over_ranks(total_s, iters)
    _, passes_all = reduce_over_ranks(total_s, passes)
    clocks = clk.summary()

    side = {}
    if not args.headline_only:
        side = side_measurements(args, nn, torch, tree, src, case, dmax, stream, flush, pre)

    # ---- end to end from host buffers through the C ABI, the pages' path:
    # host tree build + one upload of the tree + source copy + registration +
    # result read, every step
    pinned_src = torch.from_numpy(case.source).pin_memory()
    n_t = len(case.target)
    heap_slots = 2 ** (info["depth"] + 1)
    tree_bytes = heap_slots * (8 + 32) + n_t * 16       # nodes, boxes, leaf-ordered records
    e2e = None
    if not args.headline_only:
        h2d = d2h = e2e_iters = 0
        for _ in range(args.warmup):
            t_h = nn.kdtree_build(case.target, case.leaf_size)
            nn.kdtree_upload(t_h, stream=stream)
            nn.icp_align(t_h, pinned_src, case.max_iter, case.eps, dmax, prelaunch=pre, warn_overlap=False,
                         stream=stream)
            t_h.free()
        barrier()
        torch.cuda.synchronize()
        e0 = time.perf_counter()
        for _ in range(args.steps):
            t_h = nn.kdtree_build(case.target, case.leaf_size)
            nn.kdtree_upload(t_h, stream=stream)
            r = nn.icp_align(t_h, pinned_src, case.max_iter, case.eps, dmax, prelaunch=pre, warn_overlap=False,
                             stream=stream)
            e2e_iters += r["iters"]
            h2d += tree_bytes + n * 12
            # the source's box (24 B) and, per pass, the result's tagged words written to mapped memory
            d2h += 24 + (r["iters"] + 1) * nn.RESULT_WORDS * 8
            t_h.free()
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - e0
        e2e_max, e2e_iters_all = reduce_over_ranks(e2e_s, e2e_iters)
        # the same with the library's device tree build from the pinned target
        pinned_tgt = torch.from_numpy(case.target).pin_memory()
        dev_iters = 0
        for _ in range(args.warmup):
            t_e = nn.kdtree_build_device(pinned_tgt, case.leaf_size, stream=stream)
            nn.icp_align(t_e, pinned_src, case.max_iter, case.eps, dmax, prelaunch=pre, warn_overlap=False,
                         stream=stream)
            t_e.free()
        torch.cuda.synchronize()
        e1 = time.perf_counter()
        for _ in range(args.steps):
            t_e = nn.kdtree_build_device(pinned_tgt, case.leaf_size, stream=stream)
            r = nn.icp_align(t_e, pinned_src, case.max_iter, case.eps, dmax, prelaunch=pre, warn_overlap=False,
                             stream=stream)
            dev_iters += r["iters"]
            t_e.free()
        torch.cuda.synchronize()
        dev_s = time.perf_counter() - e1
        e2e = {"value": e2e_iters_all / e2e_max, "unit": UNIT,
               "h2d_bytes_per_step": h2d // args.steps, "d2h_bytes_per_step": d2h // args.steps,
               "includes": "host tree build + tree upload + source H2D from pinned memory + registration "
                           "+ per-pass result reads, via the C ABI (the pages' build-on-the-host path)",
               "with_device_build": {"value": dev_iters / dev_s, "unit": UNIT,
                                     "includes": "target H2D + device tree build + source H2D + "
                                                 "registration (rank 0's own clock)"}}

    if rank != 0:
        return None

    persistent = pre
    avg_kernel_s = statistics.mean(kernel_ms) / 1e3                   # ordinary launches, events
    avg_pass_s = statistics.mean(device_pass_ms) / 1e3 if device_pass_ms else avg_kernel_s
    # headline: one launch of the persistent kernel per registration; its
    # algorithmic bytes (every pass) over the registration's CUDA-event time
    step_s = total_s / args.steps
    bytes_per_step = ICP_BYTES_PER_QUERY * n * passes / args.steps
    achieved = bytes_per_step / step_s / 1e9
    if not persistent:
        achieved = ICP_BYTES_PER_QUERY * n / avg_kernel_s / 1e9
    hbm_peak, hbm_src = measured_hbm_peak()
    l2_peak = l2_probe_peak(nn, torch, l2)
    traffic, traffic_src = measured_traffic()
    sm_mhz = clocks.get("sm_mhz") or measured_sm_max_mhz()
    fp32_peak = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
    fp32_achieved = achieved / ICP_BYTES_PER_QUERY * ICP_FP32_FLOPS_PER_QUERY / 1e3
    last = results[-1]
    line = {
        "metric": METRIC,
        "value": iters_all / t_max,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_max * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(case, info["depth"], info["n_nodes"], iters // args.steps,
                                  passes // args.steps, ws),
        "pass_launch": "one persistent kernel per registration (cooperative launch; each pass waits on "
                       "the GPU for its transform)" if pre else "ordinary (after the solve)",
        "nn_queries_per_s": passes_all * n / t_max,
        "roofline": {
            "bound": "l2",
            "kernel": "icp_registration_kernel (one persistent launch per registration)" if persistent
                      else "icp_pass_kernel",
            "achieved": achieved, "peak": l2_peak, "unit": "GB/s", "frac": achieved / l2_peak,
            "peak_source": "live probe: icpnn_probe_l2_read, 32 L1-bypassing read passes over half the "
                           "L2 in one launch, best of 5 (the working set is L2-resident)",
            "traffic": (traffic["dram_bytes"] * (passes / args.steps if persistent else 1)) if traffic else None,
            "traffic_l2": (traffic["l2_bytes"] * (passes / args.steps if persistent else 1)) if traffic else None,
            "traffic_source": traffic_src + (f" -- per pass, measured on the same pass code launched as "
                                             f"icp_pass_kernel (the persistent kernel waits on the host, which "
                                             f"ncu blocks), times the {passes // args.steps} passes of one launch"
                                             if persistent else ""),
            "algorithmic_bytes_per_launch": bytes_per_step if persistent else ICP_BYTES_PER_QUERY * n,
            "bytes_per_query": ICP_BYTES_PER_QUERY,
            "timing": ("CUDA events around each timed registration on its stream: one launch of the "
                       "persistent kernel (plus the source ordering before it); the host's solves between "
                       "passes count as kernel time") if persistent else
                      "CUDA events around every pass, launched as ordinary launches",
            "per_pass": {"avg_device_us": avg_pass_s * 1e6,
                         "achieved": ICP_BYTES_PER_QUERY * n / avg_pass_s / 1e9,
                         "frac": ICP_BYTES_PER_QUERY * n / avg_pass_s / 1e9 / l2_peak,
                         "timing": "the persistent kernel's global timer, from the command reaching the "
                                   "GPU to the result published, mean over the passes of the registrations"
                                   if persistent else "as avg_kernel_us"},
            "avg_kernel_us": avg_kernel_s * 1e6,
            "avg_kernel_note": "icp_pass_kernel as ordinary launches, CUDA events around every pass",
            "hbm": {"achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                    "peak_source": hbm_src},
            "fp32": {"achieved": fp32_achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                     "frac": fp32_achieved / fp32_peak,
                     "flops_per_query": ICP_FP32_FLOPS_PER_QUERY,
                     "peak_source": f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 (FMA) x "
                                    f"{sm_mhz:.0f} MHz (median SM clock sampled under load)"},
        },
        "ordinary_launches": {"value": plain_iters / plain_s, "unit": UNIT,
                              "avg_pass_us": avg_kernel_s * 1e6,
                              "note": "the timed registrations again with each pass launched after its "
                                      "solve and bracketed by CUDA events"},
        "overlap": {"value": last["overlap"], "final_n_accepted": last["final_n_accepted"],
                    "low_overlap": last["low_overlap"],
                    "note": "accepted pairs under the returned transform / source points (the page "
                            "warns below 0.8)"},
        "gpu_launches": launches,
        "clocks": clocks,
        "once_per_target_ms": {"kdtree_build": build_ms, "kdtree_upload": upload_ms},
        "wall_s_timed_region": wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line.update(side)
    if "nn_query_gmm_1M_x_1M" in line and GMM_BYTES_PER_QUERY:
        g = line["nn_query_gmm_1M_x_1M"]["generation_order"]
        g_ach = GMM_BYTES_PER_QUERY * g["queries_per_s"] / 1e9
        g_flops = GMM_FP32_FLOPS_PER_QUERY * g["queries_per_s"] / 1e12
        line["nn_query_gmm_1M_x_1M"]["roofline"] = {
            "bound": "l2", "achieved": g_ach, "peak": l2_peak, "unit": "GB/s", "frac": g_ach / l2_peak,
            "hbm_frac": g_ach / hbm_peak, "bytes_per_query": GMM_BYTES_PER_QUERY,
            "fp32_frac": g_flops / fp32_peak,
            "timing": "the whole nn_query call in generation order (record gather + search kernel)"}
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, case.max_iter)
    return line


def side_measurements(args, nn, torch, tree, src, case, dmax, stream, flush, pre):
    """Measurements beside the headline: the other rows of the path and the
    NN-only stress case, each on its own synthetic workload."""
    import workloads
    out = {}
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    del props
    tgt_dev = torch.from_numpy(case.target).cuda()
    dev_build = []
    for rep in range(4):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        nn.kdtree_build_device(tgt_dev, case.leaf_size, stream=stream).free()
        if rep:
            dev_build.append((time.perf_counter() - t0) * 1e3)
    out["kdtree_build_device_ms"] = statistics.median(dev_build)

    # ---- the same registration with the section 4.4 residual rejection
    rr_ms, rr_iters = [], 0
    for k in range(args.steps):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        r = nn.icp_align(tree, src, case.max_iter, case.eps, dmax, residual_reject=True, prelaunch=pre,
                         warn_overlap=False, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        rr_ms.append(a.elapsed_time(b))
        rr_iters += r["iters"]
    out["with_residual_rejection"] = {"value": rr_iters / (sum(rr_ms) / 1e3), "unit": UNIT,
                                      "ms_per_step": statistics.mean(rr_ms),
                                      "iters_per_step": rr_iters // args.steps,
                                      "note": "3-sigma residual rejection and re-solve every iteration"}

    # ---- several frames in flight: 8 sources of the same scene, one tree
    _, frame_srcs, _ = workloads.scene_frames(8)
    frame_dev = [torch.from_numpy(f).cuda() for f in frame_srcs]
    multi = {}
    for mc in (1, 4, 8):
        nn.icp_align_batch(tree, frame_dev, case.max_iter, case.eps, dmax, max_concurrent=mc, prelaunch=pre,
                           stream=stream)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        b = nn.icp_align_batch(tree, frame_dev, case.max_iter, case.eps, dmax, max_concurrent=mc,
                               prelaunch=pre, stream=stream)
        torch.cuda.synchronize()
        secs = time.perf_counter() - t0
        multi[f"frames_in_flight_{mc}"] = {"value": float(b["iters"].sum()) / secs, "unit": UNIT,
                                           "ms_per_frame": secs * 1e3 / len(frame_dev)}
    out["multi_frame_8"] = dict(multi, note="8 independent 100k sources of the scene against one "
                                            "resident tree, icpnn_icp_align_batch, wall clock")

    # ---- the page's section 6 regression timing point: 200k <-> 200k, 30
    # iterations, tree build included as in the page's comparison (host build
    # + upload, the page's path), and the section 4.2 split-rule comparison
    u = workloads.uniform200k_case()
    u_src = torch.from_numpy(u.source).cuda()
    u_ms = []
    for rep in range(4):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ut = nn.kdtree_build(u.target, u.leaf_size)
        nn.kdtree_upload(ut, stream=stream)
        nn.icp_align(ut, u_src, u.max_iter, u.eps, math.inf, prelaunch=pre, stream=stream)
        torch.cuda.synchronize()
        if rep:
            u_ms.append((time.perf_counter() - t0) * 1e3)
        ut.free()
    out["uniform200k_30_iterations_ms"] = {"value": statistics.median(u_ms),
                                           "note": "section 6 regression, 200k<->200k, 30 iterations, host "
                                                   "tree build + upload + registration, wall clock"}
    split_cmp = {}
    lid = workloads.lidar_case()
    for cname, cc in (("lidar", lid), ("uniform200k", u)):
        csrc = torch.from_numpy(cc.source).cuda()
        row = {}
        for rule in (False, True):
            ct = nn.kdtree_build(cc.target, cc.leaf_size, round_robin=rule)
            nn.kdtree_upload(ct, stream=stream)
            nn.icp_align(ct, csrc, cc.max_iter, cc.eps, cc.max_corr_dist[0], prelaunch=pre, warn_overlap=False,
                         stream=stream)
            r = nn.icp_align(ct, csrc, cc.max_iter, cc.eps, cc.max_corr_dist[0], timing=True,
                             prelaunch=False, warn_overlap=False, stream=stream)
            row["round_robin_pass_us" if rule else "max_variance_pass_us"] = \
                1e3 * statistics.mean(x["kernel_ms"] for x in r["trace"])
            ct.free()
        split_cmp[cname] = row
    out["split_rule_mean_pass_us"] = split_cmp
    del u_src

    # ---- voxel-grid downsampling of the 4M-point large-case target (0.1 m)
    big = torch.from_numpy(workloads.large_case().target).cuda()
    nn.voxel_downsample(big, 0.1, stream=stream)
    vox_ms = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        vout = nn.voxel_downsample(big, 0.1, stream=stream)
        torch.cuda.synchronize()
        vox_ms.append((time.perf_counter() - t0) * 1e3)
    out["voxel_downsample_4M"] = {"points_per_s": big.shape[0] / (statistics.median(vox_ms) / 1e3),
                                  "ms": statistics.median(vox_ms), "n_in": int(big.shape[0]),
                                  "n_out": int(vout.shape[0]), "voxel_m": 0.1}
    del big

    # ---- nearest-neighbour queries alone: 1M Gaussian-mixture queries against
    # 1M points of the same mixture (leaf 16), in generation order and sorted
    # along the Morton curve; query only (the tree is built once)
    g = workloads.gmm_case()
    g_tree = nn.kdtree_build(g.reference, g.leaf_size)
    nn.kdtree_upload(g_tree, stream=stream)
    g_q = torch.from_numpy(g.queries).cuda()
    g_idx = torch.empty(len(g.queries), dtype=torch.int32, device="cuda")
    g_d2 = torch.empty(len(g.queries), dtype=torch.float32, device="cuda")
    nn_only = {}
    for label, qflags in (("generation_order", 0), ("morton_sorted", nn.MORTON_SORT)):
        for _ in range(3):
            nn.nn_query(g_tree, g_q, g_idx, g_d2, qflags, stream=stream)
        q_ms = []
        for _ in range(10):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            nn.nn_query(g_tree, g_q, g_idx, g_d2, qflags, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            q_ms.append(a.elapsed_time(b))
        med = statistics.median(q_ms)
        nn_only[label] = {"queries_per_s": len(g.queries) / (med / 1e3), "ms": med}
    g_tree.free()
    del g_q, g_idx, g_d2
    out["nn_query_gmm_1M_x_1M"] = dict(nn_only, note="1M Gaussian-mixture queries against 1M points, leaf 16, "
                                                     "device memory, L2 flushed before each, median of 10")
    return out


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (measured)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


def measured_sm_max_mhz():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        return 2070.0


def l2_probe_peak(nn, torch, l2_bytes):
    """L2 read bandwidth from the library's probe kernel: 32 L1-bypassing
    passes over a buffer of half the L2 size in one launch, best of 5."""
    x = torch.ones(l2_bytes // 2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    reps = 32
    for _ in range(2):
        nn.probe_l2_read(x, reps, sink)
    best = float("inf")
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nn.probe_l2_read(x, reps, sink)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) * 1e-3)
    return x.numel() * 4 * reps / best / 1e9


# ------------------------------------------------------------------ oracle

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_registration(case, max_iter, eps, workers=1):
    """Build + one registration with the CPU oracle, its nearest-neighbour
    searches split over `workers` host threads; returns (iters, seconds, tree)."""
    import oracle
    t0 = time.perf_counter()
    tree = oracle.KDTree(case.target, case.leaf_size)
    r = oracle.icp_align(tree, case.source, max_iter, eps, case.max_corr_dist[0], workers=workers)
    return r["iters"], time.perf_counter() - t0, tree


def cpu_baseline(case, iters):
    """The oracle on all host cores (queries split over threads), and on one."""
    import oracle
    oracle.build()
    cores = host_cores()
    n_it, secs, _ = oracle_registration(case, iters, case.eps, cores)
    n1, secs1, _ = oracle_registration(case, iters, case.eps, 1)
    return {"value": n_it / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one registration of the same 100k<->100k scene ({n_it} ICP iterations, tree build "
                      f"and final pass included), oracle C KD-tree search (queries split over {cores} "
                      f"threads) + NumPy/LAPACK solve; {secs:.1f} s",
            "single_thread": {"value": n1 / secs1, "unit": UNIT, "cores": 1, "seconds": round(secs1, 2)}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import workloads
    oracle.build()
    case = workloads.scene_case()
    max_iter = args.ref_iters or case.max_iter
    cores = host_cores()
    tree = None
    for _ in range(args.warmup):
        _, _, tree = oracle_registration(case, max_iter, case.eps, cores)
    total_it = 0
    total_s = 0.0
    for _ in range(args.steps):
        it, s, tree = oracle_registration(case, max_iter, case.eps, cores)
        total_it += it
        total_s += s
    value = total_it / total_s
    per_step = total_it // max(args.steps, 1)
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(case, tree.depth if tree else None, tree.n_nodes if tree else None,
                                  per_step, per_step + 1, ws),
        "impl_detail": f"CPU oracle as it stands: tree build + registration per step, nearest-neighbour "
                       f"queries split over {cores} host threads, NumPy/LAPACK solves",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} ICP iterations (+ tree build and final pass) of the scene "
                                   f"registration per step, oracle as it stands, queries split over "
                                   f"{cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-iters", type=int, default=0,
                    help="oracle iterations per reference step (0: the workload's max_iter, as the GPU arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="only the headline registrations (no e2e or side measurements): for profilers")
    ap.add_argument("--no-prelaunch", action="store_true",
                    help="launch every ICP pass after its solve (for profilers that serialise launches)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except ImportError:
        pass


if __name__ == "__main__":
    main()
