"""Benchmark of the GB300 DFlash2 candidate selector.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--requests R] [--e2e-steps E] [--graph]
                    [--no-cpu-baseline] [--no-per-workload]
    python bench.py --forward | --lmhead [--sustained SECONDS | --lmhead-only] | --best-path
                    [--workload NAME]

One step is one dflash_selector call over one batch of the workload: vocabulary top-k,
hidden projection and edge scores, with every input already in HBM. The default
workload is gemma_large (R=512 requests, S=15 steps, K=32, V=262144, H=5376, rank=256),
the largest of the five. Its 8.4 GB of inputs per step far exceed the 129 MB L2, so no
flush is needed between steps.

Rank 0 prints one JSON line. It holds:
  * value: edge scores per second (R*S*K^2 per step), summed over ranks;
  * roofline: for the dominant kernel (the top-k scan), its algorithmic bytes per launch
    over its mean duration, which the library's stage events measure on traced calls of the
    same step right after the timed region (untraced, the step's kernels overlap), against
    the measured HBM peak;
  * e2e: the same metric through the C ABI with pinned host buffers, host-to-device and
    device-to-host copies inside the timed region;
  * cpu_baseline: the CPU oracle, as it stands, on a bounded sample of the workload;
  * clocks: nvidia-smi samples taken during the timed region;
  * forward (one GPU): the selector's forward pass on the step's candidates (projection,
    then edges, the pages' DFlash2BeamCandidateSelector.forward), and each kernel alone,
    with L2 flushed before every call;
  * per_workload (one GPU): each of the other four workloads through the same call, after
    the headline's timed region: step time, the top-k's and the whole step's fraction of
    the HBM peak, and the CPU oracle timed over the whole workload.
With torchrun (N > 1) every rank runs an independent replica on its own GPU and its own
seed (weak scaling). The only collectives are a barrier and a max over ranks of the time.

The other modes time one part alone: --forward the selector's forward pass (no logits),
--lmhead the top-k straight from the LM head (with cuBLAS GEMM plus top-k beside it for
context), --best-path the max-sum path through the edge scores. --graph replays the step from
a CUDA graph; --requests takes the first R requests of the workload (small cases for ncu).

--impl reference times the CPU oracle (the reference arm of this benchmark) on a bounded
sample per step, on the host cores, and prints the same line with "impl": "reference".
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from draft_candidate_selector_gb300 import workloads as wl  # noqa: E402

METRIC = "selector edge scores/s (R*S*K^2)"
UNIT = "edge_scores/s"
PROFILE_TOPK = os.path.join(ROOT, "profiles", "topk_gemma_large.json")
TOPK_SOURCE = os.path.join(ROOT, "draft_candidate_selector_gb300", "csrc", "topk.cu")


# ----------------------------------------------------------------------------- helpers

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(ms_local: float, units_local: int, world: int, group=None) -> tuple[float, float]:
    """Max over ranks of the step time, and the whole-job throughput (units per second).

    Every rank processes units_local units per step (weak scaling), so the job processes
    world * units_local units in the slowest rank's time.
    """
    t = torch.tensor([ms_local], dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend(group) == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    ms_max = float(t.item())
    return ms_max, world * units_local / (ms_max / 1e3)


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "source": "fallback (6.8 TB/s and 1.9 PFLOP/s bf16, earlier GB300 measurement)"}


def profiled_traffic(workload: wl.Workload) -> float | None:
    """DRAM bytes per top-k launch at this workload's full size, from the committed ncu
    summary profiles/topk_gemma_large.json, if that was taken on the current top-k source
    (its sha256 is recorded with it) and on this workload; otherwise None."""
    if not os.path.exists(PROFILE_TOPK):
        return None
    with open(PROFILE_TOPK) as f:
        prof = json.load(f)
    if prof.get("workload") != workload.name or prof.get("R") != workload.R:
        return None
    with open(TOPK_SOURCE, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != prof.get("source_sha256"):
            return None
    return float(prof["traffic_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clocks and throttle reasons."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device: torch.device):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.target = str(device.index or 0)

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="dflash_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", self.target],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict | None:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(self.FIELDS):
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                try:
                    power.append(float(parts[3]))
                except ValueError:
                    pass
                for n, v in zip(names, parts[5:]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_sample(inp: wl.Inputs, n_req: int, threads: int) -> float:
    """Seconds the CPU oracle takes for the whole selector on the first n_req requests."""
    import oracle
    t0 = time.perf_counter()
    oracle.selector(inp.logits[:n_req], bits(inp.hidden[:n_req]), bits(inp.w_proj),
                    bits(inp.pred_cb), bits(inp.succ_cb), inp.anchors[:n_req],
                    inp.workload.K, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(inp: wl.Inputs, target_s: float = 15.0) -> dict:
    """The oracle on a bounded sample: requests are added until about target_s of work."""
    import oracle
    w = inp.workload
    threads = oracle.default_threads()
    t1 = oracle_sample(inp, 1, threads)
    n = int(max(1, min(w.R, target_s / max(t1, 1e-3))))
    t = oracle_sample(inp, n, threads) if n > 1 else t1
    edges = n * w.S * w.K * w.K
    return {"value": edges / t, "unit": UNIT, "cores": min(threads, n * w.S), "kind": "oracle",
            "sample": f"{n} of {w.R} requests x {w.S} steps of {w.name} (fp64 CPU oracle, "
                      f"{t:.1f} s)"}


def base_config(w: wl.Workload, world: int) -> dict:
    return {"workload": w.name, "R": w.R, "S": w.S, "K": w.K, "V": w.V, "H": w.H,
            "rank": w.rank, "description": w.description,
            "l2": "inputs larger than L2 (no flush needed)",
            "parallelism": "replicas" if world == 1 else f"replicas x{world}"}


def l2_bytes(dev) -> int:
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 129 << 20


def timed_calls(fn, steps: int, stream, flush: torch.Tensor | None) -> float:
    """Mean ms of one call of fn over `steps` calls, timed with CUDA events on `stream`.

    With a flush buffer (larger than L2), the buffer is read before every call and each call
    is timed alone, so no call finds its inputs in L2 (reading, not writing, so that the timed
    call does not pay for writing dirty lines back); otherwise the calls run back to back
    between two events.
    """
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps
    pairs = []
    for _ in range(steps):
        flush.sum()        # a read: leaves L2 holding clean lines of the flush buffer
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in pairs)


def oracle_whole(inp: wl.Inputs) -> dict:
    """The CPU oracle, as it stands, over the whole workload on all host cores."""
    import oracle
    w = inp.workload
    threads = oracle.default_threads()
    t = oracle_sample(inp, w.R, threads)
    return {"value": w.edges_per_call / t, "unit": UNIT, "cores": min(threads, w.rows),
            "kind": "oracle", "seconds": t,
            "sample": f"all {w.R} requests x {w.S} steps of {w.name} (fp64 CPU oracle, {t:.2f} s)"}


def measure_workload(ds, w: wl.Workload, dev, stream, steps: int, warmup: int, seed: int,
                     peak_gbs: float, with_cpu: bool) -> dict:
    """One smaller workload through the same public call as the headline: step time, the
    top-k's and the whole step's fraction of the HBM peak, and the oracle over all of it."""
    inp = wl.make_inputs(w, seed=seed)
    d = {"logits": torch.from_numpy(inp.logits).to(dev), "hidden": inp.hidden.to(dev),
         "w_proj": inp.w_proj.to(dev), "pred_cb": inp.pred_cb.to(dev),
         "succ_cb": inp.succ_cb.to(dev), "anchors": torch.from_numpy(inp.anchors).to(dev)}
    cand = torch.empty((w.R, w.S, w.K), dtype=torch.int32, device=dev)
    unary = torch.empty((w.R, w.S, w.K), dtype=torch.float32, device=dev)
    h = torch.empty((w.R, w.S, w.rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((w.R, w.S, w.K, w.K), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.dflash_selector_workspace_bytes(w.R, w.S, w.V, w.K), dtype=torch.uint8,
                     device=dev)

    def step():
        ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"], d["succ_cb"],
                           d["anchors"], w.K, cand, unary, h, edges, ws)

    b = w.algorithmic_bytes()
    total = sum(b.values())
    topk_bytes = b["logits"] + b["ids_unary_out"]
    # Inputs within a few times the L2 would be partly served from it: flush between steps.
    flush = (torch.zeros(2 * l2_bytes(dev) // 4, dtype=torch.float32, device=dev)
             if total < 3 * l2_bytes(dev) else None)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    ms = timed_calls(step, steps, stream, flush)
    # Stage times from traced calls right after (a traced call runs its kernels one after
    # another; untraced, the edges overlap the top-k's tail).
    ds.dflash_trace_begin(steps)
    timed_calls(step, steps, stream, flush)
    stages = ds.dflash_trace_end(steps)
    topk_ms = statistics.mean(s[1] for s in stages)
    # The same step captured once in a CUDA graph and replayed: for the small workloads the
    # eager time is mostly host launch cost.
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    graph_ms = timed_calls(graph.replay, steps, stream, flush)
    del graph
    out = {"R": w.R, "S": w.S, "K": w.K, "V": w.V, "H": w.H, "rank": w.rank,
           "steps": steps, "ms_per_step": ms,
           "value": w.edges_per_call / (ms / 1e3), "unit": UNIT,
           "l2": ("L2 flushed before every step (a buffer of twice the L2 read), each "
                  "step timed alone" if flush is not None else "inputs larger than L2"),
           "launch_mode": "eager",
           "graph_replay": {"ms_per_step": graph_ms, "value": w.edges_per_call / (graph_ms / 1e3),
                            "fused_hbm_frac": total / (graph_ms / 1e3) / 1e9 / peak_gbs},
           "stages_ms": {"projection": statistics.mean(s[0] for s in stages), "topk": topk_ms,
                         "edges": statistics.mean(s[2] for s in stages)},
           "topk_hbm": {"algorithmic_bytes": topk_bytes,
                        "achieved_gbs": topk_bytes / (topk_ms / 1e3) / 1e9,
                        "frac": topk_bytes / (topk_ms / 1e3) / 1e9 / peak_gbs},
           "fused_hbm": {"algorithmic_bytes_per_step": total,
                         "achieved_gbs": total / (ms / 1e3) / 1e9,
                         "frac": total / (ms / 1e3) / 1e9 / peak_gbs},
           "device_status": ds.dflash_device_status(clear=True)}
    del d, cand, unary, h, edges, ws, flush
    torch.cuda.empty_cache()
    if with_cpu:
        out["cpu_baseline"] = oracle_whole(inp)
    return out


def measure_forward(ds, w: wl.Workload, dev, stream, steps: int, warmup: int, peaks: dict, cand,
                    unary, hidden, anchors, w_proj, pred_cb, succ_cb, h, edges) -> dict:
    """The selector's forward pass on given candidates (projection, then edges), and each of
    its two kernels alone, with L2 flushed before every call."""
    flush = torch.zeros(2 * l2_bytes(dev) // 4, dtype=torch.float32, device=dev)
    calls = {
        "forward": lambda: ds.dflash_selector_forward(cand, unary, hidden, anchors, w_proj,
                                                      pred_cb, succ_cb, h, edges),
        "projection": lambda: ds.dflash_hidden_projection(hidden, w_proj, h),
        "edges": lambda: ds.dflash_candidate_edges(pred_cb, succ_cb, cand, unary, h, anchors,
                                                   edges),
    }
    out = {}
    for name, fn in calls.items():
        for _ in range(warmup):
            fn()
        out[f"{name}_ms"] = timed_calls(fn, steps, stream, flush)
    # The fixed cost of any launch timed this way: a one-CTA kernel that writes 4 bytes,
    # between the same two events after the same flush.
    tiny = torch.zeros(1, dtype=torch.float32, device=dev)
    for _ in range(warmup):
        tiny.zero_()
    out["launch_floor_ms"] = timed_calls(tiny.zero_, steps, stream, flush)
    b = w.algorithmic_bytes()
    proj_bytes = b["hidden"] + b["w_proj"] + b["h_out"]
    proj_flops = 2.0 * w.rows * w.H * w.rank
    bound_ms = max(proj_bytes / (peaks["hbm_gbs"] * 1e9),
                   proj_flops / (peaks["bf16_tflops"] * 1e12)) * 1e3
    out["edge_scores_per_s"] = w.edges_per_call / (out["forward_ms"] / 1e3)
    out["projection_roofline"] = {
        "bound": "hbm" if proj_bytes / peaks["hbm_gbs"] > proj_flops / peaks["bf16_tflops"] / 1e3
                 else "tensor",
        "algorithmic_bytes": proj_bytes, "flops": proj_flops, "bound_ms": bound_ms,
        "frac": bound_ms / out["projection_ms"],
        "frac_net_of_launch_floor": bound_ms / max(out["projection_ms"] - out["launch_floor_ms"], 1e-9),
        "best_frac_with_launch_floor": bound_ms / (bound_ms + out["launch_floor_ms"]),
        "what": "max(bytes / HBM peak, FLOPs / bf16 burst peak), both measured, over the "
                "projection's time; net of the launch floor, and the best a kernel at the "
                "bound could show measured this way"}
    out["l2"] = "L2 flushed before every call (a buffer of twice the L2 read)"
    del flush
    return out


# ----------------------------------------------------------------------------- arms

def run_reference(args, w: wl.Workload) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    threads = oracle.default_threads()
    inp = wl.make_inputs(w, seed=0)
    n_req = 1   # one request (S rows) per step keeps --steps K runs within minutes
    for _ in range(args.warmup):
        oracle_sample(inp, n_req, threads)
    times = [oracle_sample(inp, n_req, threads) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    edges = n_req * w.S * w.K * w.K
    value = edges / (ms / 1e3)
    sample = f"{n_req} of {w.R} requests x {w.S} steps of {w.name} per step (fp64 CPU oracle)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": base_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, n_req * w.S),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours(args, w: wl.Workload) -> None:
    import draft_candidate_selector_gb300 as ds

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    # Inputs: logits are generated straight into pinned host memory (the e2e source).
    logits_host = torch.empty((w.R, w.S, w.V), dtype=torch.float32, pin_memory=True)
    inp = wl.make_inputs(w, seed=rank, logits_out=logits_host.numpy())
    hidden_host = inp.hidden.pin_memory()
    anchors_host = torch.from_numpy(inp.anchors).pin_memory()
    logits = logits_host.to(dev)
    hidden = hidden_host.to(dev)
    anchors = anchors_host.to(dev)
    w_proj, pred_cb, succ_cb = inp.w_proj.to(dev), inp.pred_cb.to(dev), inp.succ_cb.to(dev)
    cand = torch.empty((w.R, w.S, w.K), dtype=torch.int32, device=dev)
    unary = torch.empty((w.R, w.S, w.K), dtype=torch.float32, device=dev)
    h = torch.empty((w.R, w.S, w.rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((w.R, w.S, w.K, w.K), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.dflash_selector_workspace_bytes(w.R, w.S, w.V, w.K), dtype=torch.uint8,
                     device=dev)

    def step():
        ds.dflash_selector(logits, hidden, w_proj, pred_cb, succ_cb, anchors, w.K, cand, unary,
                           h, edges, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ds.dflash_device_status(clear=True)

    graph = None
    if args.graph:
        # The whole step captured once in a CUDA graph (a memset node and three kernels).
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)

    # ---- timed region (device-resident inputs)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clocks:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(args.steps):
            if graph is None:
                step()
            else:
                graph.replay()
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    # Stage times. Untraced, the kernels of a step overlap (the top-k beside the projection,
    # the edges in the top-k's tail), so no event can sit between them inside the timed
    # region without removing the overlap. A traced call records events between its kernels,
    # which then run one after another: the same call on the same stream and inputs, right
    # after the timed region, gives each kernel's own duration.
    n_tr = min(args.steps, 50)
    ds.dflash_trace_begin(n_tr)
    for _ in range(n_tr):
        step()
    torch.cuda.synchronize(dev)
    stages = ds.dflash_trace_end(n_tr)
    stages_source = (f"stage events of {n_tr} traced calls (kernels one after another) on the "
                     f"same stream and inputs, right after the timed region")
    ms_local = start.elapsed_time(stop) / args.steps
    status = ds.dflash_device_status(clear=True)
    ms_max, value = aggregate(ms_local, w.edges_per_call, world)

    # ---- end to end through the public call, with host buffers
    out_edges = torch.empty(edges.shape, dtype=edges.dtype, pin_memory=True)
    out_cand = torch.empty(cand.shape, dtype=cand.dtype, pin_memory=True)
    out_unary = torch.empty(unary.shape, dtype=unary.dtype, pin_memory=True)
    h2d = logits_host.nbytes + hidden_host.nbytes + anchors_host.nbytes
    d2h = out_edges.nbytes + out_cand.nbytes + out_unary.nbytes

    # End to end, pipelined by chunks of requests (they are independent): the inputs of
    # chunk c+1 copy in on one stream while the selector runs on chunk c, and outputs copy
    # out on a third stream. Device buffers alternate between two sets by step, so the next
    # step's copies overlap this step's kernels; per-chunk events keep a set's chunk from
    # being overwritten before the kernel that reads it, or its outputs before they are read
    # back. The host link, not the kernels, bounds this number.
    nch = max(1, min(args.e2e_chunks, w.R))
    bounds = [w.R * c // nch // 4 * 4 for c in range(nch)] + [w.R]   # 16-byte aligned chunks
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [dict(logits=logits, hidden=hidden, anchors=anchors, cand=cand, unary=unary, h=h,
                 edges=edges)]
    sets.append({k: torch.empty_like(v) for k, v in sets[0].items()})
    ev_in = [[torch.cuda.Event() for _ in range(nch)] for _ in range(2)]
    ev_kernel = [[torch.cuda.Event() for _ in range(nch)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(nch)] for _ in range(2)]
    recorded = [False, False]
    step_no = [0]

    def e2e_step():
        p = step_no[0] % 2
        d = sets[p]
        for c in range(nch):
            r0, r1 = bounds[c], bounds[c + 1]
            if r1 <= r0:
                continue
            with torch.cuda.stream(copy_in):
                if recorded[p]:
                    copy_in.wait_event(ev_kernel[p][c])      # the set's last reader is done
                d["logits"][r0:r1].copy_(logits_host[r0:r1], non_blocking=True)
                d["hidden"][r0:r1].copy_(hidden_host[r0:r1], non_blocking=True)
                d["anchors"][r0:r1].copy_(anchors_host[r0:r1], non_blocking=True)
                ev_in[p][c].record(copy_in)
            stream.wait_event(ev_in[p][c])
            if recorded[p]:
                stream.wait_event(ev_out[p][c])              # its outputs were read back
            ds.dflash_selector(d["logits"][r0:r1], d["hidden"][r0:r1], w_proj, pred_cb, succ_cb,
                               d["anchors"][r0:r1], w.K, d["cand"][r0:r1], d["unary"][r0:r1],
                               d["h"][r0:r1], d["edges"][r0:r1], ws)
            ev_kernel[p][c].record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(ev_kernel[p][c])
                out_edges[r0:r1].copy_(d["edges"][r0:r1], non_blocking=True)
                out_cand[r0:r1].copy_(d["cand"][r0:r1], non_blocking=True)
                out_unary[r0:r1].copy_(d["unary"][r0:r1], non_blocking=True)
                ev_out[p][c].record(copy_out)
        recorded[p] = True
        step_no[0] += 1

    def link_rate() -> float:
        """GB/s of the host link alone: the same chunked host-to-device copies as one e2e
        step, on the copy stream with nothing else running. One untimed pass wakes the link;
        three passes back to back are then timed together."""
        def copies():
            with torch.cuda.stream(copy_in):
                for c in range(nch):
                    r0, r1 = bounds[c], bounds[c + 1]
                    logits[r0:r1].copy_(logits_host[r0:r1], non_blocking=True)
                    hidden[r0:r1].copy_(hidden_host[r0:r1], non_blocking=True)
                    anchors[r0:r1].copy_(anchors_host[r0:r1], non_blocking=True)
        torch.cuda.synchronize(dev)
        copies()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(copy_in)
        for _ in range(3):
            copies()
        l1.record(copy_in)
        torch.cuda.synchronize(dev)
        return 3 * h2d / (l0.elapsed_time(l1) / 1e3) / 1e9

    link_before = link_rate()
    e2e_step()
    e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    stream.wait_stream(copy_out)                 # the last step's outputs are on the host
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, e2e_value = aggregate(e0.elapsed_time(e1) / args.e2e_steps, w.edges_per_call, world)
    # The bound of the e2e number: the faster of two measurements of the link, taken just
    # before and just after the e2e loop. Both are reported: host memory and its link are shared
    # with the machine's other jobs, and a drop between the two shows their copies.
    link_after = link_rate()
    link_gbs = max(link_before, link_after)

    if rank == 0:
        topk_ms = statistics.mean(s[1] for s in stages)
        proj_ms = statistics.mean(s[0] for s in stages)
        edge_ms = statistics.mean(s[2] for s in stages)
        b = w.algorithmic_bytes()
        topk_bytes = b["logits"] + b["ids_unary_out"]
        peaks = measured_peaks()
        achieved = topk_bytes / (topk_ms / 1e3) / 1e9
        traffic = profiled_traffic(w)
        total_bytes = sum(b.values())
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32",
            "dtype_detail": "f32 logits compared in f32; projection and edges: bf16 inputs, "
                            "f32 products and sums",
            "data": "synthetic (seeded, shapes and distributions of the workload)",
            "config": base_config(w, world),
            "roofline": {"bound": "hbm", "kernel": "topk_kernel", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes_per_launch": topk_bytes,
                         "peak_source": peaks["source"]},
            "fused_hbm": {"algorithmic_bytes_per_step": total_bytes,
                          "achieved_gbs": total_bytes / (ms_max / 1e3) / 1e9,
                          "frac": total_bytes / (ms_max / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "stages_ms": {"projection": proj_ms, "topk": topk_ms, "edges": edge_ms,
                          "source": stages_source},
            "launch_mode": "cuda_graph_replay" if graph is not None else "eager",
            "e2e": {"value": e2e_value, "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipeline_chunks": nch, "device_buffer_sets": 2,
                    "h2d_gbs_effective": h2d / (e2e_ms / 1e3) / 1e9,
                    "link_h2d_gbs_measured": link_gbs,
                    "link_h2d_gbs_before_after": [link_before, link_after],
                    "link_frac": h2d / (e2e_ms / 1e3) / 1e9 / link_gbs},
            "gpu_launches": 3 * args.steps,   # projection, top-k, edges per step
            "device_status": status,
            "clocks": clocks.summary(),
        }
        if world == 1 and not args.no_per_workload:
            # The pages' DFlash2BeamCandidateSelector.forward on the step's own candidates.
            line["forward"] = measure_forward(ds, w, dev, stream, args.steps, args.warmup, peaks,
                                              cand, unary, hidden, anchors, w_proj, pred_cb,
                                              succ_cb, h, edges)
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(inp)
        if world == 1 and not args.no_per_workload:
            # The other workloads through the same call: their own step times, HBM fractions
            # and the oracle over each of them in full. Not part of the timed region above.
            del logits, hidden, anchors, w_proj, pred_cb, succ_cb, cand, unary, h, edges, ws
            del logits_host, hidden_host, anchors_host, inp, sets
            torch.cuda.empty_cache()
            line["per_workload"] = {
                name: measure_workload(ds, wl.WORKLOADS[name], dev, stream, args.steps,
                                       args.warmup, rank, peaks["hbm_gbs"],
                                       with_cpu=not args.no_cpu_baseline)
                for name in wl.WORKLOAD_ORDER if name != w.name}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_forward(args, w: wl.Workload) -> None:
    """The selector's forward pass alone (projection, then edges; the pages'
    DFlash2BeamCandidateSelector.forward) on the workload's shapes, one GPU, no logits.

    Inputs: the workload's seeded hidden states, projection weight, codebooks and anchors,
    and seeded candidates (uniform ids, N(0, 1) unary values) standing in for the top-k's.
    L2 is flushed (by a read) before every call. About 0.4 GB on the device at gemma_large,
    so this is also the small case for full ncu captures of the projection and edges kernels.
    """
    import draft_candidate_selector_gb300 as ds
    dev = torch.device("cuda", dist_env()[2])
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hidden = wl._bf16_normal(0, wl._TAG_HIDDEN, (w.R, w.S, w.H), 1.0).to(dev)
    w_proj = wl._bf16_normal(0, wl._TAG_W, (w.rank, w.H), 1.0 / w.H ** 0.5).to(dev)
    pred_cb = wl._bf16_normal(0, wl._TAG_PRED, (w.V, w.rank), 1.0 / w.rank ** 0.5).to(dev)
    succ_cb = wl._bf16_normal(0, wl._TAG_SUCC, (w.V, w.rank), 1.0 / w.rank ** 0.5).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    anchors = torch.randint(0, w.V, (w.R,), generator=g, device=dev, dtype=torch.int32)
    cand = torch.randint(0, w.V, (w.R, w.S, w.K), generator=g, device=dev, dtype=torch.int32)
    unary = torch.randn((w.R, w.S, w.K), generator=g, device=dev)
    h = torch.empty((w.R, w.S, w.rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((w.R, w.S, w.K, w.K), dtype=torch.float32, device=dev)
    with ClockSampler(dev) as clocks:
        f = measure_forward(ds, w, dev, stream, args.steps, args.warmup, measured_peaks(), cand,
                            unary, hidden, anchors, w_proj, pred_cb, succ_cb, h, edges)
    print(json.dumps({
        "metric": "selector forward edge scores/s (R*S*K^2, given candidates)",
        "value": f["edge_scores_per_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": f["forward_ms"], "higher_is_better": True,
        "dtype": "bf16 x bf16 -> f32", "data": "synthetic (seeded)", "config": base_config(w, 1),
        "forward": f, "gpu_launches": 2 * args.steps,
        "device_status": ds.dflash_device_status(clear=True), "clocks": clocks.summary(),
    }), flush=True)


def run_lmhead(args, w: wl.Workload) -> None:
    """The candidate head straight from the LM head (no logits in memory), one GPU.

    Inputs: the workload's hidden states as the drafter's final hidden state, and a seeded
    synthetic LM head [V, H] bf16 ~ N(0, 1/sqrt(H)) drawn on the device. For context, the
    unfused route is timed too: a cuBLAS bf16 GEMM writing the logits, then this library's
    top-k over them (fp32 logits of the same shape). Last, the whole draft step from the LM
    head (dflash_selector_lmhead: projection, LM-head top-k, edges) with seeded synthetic
    projection weights and codebooks of the workload's rank.
    """
    import draft_candidate_selector_gb300 as ds
    dev = torch.device("cuda", dist_env()[2])
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hidden = wl._bf16_normal(0, wl._TAG_HIDDEN, (w.R, w.S, w.H), 1.0).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    lm_head = (torch.randn((w.V, w.H), generator=g, device=dev) / w.H ** 0.5).to(torch.bfloat16)
    cand = torch.empty((w.R, w.S, w.K), dtype=torch.int32, device=dev)
    unary = torch.empty((w.R, w.S, w.K), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, ds._native.load().dflash_lmhead_topk_workspace_bytes(w.R, w.S, w.V, w.K)),
                     dtype=torch.uint8, device=dev)

    def step():
        ds.dflash_lmhead_topk(hidden, lm_head, w.K, cand, unary, ws)

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    with ClockSampler(dev) as clocks:
        ms = timed(step, args.steps)
    status = ds.dflash_device_status(clear=True)
    if args.lmhead_only:
        # The LM-head top-k alone (hidden states and the LM head on the device, nothing else):
        # the small footprint a profiler capture of this kernel wants.
        print(json.dumps({
            "metric": "candidate-head rows/s from the LM head (R*S)", "value": w.rows / (ms / 1e3),
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16 x bf16 -> f32",
            "data": "synthetic (seeded)", "config": base_config(w, 1),
            "gpu_launches": args.steps, "device_status": status, "clocks": clocks.summary(),
        }), flush=True)
        return
    h2 = hidden.reshape(w.rows, w.H)
    gemm_ms = timed(lambda: torch.matmul(h2, lm_head.t()), max(3, args.steps // 4))
    logits = torch.empty((w.R, w.S, w.V), dtype=torch.float32, device=dev).normal_()
    topk_ms = timed(lambda: ds.dflash_topk_candidates(logits, w.K, cand, unary), max(3, args.steps // 4))
    del logits
    # The whole draft step from the LM head (projection, LM-head top-k, edges) in one call.
    w_proj = (torch.randn((w.rank, w.H), generator=g, device=dev) / w.H ** 0.5).to(torch.bfloat16)
    pred_cb = (torch.randn((w.V, w.rank), generator=g, device=dev) / w.rank ** 0.5).to(torch.bfloat16)
    succ_cb = (torch.randn((w.V, w.rank), generator=g, device=dev) / w.rank ** 0.5).to(torch.bfloat16)
    anchors = torch.randint(0, w.V, (w.R,), generator=g, device=dev, dtype=torch.int32)
    h_out = torch.empty((w.R, w.S, w.rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((w.R, w.S, w.K, w.K), dtype=torch.float32, device=dev)
    sel_ms = timed(lambda: ds.dflash_selector_lmhead(hidden, lm_head, w_proj, pred_cb, succ_cb,
                                                     anchors, w.K, cand, unary, h_out, edges, ws),
                   max(3, args.steps // 4))
    sustained = None
    if args.sustained:
        # Each of the fused kernel and the cuBLAS GEMM alone, back to back for about
        # args.sustained seconds with clocks sampled: under the power cap the clock settles
        # where the power allows, so work per cycle decides the rate.
        sustained = {}
        h2 = hidden.reshape(w.rows, w.H)
        for name, fn in [("lmhead_topk_kernel", step),
                         ("cublas_bf16_gemm", lambda: torch.matmul(h2, lm_head.t()))]:
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            n = max(5, int(args.sustained * 1e3 / max(a.elapsed_time(b), 1e-3)))
            with ClockSampler(dev) as ck:
                a.record(stream)
                for _ in range(n):
                    fn()
                b.record(stream)
                torch.cuda.synchronize(dev)
            s_ms = a.elapsed_time(b) / n
            ck_s = ck.summary() or {}
            tflops = 2.0 * w.rows * w.V * w.H / (s_ms / 1e3) / 1e12
            mhz = ck_s.get("sm_mhz")
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            sustained[name] = {
                "ms": s_ms, "tflops": tflops, "calls": n, "clocks": ck_s,
                "flop_per_sm_cycle": tflops * 1e12 / (sms * mhz * 1e6) if mhz else None}
    # End to end: each step copies its hidden states in from pinned host memory and its edge
    # scores out (the LM head, projection and codebooks stay resident, as model weights do).
    hidden_host = hidden.cpu().pin_memory()
    edges_host = torch.empty(edges.shape, dtype=edges.dtype).pin_memory()

    def e2e_step():
        hidden.copy_(hidden_host, non_blocking=True)
        ds.dflash_selector_lmhead(hidden, lm_head, w_proj, pred_cb, succ_cb, anchors, w.K, cand,
                                  unary, h_out, edges, ws)
        edges_host.copy_(edges, non_blocking=True)

    e2e_ms = timed(e2e_step, max(3, args.steps // 4))
    status |= ds.dflash_device_status(clear=True)
    flops = 2.0 * w.rows * w.V * w.H
    peak = None
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peak = float(json.load(f)["bf16_tflops_sustained"])
    achieved = flops / (ms / 1e3) / 1e12
    print(json.dumps({
        "metric": "candidate-head rows/s from the LM head (R*S)", "value": w.rows / (ms / 1e3),
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16 x bf16 -> f32",
        "data": "synthetic (seeded)", "config": base_config(w, 1),
        "roofline": {"bound": "tensor", "kernel": "lmhead_topk_kernel", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak if peak else None,
                     "traffic": None, "peak_source": "measured sustained bf16 (MEASURED_PEAKS.json)"},
        "unfused_reference": {"cublas_bf16_gemm_ms": gemm_ms, "logits_topk_ms": topk_ms,
                              "sum_ms": gemm_ms + topk_ms},
        "selector_lmhead": {"ms_per_step": sel_ms,
                            "edge_scores_per_s": w.rows * w.K * w.K / (sel_ms / 1e3),
                            "what": "projection, LM-head top-k and edges in one call",
                            "e2e": {"ms_per_step": e2e_ms,
                                    "edge_scores_per_s": w.rows * w.K * w.K / (e2e_ms / 1e3),
                                    "h2d_bytes_per_step": hidden_host.numel() * 2,
                                    "d2h_bytes_per_step": edges_host.numel() * 4}},
        "sustained": sustained,
        "gpu_launches": args.steps, "device_status": status, "clocks": clocks.summary(),
    }), flush=True)


def run_best_path(args, w: wl.Workload) -> None:
    """The best path through edge scores of the workload's shape (R, S, K), one GPU.

    Inputs: seeded N(0, 1) edge scores [R, S, K, K] and uniform candidate ids, on the device.
    --path-steps overrides S. The calls are captured once in a CUDA graph (20 per replay), so
    the time is the kernel's own, without host launch latency.
    """
    import draft_candidate_selector_gb300 as ds
    dev = torch.device("cuda", dist_env()[2])
    torch.cuda.set_device(dev)
    S = args.path_steps or w.S
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    per_replay = 20
    edges = [torch.randn((w.R, S, w.K, w.K), generator=g, device=dev) for _ in range(per_replay)]
    cand = torch.randint(0, w.V, (w.R, S, w.K), generator=g, device=dev, dtype=torch.int32)
    path = torch.empty((w.R, S), dtype=torch.int32, device=dev)
    tokens = torch.empty((w.R, S), dtype=torch.int32, device=dev)
    score = torch.empty((w.R,), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            ds.dflash_best_path(edges[0], cand, path, tokens, score)
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for e in edges:
            ds.dflash_best_path(e, cand, path, tokens, score)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, args.steps // per_replay)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / (reps * per_replay)
    nbytes = w.R * S * w.K * w.K * 4
    print(json.dumps({
        "metric": "best paths/s (requests)", "value": w.R / (ms / 1e3), "unit": "requests/s",
        "n_gpus": 1, "steps": reps * per_replay, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "R": w.R, "S": S, "K": w.K,
                   "l2": "20 distinct edge tensors per replay"},
        "edge_bytes_per_call": nbytes, "achieved_gbs": nbytes / (ms / 1e3) / 1e9,
        "gpu_launches": reps * per_replay, "device_status": ds.dflash_device_status(clear=True),
    }), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemma_large", choices=wl.WORKLOAD_ORDER)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="request chunks the end-to-end loop pipelines copies and kernels over")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the forward pass and the other workloads after the headline")
    ap.add_argument("--lmhead", action="store_true",
                    help="time the candidate head straight from a synthetic LM head instead")
    ap.add_argument("--lmhead-only", action="store_true",
                    help="with --lmhead: the LM-head top-k alone, without the unfused route, "
                         "the draft step or the end-to-end timing")
    ap.add_argument("--sustained", type=float, default=0.0,
                    help="with --lmhead: also run the fused kernel and the cuBLAS GEMM back to "
                         "back for this many seconds each, sampling clocks and power")
    ap.add_argument("--forward", action="store_true",
                    help="time the selector's forward pass alone (projection, then edges) on "
                         "given candidates, without logits")
    ap.add_argument("--best-path", action="store_true",
                    help="time the best path through edge scores of the workload's shape instead")
    ap.add_argument("--path-steps", type=int, default=None,
                    help="with --best-path: override S")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the step captured once in a CUDA graph")
    ap.add_argument("--requests", type=int, default=None,
                    help="override R (a smaller case of the same shape, e.g. for ncu captures)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps, always
    w = wl.WORKLOADS[args.workload]
    if args.requests is not None:
        import dataclasses
        w = dataclasses.replace(w, R=args.requests,
                                description=f"{w.description}; R overridden to {args.requests}")
    if args.impl == "reference":
        run_reference(args, w)
    elif args.lmhead:
        run_lmhead(args, w)
    elif args.best_path:
        run_best_path(args, w)
    elif args.forward:
        run_forward(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
