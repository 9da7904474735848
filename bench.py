"""Throughput of the sparse-MoE FFN forward on B300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one forward pass of the whole layer (router GEMM + selection,
dispatch, grouped expert GEMMs, shared experts, combine, balance statistic)
over one batch of seeded synthetic tokens.  The default workload is the
Qwen3-style layer: 16384 tokens, d_model 2048, 128 SwiGLU experts of width
768, top-8 with Zipf-skewed routing.

`value` is tokens/s with inputs resident in HBM, timed with CUDA events on
the launching stream over the K steps (each stage bracketed by its own
events, which also give the per-stage times and the roofline of the
dominant kernel).  `e2e` is the same metric through moe_forward_host: the
timed region includes the copy of x from page-locked host memory and the
copy of the output back.  The layer's working set (x, 1.2 GB of expert
weights, the 1.3 GB of grouped intermediates) is far larger than the 126 MB
L2, so no flush is needed between steps.  The decode workload (64 tokens)
reads 1.2 GB of expert weights per step, of which the L2 could keep the last
126 MB for the next step: there 512 MB are written between timed steps
(`--flush-l2` does the same for any workload) and each step is timed between
its own events.

Several GPUs run independent replicas (the layer has no exchange step
without a global capacity): one process per GPU under torchrun, a barrier
and the max over ranks around the timed region, and `value` counts the
tokens of all ranks.

On one GPU the run then times the DeepSeek-style layer (8192 tokens, two
shared experts) and the decode-shaped layer (64 tokens, L2 flushed between
steps) the same way and reports them under `config.workloads`: ms per step,
the expert GEMMs' TFLOP/s against the burst bf16 roof, and for the decode
layer the expert-weight bytes it streams per step against the HBM roof
(`--no-extra-workloads` skips them).

The tensor-core roofline divides by the measured burst bf16 figure (a
cuBLAS GEMM timed alone, at the clocks a millisecond-scale step runs at);
the power-capped sustained figure is reported beside it.

`--impl reference` times the CPU oracle (the only reference there is) on a
bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time


ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from routing_dispatch_expert_05_b300 import workloads as W  # noqa: E402

METRIC = "MoE-layer fwd tokens/s on 1 B300; grouped-GEMM % bf16 peak; routing % HBM BW"
# DRAM bytes (read + write) of one launch of the up projection at full size,
# from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` (one pass)
# on the current kernel: 1.346 GB read + 0.197 GB written on the Qwen3-style
# layer.  Reset to None whenever that kernel changes.
UP_TRAFFIC_BYTES = {"qwen3_moe": 1.346e9 + 0.197e9}
# the profiling recipe's fallback roofs, used only without MEASURED_PEAKS.json
# (it gives no sustained figure, so none is invented here)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}
# the workloads timed after the headline one, in the same run
EXTRA_WORKLOADS = ("deepseek_v3_block", "decode_stream")


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def build_library():
    """Build the CUDA library if it is out of date, once per host: ranks
    started together take a file lock in turn, so the first compiles and the
    others find the library up to date."""
    import fcntl
    from routing_dispatch_expert_05_b300 import build as B
    os.makedirs(B.BUILD_DIR, exist_ok=True)
    with open(os.path.join(B.BUILD_DIR, "build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return B.build()
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs.

    Samples are taken every 50 ms and carry nvidia-smi's own timestamp;
    `stop(region)` keeps those taken between the host times (time.time())
    that bracket the timed region, so an idle sample from before or after it
    does not enter the median.  If the region is shorter than one interval
    and no sample falls inside it, the nearest samples are reported with
    "in_region": 0."""
    FIELDS = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.out = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=open(self.out, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, region=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        try:
            with open(self.out) as f:
                text = f.read()
            os.unlink(self.out)
        except OSError:
            return None
        return self.summarise(text, self.uuid, region)

    @staticmethod
    def summarise(text, uuid=None, region=None):
        """Median SM clock, max clock and the throttle reasons seen, from
        nvidia-smi's CSV rows (the FIELDS order)."""
        import datetime
        rows = []
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            if uuid and parts[2] != uuid:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            rows.append((ts, parts))
        if not rows:
            return None
        chosen = rows
        in_region = None
        if region is not None:
            t0, t1 = region
            inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
            in_region = len(inside)
            if inside:
                chosen = inside
            else:
                # the region fell between two samples: the one before it and
                # the one after it
                timed = [r for r in rows if r[0] is not None]
                before = [r for r in timed if r[0] < t0][-1:]
                after = [r for r in timed if r[0] > t1][:1]
                chosen = before + after or rows
        num = lambda v: v.replace(".", "", 1).isdigit()
        sm = [float(p[3]) for _, p in chosen if num(p[3])]
        mx = [float(p[4]) for _, p in chosen if num(p[4])]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for _, p in chosen:
            for name, v in zip(names, p[7:11]):
                if v.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None,
               "reasons": sorted(reasons), "samples": len(chosen)}
        if in_region is not None:
            out["in_region"] = in_region
        return out


def oracle_sample(shape, inputs, target_s=12.0, max_tokens=None):
    """Time the CPU oracle's forward on the first n tokens of the workload
    (same layer parameters), n grown until one run takes ~target_s."""
    from oracle import moe_oracle as O
    n = min(64, shape.n_tokens)
    elapsed = 0.0
    while True:
        sub = inputs.first_tokens(n)
        t0 = time.perf_counter()
        O.forward(sub.shape, sub.values)
        elapsed = time.perf_counter() - t0
        if elapsed >= target_s / 4 or n >= shape.n_tokens or (max_tokens and n >= max_tokens):
            break
        n = min(shape.n_tokens, n * 4)
    return n, elapsed


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (ms) over all ranks of the default
    process group (the slowest rank sets the job's time); identity when no
    group is initialised.  Works on any backend (nccl on GPUs, gloo on CPU)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(tokens_per_rank, n_ranks, ms_step_max):
    """Whole-job throughput: every rank's tokens over the slowest rank's time
    (independent replicas, weak scaling)."""
    return tokens_per_rank * n_ranks / (ms_step_max * 1e-3)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [os.cpu_count() or 1])
    except Exception:
        return os.cpu_count() or 1


SMALL_WORKLOADS = ("toy_top2_fp32", "capacity_top2_fp32", "capacity_top2_bf16")


def single_thread_rate(shape, inputs, n_tokens):
    """The oracle's tokens/s on one thread (BLAS limited to one thread) for
    the first n_tokens; reported beside the all-core figure for the small
    workloads, where the threads have little to share."""
    from oracle import moe_oracle as O
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        return None
    sub = inputs.first_tokens(n_tokens)
    with threadpool_limits(limits=1):
        O.forward(sub.shape, sub.values)
        t0 = time.perf_counter()
        O.forward(sub.shape, sub.values)
        el = time.perf_counter() - t0
    return round(n_tokens / el, 2)


def host_description():
    """The host the CPU baseline ran on: logical CPUs, CPU model and the
    thread-count settings in the environment."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    env = {k: os.environ[k] for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
           if k in os.environ}
    return {"nproc": os.cpu_count(), "cpu_model": model, "thread_env": env}


def kernel_launches_per_step(shape):
    """Kernels the library launches for one moe_forward of this layer."""
    router = 2          # logits GEMM, selection (+ statistic, last CTA)
    dispatch = 4        # count, scan, rank, row copy
    experts = 2         # grouped up (with activation), grouped down
    shared = 2 if shape.n_shared > 0 else 0
    combine = 1
    return router + dispatch + experts + shared + combine


# ---------------------------------------------------------------- our arm
def staged_forward_times(M, cfg, x, weights, out, fstats, ws, steps, stream, flush=None):
    """K forwards through moe_forward_timed, one event before the layer and
    one after each stage.  Returns (total ms over the K steps, per-step
    stage durations {stage: [ms]}).  With `flush` (a byte tensor), it is
    written between steps and the total sums each step's own first-to-last
    event span, so the flushes are not timed."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(M.MOE_FORWARD_EVENTS)]
           for _ in range(steps)]
    for row in evs:
        for ev in row:
            ev.record(stream)          # creates the CUDA events before timing
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s_ in range(steps):
        if flush is not None:
            flush.fill_(s_ & 0xFF)
        M.moe_forward_timed(cfg, x, weights, out, fstats, ws, evs[s_])
    t_end.record(stream)
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    if flush is not None:
        total_ms = sum(evs[s_][0].elapsed_time(evs[s_][-1]) for s_ in range(steps))
    names = list(M.FORWARD_STAGES)
    stages = {name: [evs[s_][i].elapsed_time(evs[s_][i + 1]) for s_ in range(steps)]
              for i, name in enumerate(names)}
    return total_ms, stages


def workload_entry(shape, peaks, args, dev):
    """Time one more workload in this process (one GPU): ms per step, the
    expert GEMMs' TFLOP/s and fraction of the burst bf16 peak, the HBM-bound
    stages' GB/s; for the decode-shaped layer, the expert weights it streams
    per step and their rate against the HBM roof.  The decode layer is timed
    with 512 MB written between steps, so no weight stays in L2."""
    import torch
    from routing_dispatch_expert_05_b300 import moe as M
    inputs = W.make_inputs(shape)
    t = M.upload(inputs, device=dev)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    ws = M.MoEWorkspace(cfg, device=dev)
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    out = torch.empty(N, d, dtype=M.torch_dtype(shape.dtype), device=dev)
    kept = torch.empty(E, dtype=torch.int32, device=dev)
    fstats = M.make_stats(kept=kept)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        M.moe_forward(cfg, t["x"], weights, out, fstats, ws)
    flush = None
    if shape.name == "decode_stream":
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    total_ms, st = staged_forward_times(M, cfg, t["x"], weights, out, fstats, ws, args.steps,
                                        stream, flush)
    if M.moe_read_device_error(ws) != M.MOE_OK:
        raise RuntimeError(f"{shape.name}: device error word set")
    med = {name: statistics.median(v) for name, v in st.items()}
    m_kept = int(kept.sum().item())
    up_cols = 2 * F if shape.expert == W.EXPERT_SWIGLU else F
    gemm_flop = 2.0 * m_kept * d * (up_cols + F)
    gemm_ms = med["expert_up"] + med["expert_down"]
    bf16 = peaks["bf16_tflops"]
    ms = total_ms / args.steps
    entry = {"n_tokens": N, "d_model": d, "n_experts": E, "top_k": k, "d_ff": F,
             "n_shared": shape.n_shared, "ms_per_step": round(ms, 4),
             "tokens_per_s": round(N / (ms * 1e-3), 1),
             "stages_ms": {name: round(v, 4) for name, v in med.items()},
             "expert_gemm_tflops": round(gemm_flop / (gemm_ms * 1e-3) / 1e12, 1),
             "expert_gemm_frac_of_burst_bf16": round(
                 gemm_flop / (gemm_ms * 1e-3) / 1e12 / bf16, 4)}
    if shape.n_shared > 0:
        sf = 2.0 * N * d * 3 * shape.n_shared * shape.d_ff_shared
        entry["shared_tflops"] = round(sf / (med["shared"] * 1e-3) / 1e12, 1)
    # the same forward replayed from a CUDA graph (how a decode loop runs
    # it: no per-launch host cost, no events between stages), each replay
    # timed between its own events, after the flush when there is one
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                M.moe_forward(cfg, t["x"], weights, out, fstats, ws)
        stream.wait_stream(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        spans = []
        for s_ in range(args.steps):
            if flush is not None:
                flush.fill_(s_ & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            spans.append((a, b))
        torch.cuda.synchronize()
        graph_ms = sum(a.elapsed_time(b) for a, b in spans) / args.steps
        entry["graph_ms_per_step"] = round(graph_ms, 4)
        entry["graph_tokens_per_s"] = round(N / (graph_ms * 1e-3), 1)
    except Exception as exc:  # report, do not hide, a capture failure
        graph_ms = None
        entry["graph_ms_per_step"] = f"capture failed: {exc}"
    if flush is not None:
        # expert weights the step streams: every expert some token chose
        idx = torch.empty(N, k, dtype=torch.int32, device=dev)
        wts = torch.empty(N, k, dtype=torch.float32, device=dev)
        M.moe_router_topk(cfg, t["x"], weights, None, idx, wts, None, ws)
        touched = int(torch.unique(idx).numel())
        wbytes = touched * up_cols * d * 2 + touched * d * F * 2
        entry["l2"] = "flushed between timed steps (512 MB written)"
        entry["experts_touched"] = touched
        entry["weight_bytes_per_step"] = wbytes
        entry["weight_gbs_expert_gemms"] = round(wbytes / (gemm_ms * 1e-3) / 1e9, 1)
        entry["weight_gbs_step"] = round(wbytes / (ms * 1e-3) / 1e9, 1)
        entry["hbm_frac_expert_gemms"] = round(wbytes / (gemm_ms * 1e-3) / 1e9 /
                                               peaks["hbm_gbs"], 4)
        entry["hbm_frac_step"] = round(wbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
        if graph_ms is not None:
            entry["weight_gbs_graph"] = round(wbytes / (graph_ms * 1e-3) / 1e9, 1)
            entry["hbm_frac_graph"] = round(wbytes / (graph_ms * 1e-3) / 1e9 /
                                            peaks["hbm_gbs"], 4)
    del t, ws, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_ours(args, shape, peaks, peaks_kind):
    import torch
    import torch.distributed as dist
    from routing_dispatch_expert_05_b300 import moe as M

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)            # before the group, so NCCL binds this GPU
    dev = torch.device("cuda", local)
    if ws_n > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    inputs = W.make_inputs(shape)
    t = M.upload(inputs, device=dev)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    ws = M.MoEWorkspace(cfg, device=dev)
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    td = M.torch_dtype(shape.dtype)
    es = 2 if shape.dtype == W.DTYPE_BF16 else 4
    x = t["x"]
    out = torch.empty(N, d, dtype=td, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    kept = torch.empty(E, dtype=torch.int32, device=dev)
    dropped = torch.empty(E, dtype=torch.int32, device=dev)
    bal = torch.empty(1, dtype=torch.float32, device=dev)
    fstats = M.make_stats(counts=counts, kept=kept, dropped=dropped, balance=bal)
    stream = torch.cuda.current_stream(dev)
    stages = [s_ for s_ in M.FORWARD_STAGES if s_ != "shared" or shape.n_shared > 0]

    def barrier():
        torch.cuda.synchronize(dev)
        if ws_n > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        M.moe_forward(cfg, x, weights, out, fstats, ws)
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    flush = None
    if args.flush_l2 or shape.name == "decode_stream":
        # written between the timed steps: 512 MB is four times the L2, so no
        # weight one step reads is still cached for the next
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    barrier()
    h_start = time.time()
    # one event before the layer and one after each stage, per step
    total_ms, st_times = staged_forward_times(M, cfg, x, weights, out, fstats, ws, args.steps,
                                              stream, flush)
    barrier()
    h_end = time.time()
    clocks = sampler.stop(region=(h_start, h_end))
    stage_ms = {name: statistics.median(st_times[name]) for name in stages}
    stage_mean = {name: sum(st_times[name]) / args.steps for name in stages}
    ms_step = max_over_ranks([total_ms / args.steps], device=dev)[0]

    # the plain moe_forward call, eager and replayed from a CUDA graph
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        M.moe_forward(cfg, x, weights, out, fstats, ws)
    f1.record(stream)
    barrier()
    fwd_ms = f0.elapsed_time(f1) / args.steps
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                M.moe_forward(cfg, x, weights, out, fstats, ws)
        stream.wait_stream(cap)
        for _ in range(2):
            g.replay()
        barrier()
        f0.record(stream)
        for _ in range(args.steps):
            g.replay()
        f1.record(stream)
        barrier()
        graph_ms = f0.elapsed_time(f1) / args.steps
    except Exception as exc:  # report, do not hide, a capture failure
        graph_ms = f"capture failed: {exc}"

    # end to end through moe_forward_host: H2D of x and D2H of out inside
    xh = x.cpu().pin_memory()
    oh = torch.empty(N, d, dtype=td).pin_memory()
    for _ in range(2):
        M.moe_forward_host(cfg, xh, weights, oh, fstats, ws)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        M.moe_forward_host(cfg, xh, weights, oh, fstats, ws)
    e1.record(stream)
    barrier()
    e2e_ms, fwd_ms = max_over_ranks([e0.elapsed_time(e1) / args.steps, fwd_ms], device=dev)
    err = M.moe_read_device_error(ws)
    if err != M.MOE_OK:
        raise RuntimeError(f"device error word set: {M.STATUS_NAMES.get(err, err)}")

    # roofline of the dominant kernel: the grouped up projection (2/3 of the
    # routed FLOPs): 2 * d * (2F for SwiGLU, F otherwise) per kept assignment
    m_kept = int(kept.sum().item())
    up_cols = 2 * F if shape.expert == W.EXPERT_SWIGLU else F
    up_flop = 2.0 * m_kept * d * up_cols
    down_flop = 2.0 * m_kept * F * d
    up_ms = stage_mean["expert_up"]
    # the step is a millisecond-scale burst: its roof is the burst bf16 figure
    # (a cuBLAS GEMM timed alone); the power-capped sustained figure, where
    # measured, is reported beside it
    peak_tf = peaks["bf16_tflops"]
    sustained_tf = peaks.get("bf16_tflops_sustained")
    achieved = up_flop / (up_ms * 1e-3) / 1e12
    traffic = args.up_traffic_bytes
    if traffic is None:
        traffic = UP_TRAFFIC_BYTES.get(shape.name)
    roofline = {"bound": "tensor", "kernel": "grouped expert up-projection (tcgen05)",
                "achieved": round(achieved, 1), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(achieved / peak_tf, 4),
                "peak_kind": f"{peaks_kind} burst bf16",
                "algorithmic_flop_per_launch": up_flop,
                "traffic": traffic}
    if sustained_tf:
        roofline["frac_of_sustained"] = round(achieved / sustained_tf, 4)
    hbm = peaks["hbm_gbs"]
    # algorithmic bytes of the HBM-bound stages (per step)
    router_bytes = N * d * es + E * d * es + N * k * 8
    # idx read twice, row_of_slot and token_of_row written, rows copied
    dispatch_bytes = N * k * 4 * 4 + N * d * es + m_kept * d * es
    # expert outputs: fp16 + one exponent byte per 32 columns (bf16 layers,
    # already weighted, in slot order) or fp32 with the weights read separately
    if shape.dtype == W.DTYPE_BF16:
        y_row_bytes = d * 2 + (d + 31) // 32
        slot_bytes = N * k * 4                     # row_of_slot (drop flags)
    else:
        y_row_bytes = d * 4
        slot_bytes = N * k * 8                     # row_of_slot and w
    combine_bytes = m_kept * y_row_bytes + N * d * es + slot_bytes + \
        (N * d * 4 if shape.n_shared > 0 else 0)
    stage_report = {}
    for name in stages:
        entry = {"ms": round(stage_ms[name], 4)}
        if name == "expert_up":
            entry["tflops"] = round(up_flop / (stage_ms[name] * 1e-3) / 1e12, 1)
        if name == "expert_down":
            entry["tflops"] = round(down_flop / (stage_ms[name] * 1e-3) / 1e12, 1)
        if name == "shared":
            sf = 2.0 * N * d * 3 * shape.n_shared * shape.d_ff_shared
            entry["tflops"] = round(sf / (stage_ms[name] * 1e-3) / 1e12, 1)
        if name in ("router", "dispatch", "combine"):
            b = {"router": router_bytes, "dispatch": dispatch_bytes,
                 "combine": combine_bytes}[name]
            gbs = b / (stage_ms[name] * 1e-3) / 1e9
            entry["gbs"] = round(gbs, 1)
            entry["hbm_frac"] = round(gbs / hbm, 4)
        stage_report[name] = entry
    grouped_flop = up_flop + down_flop
    grouped_ms = stage_ms["expert_up"] + stage_ms["expert_down"]

    res = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(N, ws_n, ms_step), 1),
        "unit": "tokens/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if shape.dtype == W.DTYPE_BF16 else "f32",
        "data": "synthetic (seeded PCG64; random-init weights of the layer's shapes)",
        "config": {"workload": shape.name, "n_tokens": N, "d_model": d,
                   "n_experts": E, "top_k": k, "d_ff": F,
                   "n_shared": shape.n_shared, "route": shape.route,
                   "capacity_factor": shape.capacity_factor,
                   "parallelism": f"replicas x{ws_n}",
                   "l2": ("flushed between timed steps (512 MB written), steps timed "
                          "between their own events" if flush is not None else
                          "working set > 126 MB L2 (no flush needed)"),
                   "forward_api_ms_per_step": round(fwd_ms, 4),
                   "forward_graph_ms_per_step": (round(graph_ms, 4)
                                                 if isinstance(graph_ms, float) else graph_ms),
                   "timed_api": "moe_forward_timed (events between stages)",
                   "timed_region": {
                       "seconds": round(h_end - h_start, 3),
                       "regime": ("power-capped (sw_power_cap seen in the region)"
                                  if clocks and "sw_power_cap" in clocks.get("reasons", [])
                                  else "no power cap seen in the region"),
                       "note": "the default 200 steps are long enough for clock samples "
                               "inside the region; short bursts (--steps 20) run faster "
                               "before the power cap engages"},
                   "grouped_gemm_tflops": round(grouped_flop / (grouped_ms * 1e-3) / 1e12, 1),
                   "grouped_gemm_frac_of_burst": round(
                       grouped_flop / (grouped_ms * 1e-3) / 1e12 / peak_tf, 4),
                   "stages": stage_report},
        "roofline": roofline,
        "e2e": {"value": round(job_tokens_per_s(N, ws_n, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": N * d * es, "d2h_bytes_per_step": N * d * es,
                "ms_per_step": round(e2e_ms, 4), "api": "moe_forward_host"},
        "gpu_launches": kernel_launches_per_step(shape) * args.steps,
        "clocks": clocks,
    }
    if sustained_tf:
        res["config"]["grouped_gemm_frac_of_sustained"] = round(
            grouped_flop / (grouped_ms * 1e-3) / 1e12 / sustained_tf, 4)
    if not args.no_extra_workloads and ws_n == 1:
        # the other large workloads, timed in the same run on the same GPU
        # (the other configurations are parity cases)
        extra = {}
        for name in EXTRA_WORKLOADS:
            if name != shape.name:
                extra[name] = workload_entry(W.WORKLOADS[name], peaks, args, dev)
        # the backward pass of the same layer (moe_backward, routing held
        # fixed), outside the timed forward steps
        if (shape.expert == W.EXPERT_SWIGLU and shape.dtype == W.DTYPE_BF16 and
                shape.n_shared == 0 and not shape.has_bias):
            extra["backward_" + shape.name] = backward_times(shape, peaks, steps=10, warmup=3)
        res["config"]["workloads"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        n_s, el = oracle_sample(shape, inputs, target_s=args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(n_s / el, 2), "unit": "tokens/s",
                               "cores": blas_threads(), "kind": "oracle",
                               "host": host_description(),
                               "sample": f"first {n_s} tokens of the workload, one "
                                         f"forward, {el:.2f} s"}
        if shape.name in SMALL_WORKLOADS:
            res["cpu_baseline"]["single_thread_value"] = single_thread_rate(shape, inputs, n_s)
    if ws_n > 1:
        dist.barrier()
        dist.destroy_process_group()
    return res, rank


# ---------------------------------------------------------- reference arm
def run_reference(args, shape):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None, rank
    inputs = W.make_inputs(shape)
    from oracle import moe_oracle as O
    # each step's sample shrinks with the step count, so that the whole run
    # stays near a minute and a half of CPU time
    per_step = min(args.cpu_seconds / 2, 90.0 / (args.steps + args.warmup))
    n_s, el = oracle_sample(shape, inputs, target_s=max(0.05, per_step),
                            max_tokens=args.ref_tokens)
    sub = inputs.first_tokens(n_s)
    for _ in range(args.warmup):
        O.forward(sub.shape, sub.values)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        O.forward(sub.shape, sub.values)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    v = round(n_s / sec, 2)
    cores = blas_threads()
    res = {
        "impl": "reference",
        "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.dtype == W.DTYPE_BF16 else "f32",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": shape.name, "n_tokens": shape.n_tokens,
                   "sample_tokens": n_s},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "host": host_description(),
                         "sample": f"first {n_s} tokens of the workload per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    if shape.name in SMALL_WORKLOADS:
        res["cpu_baseline"]["single_thread_value"] = single_thread_rate(shape, inputs, n_s)
    return res, rank


def backward_times(shape, peaks, steps, warmup):
    """Time moe_backward (one GPU): recompute + data and weight gradients.

    Algorithmic FLOPs per step, SwiGLU experts: the recomputed g, u (2 d F)
    per kept assignment, the data gradients dh (d F) and dx_perm (2 d F), the
    weight gradients dW2 (d F) and dW1, dW3 (2 d F) -- 16 d F FLOP per
    assignment (two each per multiply-add) -- plus the router's three
    N x E x d products.  The expert outputs y are not recomputed: the routing
    weights' gradient <dout, y> is taken as <dout W2, h>, a row dot of the
    dh product with h, so no down projection is counted or run.
    """
    import torch
    from routing_dispatch_expert_05_b300 import moe as M

    inputs = W.make_inputs(shape)
    t = M.upload(inputs)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    gen = torch.Generator(device="cuda").manual_seed(7)
    dout = torch.randn(N, d, device="cuda", generator=gen).to(torch.bfloat16)
    f32 = lambda *s_: torch.empty(s_, dtype=torch.float32, device="cuda")
    g = dict(dx=f32(N, d), d_w_router=f32(E, d), d_w1=f32(E, F, d), d_w3=f32(E, F, d),
             d_w2=f32(E, d, F))
    if "b_router" in inputs.values:
        g["d_b_router"] = f32(E)
    grads = M.make_grads(**g)
    ws = M.MoEWorkspace(cfg, backward=True)
    for _ in range(warmup):
        M.moe_backward(cfg, t["x"], weights, dout, 1.0, grads, ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        M.moe_backward(cfg, t["x"], weights, dout, 1.0, grads, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flop = 16.0 * d * F * N * k + 3 * 2.0 * N * E * d
    tflops = flop / (ms * 1e-3) / 1e12
    assert M.moe_read_device_error(ws) == M.MOE_OK
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(N / (ms * 1e-3), 1),
            "gemm_tflops_effective": round(tflops, 1),
            "frac_of_burst_bf16": round(tflops / peaks["bf16_tflops"], 4),
            "steps": steps, "warmup": warmup}


def run_backward(args, shape, peaks, peaks_kind):
    """Time moe_backward alone (one GPU) as the bench line's metric."""
    bt = backward_times(shape, peaks, args.steps, args.warmup)
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    return {"metric": "MoE-layer bwd tokens/s on 1 B300 (routing held fixed)",
            "value": bt["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": bt["ms_per_step"],
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": shape.name, "n_tokens": N, "d_model": d, "n_experts": E,
                       "top_k": k, "d_ff": F},
            "gemm_tflops_effective": bt["gemm_tflops_effective"],
            "frac_of_burst_bf16": bt["frac_of_burst_bf16"],
            "peak_kind": f"{peaks_kind} burst bf16"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="qwen3_moe", choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=1024)
    ap.add_argument("--up-traffic-bytes", type=float, default=None,
                    help="DRAM bytes per launch of the up projection from an ncu capture")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the token count (smaller cases for profiler captures)")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write 512 MB between timed steps (always on for decode_stream)")
    ap.add_argument("--backward", action="store_true",
                    help="time moe_backward instead of the forward (one GPU)")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the chosen workload (not also the DeepSeek-style and "
                         "decode layers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    shape = W.WORKLOADS[args.workload]
    if args.tokens is not None and args.tokens != shape.n_tokens:
        shape = shape.replace(name=f"{shape.name}@{args.tokens}tok", n_tokens=args.tokens)
    if args.impl == "reference":
        res, rank = run_reference(args, shape)
    else:
        build_library()
        peaks, kind = load_peaks()
        if args.backward:
            res, rank = run_backward(args, shape, peaks, kind), 0
        else:
            res, rank = run_ours(args, shape, peaks, kind)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
