"""Benchmark of the Prox sparse SwiGLU FFN decode path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--batch B] [--sparsity S] [--input-sparsity S_in] [--layers L]

Workload: one Llama-3-8B-shaped FFN layer (d_model 4096, d_ff 14336), bf16 weights
N(0, 0.02^2), inputs Student-t(4), 70% channel sparsity and 50% input sparsity, batch 1
(seeded synthetic data, see workloads/). A step is one pass of the whole hot path (input
selection, Stage-1 proxy GEMV + salience, top-k, Stage-2 gather GEMV + SwiGLU + down
projection) over one batch of tokens on one layer. Steps rotate over L independently seeded
layer copies (4 x 0.41 GB by default), so every step streams its weights from HBM rather
than from the 126 MB L2. The K timed steps are replayed from CUDA graphs on one stream and
timed with CUDA events; with torchrun each rank runs its own replica on its own GPU
(independent tokens, no collective on the data path) and the slowest rank's time counts.

One JSON line is printed (rank 0): the metric (tokens/s per layer), the Stage-2 kernel's
roofline fraction against the measured HBM copy bandwidth, the dense-FFN speedup, the
end-to-end number through the host-buffer entry point, SM clocks sampled during the timed
region, and the CPU oracle timed on a bounded sample on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse SwiGLU FFN decode tokens/s/layer"
UNIT = "tokens/s/layer"
WORKLOAD_KEY = 3   # the Llama-3-8B-shaped 4096 x 14336 layer of the workloads module


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--sparsity", type=float, default=0.7)
    ap.add_argument("--input-sparsity", type=float, default=0.5)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(v: float, world: int, device: str) -> float:
    """The maximum of v over all ranks (each rank's own v when running alone)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank units (weak scaling) and the
    job took the slowest rank's time."""
    return world * units_per_rank / seconds


def workload_name(batch, sparsity, s_in):
    return (f"llama3-8b-ffn-4096x14336-b{batch}-s{round(sparsity * 100)}"
            f"-in{round(s_in * 100)}")


def algorithmic_bytes(d, F, k_in_rows, k_rows, batch):
    """Bytes the method must move per step: kept int4 proxy rows (gate+up, one byte per
    channel), fp16 group scales of both proxies, the selected bf16 rows of W_gate, W_up and
    W_down^T, plus x, y, the mask and the salience."""
    G = d // 128
    return (k_in_rows * F + 4 * G * F + 6 * k_rows * d
            + batch * (8 * d + 8 * F) + 4 * batch * k_rows)


def stage2_bytes(d, k_rows, batch):
    return 6 * k_rows * d + batch * 8 * d + 4 * batch * k_rows


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [ln.split(",") for ln in out.strip().splitlines() if ln.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[4 + i].strip().lower() == "active"})
        under_load = [v for v in sm if smax and v >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(under_load) if under_load else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle

def cpu_oracle_rate(layer_mats, X, sparsity, s_in, seconds, threads=None):
    """Tokens/s of the CPU oracle's whole path on this host, over a bounded sample; with
    threads=1 the numerical libraries are limited to one thread for the sample."""
    import contextlib
    import numpy as np
    import oracle as O
    try:
        from threadpoolctl import threadpool_info, threadpool_limits
        limit = threadpool_limits(threads) if threads else contextlib.nullcontext()
    except Exception:
        threadpool_info, limit = None, contextlib.nullcontext()
    ol = O.prepare_layer(*(layer_mats[n].float().numpy() for n in ("w_gate", "w_up", "w_down")))
    n = 0
    with limit:
        if threadpool_info is not None:
            blas_threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
        else:
            blas_threads = threads or len(os.sched_getaffinity(0))
        t0 = time.perf_counter()
        while True:
            O.ffn_token(ol, np.asarray(X[n % len(X)]), sparsity, s_in)
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    return n / dt, n, dt, blas_threads


def run_reference(args):
    """The reference arm: the fp64 CPU oracle on the host cores, same workload, metric and
    unit as the GPU arm. A step is one token of the workload through the oracle's whole path
    (about a second each), so the timed steps are bounded by time rather than by --steps."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle as O
    import workloads as WL
    mats = WL.make_layer(WORKLOAD_KEY, 0)
    X = WL.make_tokens(WORKLOAD_KEY, range(max(args.tokens, args.batch)))
    d, F = mats["w_gate"].shape[1], mats["w_gate"].shape[0]
    ol = O.prepare_layer(*(mats[n].float().numpy() for n in ("w_gate", "w_up", "w_down")))
    warm = min(max(args.warmup, 0), 3)
    for i in range(warm):
        O.ffn_token(ol, np.asarray(X[i % len(X)]), args.sparsity, args.input_sparsity)
    budget = min(120.0, max(5.0, args.cpu_seconds * 4))
    rate, n, dt, threads = cpu_oracle_rate(mats, X, args.sparsity, args.input_sparsity, budget)
    sample = (f"{n} tokens of the {workload_name(args.batch, args.sparsity, args.input_sparsity)}"
              f" workload through the fp64 numpy oracle in {dt:.1f} s (tokens are independent, so "
              f"the rate holds for any batch); bounded by time: {args.steps} steps were requested")
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": 0,
            "steps": n, "warmup": warm, "ms_per_step": 1000.0 * dt / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args.batch, args.sparsity, args.input_sparsity),
                       "d_model": d, "d_ff": F, "batch": args.batch, "sparsity": args.sparsity,
                       "input_sparsity": args.input_sparsity,
                       "k": O.k_for(args.sparsity, F), "k_in": O.k_for(args.input_sparsity, d)},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def source_hash(names=None) -> str:
    """Hash of the CUDA sources `names` (file names under csrc/; all of them by default)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "free_sparse_swiglu_stage1_b300", "csrc")
    for name in sorted(names or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str) -> tuple[float | None, str | None]:
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken on
    the current sources of that kernel (its translation unit and the headers it includes,
    listed in the record)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None, None
    if not rec or rec.get("source_hash") != source_hash(rec.get("sources")):
        return None, None
    return rec.get("dram_bytes_per_launch"), rec.get("note")


def timed_graph_replays(torch, stream, graphs, barrier, name, per_graph=None):
    """Seconds for replaying `graphs` on `stream`, by CUDA events on that stream. The replays
    sit in an NVTX range called `name`, so a profiler can be limited to them. If per_graph is
    a list, the seconds of each replay (events between replays) are appended to it."""
    barrier()
    torch.cuda.synchronize()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
    torch.cuda.nvtx.range_push(name)
    with torch.cuda.stream(stream):   # replays go to the stream the events are on
        events[0].record(stream)
        for i, g in enumerate(graphs):
            g.replay()
            events[i + 1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier()
    if per_graph is not None:
        per_graph += [events[i].elapsed_time(events[i + 1]) / 1000.0 for i in range(len(graphs))]
    return events[0].elapsed_time(events[-1]) / 1000.0


def step_stats(chunk_seconds, chunk_steps):
    """Median, 10th and 90th percentile of the microseconds per step over replayed chunks of
    chunk_steps steps each (nearest-rank percentiles)."""
    per = sorted(1e6 * t / n for t, n in zip(chunk_seconds, chunk_steps) if n > 0)
    if not per:
        return None

    def pct(q):
        return per[min(len(per) - 1, max(0, int(round(q * (len(per) - 1)))))]
    return {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9), "chunks": len(per)}


def capture(torch, stream, fn, n):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    return g


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import free_sparse_swiglu_stage1_b300 as P
    import workloads as WL

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return reduce_max(v, world, "cuda")

    B, sp, s_in, L = args.batch, args.sparsity, args.input_sparsity, args.layers
    d, F = 4096, 14336
    k, k_in = P.prox_k_for(sp, F), P.prox_k_for(s_in, d)
    T = max(B, args.tokens // B * B)

    layers, mats0 = [], None
    for li in range(L):
        mats = WL.make_layer(WORKLOAD_KEY, li)
        if li == 0:
            mats0 = mats
        dev = {n: v.cuda() for n, v in mats.items() if n.startswith("w_")}
        layers.append(P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"]))
        del dev
    torch.cuda.synchronize()
    X_np = WL.make_tokens(WORKLOAD_KEY, range(rank * T, (rank + 1) * T))
    X = torch.from_numpy(X_np).cuda()
    Y = torch.empty_like(X)
    ws = P.prox_workspace(d, F, B)
    stream = torch.cuda.Stream()
    nb_batches = T // B
    # one token: input_quant, Stage 1, top-k, Stage 2, reduce; a batch adds split_x (the
    # tensor-core Stage 2 takes its activations as bf16 pairs)
    per_step_kernels = 5 if B == 1 else 6

    def step_fwd(i):
        li, t = i % L, (i // L) % nb_batches
        P.prox_ffn_forward(layers[li], X[t * B:(t + 1) * B], sp, s_in, ws,
                           y=Y[t * B:(t + 1) * B], stream=stream)

    def step_dense(i):
        li, t = i % L, (i // L) % nb_batches
        P.prox_dense_ffn(layers[li], X[t * B:(t + 1) * B], ws, y=Y[t * B:(t + 1) * B],
                         stream=stream)

    # masks of every (layer, token batch) pair, for timing Stage 2 alone
    cycle = L * nb_batches
    masks = []
    with torch.cuda.stream(stream):
        for i in range(cycle):
            li, t = i % L, (i // L) % nb_batches
            masks.append(P.prox_build_mask(layers[li], X[t * B:(t + 1) * B], sp, s_in, ws,
                                           stream=stream))

    def step_s2(i):
        li, t = i % L, (i // L) % nb_batches
        P.prox_sparse_ffn(layers[li], X[t * B:(t + 1) * B], masks[i % cycle], ws,
                          y=Y[t * B:(t + 1) * B], stream=stream)

    # warm-up (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step_fwd(i)
            step_dense(i)
            step_s2(i)
    torch.cuda.synchronize()
    st = P.prox_get_status(ws, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {P.prox_error_string(st)}")

    graph_steps = {}   # steps per captured graph

    def graphs_for(fn, K):
        chunk = min(K, 4 * cycle) if K > 0 else 0
        gs = []
        if chunk:
            g = capture(torch, stream, fn, chunk)
            graph_steps[id(g)] = chunk
            gs += [g] * (K // chunk)
            if K % chunk:
                g2 = capture(torch, stream, fn, K % chunk)
                graph_steps[id(g2)] = K % chunk
                gs.append(g2)
        return gs

    K = args.steps
    g_fwd = graphs_for(step_fwd, K)
    with torch.cuda.stream(stream):
        if g_fwd:
            g_fwd[0].replay()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    chunk_t = []
    t_fwd = max_over_ranks(timed_graph_replays(torch, stream, g_fwd, barrier, "timed_fwd",
                                               per_graph=chunk_t))
    chunk_n = []
    for g in g_fwd:
        chunk_n.append(graph_steps[id(g)])
    fwd_stats = step_stats(chunk_t, chunk_n)
    clocks = sampler.stop()
    del g_fwd

    K2 = min(K, 20000)
    g_s2 = graphs_for(step_s2, K2)
    t_s2 = max_over_ranks(timed_graph_replays(torch, stream, g_s2, barrier, "timed_stage2"))
    del g_s2
    Kd = min(K, 5000)
    g_d = graphs_for(step_dense, Kd)
    t_dense = max_over_ranks(timed_graph_replays(torch, stream, g_d, barrier, "timed_dense"))
    del g_d

    # end to end through the host-buffer entry point: H2D of x, the path, D2H of y, each step
    Ke = min(K, 3000)
    xh = torch.from_numpy(X_np).pin_memory()
    yh = torch.empty((B, d), dtype=torch.float32).pin_memory()
    for i in range(3):
        P.prox_ffn_forward_host(layers[i % L], xh[:B], sp, s_in, ws, y_host=yh, stream=stream)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(Ke):
        li, t = i % L, (i // L) % nb_batches
        P.prox_ffn_forward_host(layers[li], xh[t * B:(t + 1) * B], sp, s_in, ws, y_host=yh,
                                stream=stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(time.perf_counter() - t0)
    barrier()
    st = P.prox_get_status(ws, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status after timing: {P.prox_error_string(st)}")

    # bytes: for a batch the union of kept inputs and of masks is what is read
    if B == 1:
        rows_in, rows_ch = k_in, k
    else:
        kept_sizes, union_sizes = [], []
        for t in range(nb_batches):
            xb = X_np[t * B:(t + 1) * B]
            kept = set()
            for r in xb:
                kept |= set(np.argsort(-np.abs(r), kind="stable")[:k_in].tolist())
            kept_sizes.append(len(kept))
        for m in masks:
            union_sizes.append(len(np.unique(m.cpu().numpy())))
        rows_in, rows_ch = statistics.mean(kept_sizes), statistics.mean(union_sizes)
    path_bytes = algorithmic_bytes(d, F, rows_in, rows_ch, B)
    s2_bytes = stage2_bytes(d, rows_ch, B)

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm_peak = peaks.get("hbm_gbs", 6400.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    s_fwd = t_fwd / K
    s_s2 = t_s2 / K2
    s_dense = t_dense / Kd
    value = job_rate(world, B * K, t_fwd)
    achieved = s2_bytes / s_s2 / 1e9
    s2_kernel = "stage2_kernel" if B == 1 else "stage2_tc_kernel"
    traffic, traffic_note = profiled_traffic(s2_kernel)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, threads = cpu_oracle_rate(mats0, X_np, sp, s_in, args.cpu_seconds)
        rate1, n1, dt1, _ = cpu_oracle_rate(mats0, X_np, sp, s_in, args.cpu_seconds, threads=1)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "value_1core": rate1,
               "sample_1core": f"{n1} tokens in {dt1:.1f} s with the numerical libraries "
                               f"limited to one thread",
               "sample": f"{n} tokens (batch 1) of this workload, layer 0, through the fp64 "
                         f"numpy oracle in {dt:.1f} s"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": 1000.0 * s_fwd,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(B, sp, s_in), "d_model": d, "d_ff": F,
                   "batch": B, "sparsity": sp, "input_sparsity": s_in, "k": k, "k_in": k_in,
                   "layer_copies": L, "tokens": T,
                   "l2": f"inputs larger than L2: steps rotate over {L} layer copies "
                         f"({L * layers[0].buffer.numel() / 1e9:.2f} GB)",
                   "parallelism": f"replicas x{world}"},
        "us_per_layer": 1e6 * s_fwd,
        "us_per_layer_chunks": fwd_stats,
        "hbm_gbs_path": path_bytes / s_fwd / 1e9,
        "path_frac": path_bytes / s_fwd / 1e9 / hbm_peak,
        "algorithmic_bytes_per_step": path_bytes,
        "dense_us_per_layer": 1e6 * s_dense,
        "speedup_vs_dense": s_dense / s_fwd,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": (f"{s2_kernel} (+ its fixed-order partial-sum reduce"
                                + (")" if B == 1 else
                                   ", the batch's channel bitmap and the bf16 split of x)")),
                     "algorithmic_bytes_per_launch": s2_bytes,
                     "us_per_launch": 1e6 * s_s2,
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "traffic_note": traffic_note},
        "e2e": {"value": job_rate(world, B * Ke, t_e2e), "unit": UNIT,
                "h2d_bytes_per_step": B * d * 4, "d2h_bytes_per_step": B * d * 4,
                "api": "prox_ffn_forward_host (pinned host x/y, synchronous per step)"},
        "gpu_launches": K * per_step_kernels,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "dtype_detail": ("Stage 1: int4 x int8 products, exact int32 sums, fp32 double-float "
                         "combine; Stage 2: bf16 weights, fp32 activations and accumulation"
                         if B == 1 else
                         "Stage 1: int4 x int8 products, exact integer sums (dp4a, or f16 "
                         "tcgen05 MMAs with fp32 accumulation past one token tile), fp32 "
                         "double-float combine; Stage 2: bf16 tcgen05 MMAs, activations as "
                         "bf16 hi/lo pairs, fp32 accumulation"),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
