"""Benchmark of the Prox sparse SwiGLU FFN decode path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5] [--batch B] [--sparsity S] [--input-sparsity S_in]
                    [--layers L]

Workloads (seeded synthetic data, see workloads/):
  1  1024 x 2816 layer, N(0,1) inputs with 1% x20 outliers, 50% channel / 50% input sparsity
  2  Llama-2-7B-shaped 4096 x 11008 layer, per-channel LogNormal weight scales, Student-t(4)
  3  Llama-3-8B-shaped 4096 x 14336 layer, Student-t(4), 70% / 50% (the default)
  4  decode step through 32 independently seeded 4096 x 14336 layers with a unit-gain RMSNorm
     between them (one step = one token through all 32 layers)
  5  Llama-2-70B-shaped 8192 x 28672 layer, per-channel LogNormal scales, Student-t(3)
A step is one pass of the whole hot path (input selection, Stage-1 proxy GEMV + salience,
top-k, Stage-2 gather GEMV + SwiGLU + down projection) over one batch of tokens on one layer
(on all 32 layers for workload 4). Steps rotate over independently seeded layer copies whose
total size is several times the 126 MB L2, so every step streams its weights from HBM. The K
timed steps are replayed from CUDA graphs on one stream and timed with CUDA events on that
stream; with torchrun each rank runs its own replica on its own GPU (independent tokens, no
collective on the data path) and the slowest rank's time counts.

One JSON line is printed (rank 0): the metric (tokens/s per layer) over exactly the K timed
steps, the per-chunk spread of a longer run of the same graph, the Stage-2 kernel's roofline
fraction against the measured HBM copy bandwidth, the dense-FFN speedup, the end-to-end
number through the host-buffer entry point, SM clocks sampled during the timed region, and
the CPU oracle timed on a bounded sample on the host cores.
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
DEFAULT_WORKLOAD = 3   # the Llama-3-8B-shaped 4096 x 14336 layer
L2_BYTES = 126 * 2 ** 20
CHAIN_WORKLOAD = 4     # the 32-layer stack


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 20000; 400 for the 32-layer stack)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, choices=[1, 2, 3, 4, 5], default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--sparsity", type=float, default=None)
    ap.add_argument("--input-sparsity", type=float, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="layer copies the steps rotate over (default: enough for 3x L2)")
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="Stage-2 rows as FP8 E4M3 with row scales (single token only)")
    ap.add_argument("--spread-ms", type=float, default=300.0,
                    help="wall time of the extra chunked run that gives the p10/p50/p90 spread")
    ap.add_argument("--allocate", type=float, nargs="*", default=None,
                    help="fit the path's cost model to measured times, then time the sparsity "
                         "allocation prox_choose_sparsity picks for these target effective sparsities")
    ap.add_argument("--window", type=int, default=None,
                    help="32-layer stack only: keep the Stage-1 proxies in pinned host memory "
                         "and page them through this many device slots (prox_window_*)")
    return ap.parse_args(argv)


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


# ----------------------------------------------------------------------------- workload

def resolve(args) -> dict:
    """The workload's shape and the run's batch, sparsities, layer copies and chain depth."""
    import workloads as WL
    w = WL.WORKLOADS[args.workload]
    batch = args.batch if args.batch is not None else w.batches[0]
    sp = args.sparsity if args.sparsity is not None else (0.7 if 0.7 in w.sparsities
                                                          else w.sparsities[0])
    s_in = args.input_sparsity if args.input_sparsity is not None else w.input_sparsity
    chain = args.workload == CHAIN_WORKLOAD
    d, F = w.d_model, w.d_ff
    packed = d * F + 4 * (d // 128) * F + (3 * d + 16 if getattr(args, "fp8", False) else 6 * d) * F
    if chain:
        layers = w.layers
    elif args.layers is not None:
        layers = args.layers
    else:
        layers = max(4, math.ceil(3 * L2_BYTES / packed))
    name = (f"{w.name}-b{batch}-s{round(sp * 100)}-in{round(s_in * 100)}"
            + ("-fp8" if getattr(args, "fp8", False) else ""))
    row = 3 * d + 16 if getattr(args, "fp8", False) else 6 * d
    return {"key": args.workload, "name": name, "d": d, "F": F, "batch": batch,
            "sparsity": sp, "input_sparsity": s_in, "layers": layers, "chain": chain,
            "depth": w.layers if chain else 1, "packed_bytes": packed, "row_bytes": row,
            "fp8": bool(getattr(args, "fp8", False))}


def workload_config(cfg: dict, world: int, tokens: int, k: int, k_in: int) -> dict:
    """The `config` object of the JSON line (identical for both arms; k and k_in come from
    the arm's own implementation of the kept-count rule)."""
    c = {"workload": cfg["name"], "d_model": cfg["d"], "d_ff": cfg["F"],
         "batch": cfg["batch"], "sparsity": cfg["sparsity"],
         "input_sparsity": cfg["input_sparsity"], "k": k, "k_in": k_in,
         "layer_copies": cfg["layers"], "tokens": tokens,
         "l2": (f"inputs larger than L2: steps rotate over {cfg['layers']} layer copies "
                f"({cfg['layers'] * cfg['packed_bytes'] / 1e9:.2f} GB)"),
         "parallelism": f"replicas x{world}"}
    if cfg["chain"]:
        c["layers_per_step"] = cfg["depth"]
        c["l2"] = (f"inputs larger than L2: each step runs through {cfg['depth']} layers "
                   f"({cfg['depth'] * cfg['packed_bytes'] / 1e9:.2f} GB)")
    return c


def algorithmic_bytes(d, F, k_in_rows, k_rows, batch, row_bytes=None):
    """Bytes the method must move per layer pass: kept int4 proxy rows (gate+up, one byte per
    channel), fp16 group scales of both proxies, the selected channels' Stage-2 rows (bf16
    W_gate, W_up and W_down^T rows: 6 d bytes; FP8 rows with scales: 3 d + 16), plus x, y,
    the mask and the salience."""
    G = d // 128
    rb = 6 * d if row_bytes is None else row_bytes
    return (k_in_rows * F + 4 * G * F + rb * k_rows
            + batch * (8 * d + 8 * F) + 4 * batch * k_rows)


def stage2_bytes(d, k_rows, batch, row_bytes=None):
    rb = 6 * d if row_bytes is None else row_bytes
    return rb * k_rows + batch * 8 * d + 4 * batch * k_rows


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None

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
        return summarize_clocks(out)


def summarize_clocks(text: str) -> dict | None:
    rows = [ln.split(",") for ln in text.strip().splitlines() if ln.count(",") >= 7]
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

def cpu_oracle_rate(layer_mats, X, sparsity, s_in, seconds, threads=None, max_tokens=None):
    """Tokens/s of the CPU oracle's whole path on this host, over a bounded sample (at least
    one token, then until `seconds` have passed or max_tokens are done); with threads=1 the
    numerical libraries are limited to one thread for the sample."""
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
            if time.perf_counter() - t0 >= seconds or (max_tokens and n >= max_tokens):
                break
        dt = time.perf_counter() - t0
    return n / dt, n, dt, blas_threads


def run_reference(args):
    """The reference arm: the fp64 CPU oracle on the host cores, on the GPU arm's workload,
    config, metric and unit. A step is one batch of the workload's tokens through the oracle's
    whole path (for the 32-layer stack: one token through every layer, RMSNorm between); W
    untimed steps, then exactly K timed steps, unless K steps would run past a four-minute
    budget, in which case the steps that fit are timed and the line says so."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle as O
    import workloads as WL
    cfg = resolve(args)
    B = cfg["batch"]
    depth = cfg["depth"]
    n_layers = depth if cfg["chain"] else 1
    ols = []
    for li in range(n_layers):
        m = WL.make_layer(cfg["key"], li)
        ols.append(O.prepare_layer(*(m[n].float().numpy() for n in ("w_gate", "w_up", "w_down"))))
    T = max(B, args.tokens // B * B)
    X = WL.make_tokens(cfg["key"], range(T))
    nb = T // B

    def step(i):
        xs = X[(i % nb) * B:(i % nb + 1) * B]
        for x in xs:
            xc = np.asarray(x, np.float64)
            for li, ol in enumerate(ols):
                out = O.ffn_token(ol, xc.astype(np.float32), cfg["sparsity"],
                                  cfg["input_sparsity"])
                xc = O.rmsnorm(out["y"][None])[0] if li + 1 < len(ols) else out["y"]

    warm = max(0, args.warmup if args.warmup is not None else 3)
    warm = min(warm, 3)
    for i in range(warm):
        step(i)
    budget = 240.0
    t0 = time.perf_counter()
    n = 0
    per_step = None
    while n < args.steps:
        step(warm + n)
        n += 1
        el = time.perf_counter() - t0
        per_step = el / n
        if el + per_step > budget:
            break
    dt = time.perf_counter() - t0
    threads = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [threads])
    except Exception:
        pass
    units = n * B * (depth if cfg["chain"] else 1)
    rate = units / dt
    sample = (f"{n} steps of batch {B} ({n * B} tokens"
              + (f" x {depth} layers" if cfg["chain"] else "")
              + f") of the {cfg['name']} workload through the fp64 numpy oracle in {dt:.1f} s")
    if n < args.steps:
        sample += f"; {args.steps} steps were requested, stopped at the {budget:.0f} s budget"
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": 0,
            "steps": n, "warmup": warm, "ms_per_step": 1000.0 * dt / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(cfg, world, T, O.k_for(cfg["sparsity"], cfg["F"]),
                                      O.k_for(cfg["input_sparsity"], cfg["d"])),
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


def profiled_traffic(kernel: str, workload: str) -> tuple[float | None, str | None]:
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, if it was
    taken on the current sources of that kernel (its translation unit and the headers it
    includes, listed in the record)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel}@{workload}")
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
        # keep the device busy (about 0.2 ms, untimed) while the host submits the replays, so
        # the start event is not followed by the host's graph-submission latency
        torch.cuda._sleep(400_000)
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


def capture(torch, stream, fn, n, start=0):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(start, start + n):
            fn(i)
    return g


def plan_chunks(K: int, cycle: int) -> list[int]:
    """Step counts of the graphs that together replay exactly K steps: chunks of a whole
    number of rotation cycles (at most 4), then the remainder."""
    if K <= 0:
        return []
    chunk = max(1, min(K, 4 * cycle))
    out = [chunk] * (K // chunk)
    if K % chunk:
        out.append(K % chunk)
    return out


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

    cfg = resolve(args)
    B, sp, s_in, L = cfg["batch"], cfg["sparsity"], cfg["input_sparsity"], cfg["layers"]
    d, F, chain, depth = cfg["d"], cfg["F"], cfg["chain"], cfg["depth"]
    k, k_in = P.prox_k_for(sp, F), P.prox_k_for(s_in, d)
    T = max(B, args.tokens // B * B)

    layers, mats0 = [], None
    for li in range(L):
        mats = WL.make_layer(cfg["key"], li)
        if li == 0:
            mats0 = mats
        dev = {n: v.cuda() for n, v in mats.items() if n.startswith("w_")}
        layers.append(P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"],
                                          fp8=cfg["fp8"]))
        del dev
    torch.cuda.synchronize()
    X_np = WL.make_tokens(cfg["key"], range(rank * T, (rank + 1) * T))
    X = torch.from_numpy(X_np).cuda()
    Y = torch.empty_like(X)
    Xa = torch.empty((2, B, d), dtype=torch.float32, device="cuda")   # chain activations
    Ya = torch.empty((B, d), dtype=torch.float32, device="cuda")
    ws = P.prox_workspace(d, F, B)
    stream = torch.cuda.Stream()
    nb_batches = T // B

    def layer_of(i):
        return i % L

    def batch_of(i):
        return (i // L) % nb_batches if not chain else i % nb_batches

    def step_fwd(i):
        t = batch_of(i)
        if chain:
            xin = X[t * B:(t + 1) * B]
            for li in range(depth):
                out = Y[t * B:(t + 1) * B] if li + 1 == depth else Ya
                P.prox_ffn_forward(layers[li], xin, sp, s_in, ws, y=out, stream=stream)
                if li + 1 < depth:
                    P.prox_rmsnorm(Ya, 1e-6, out=Xa[li % 2], stream=stream)
                    xin = Xa[li % 2]
        else:
            P.prox_ffn_forward(layers[layer_of(i)], X[t * B:(t + 1) * B], sp, s_in, ws,
                               y=Y[t * B:(t + 1) * B], stream=stream)

    def step_dense(i):
        t = batch_of(i)
        if chain:
            xin = X[t * B:(t + 1) * B]
            for li in range(depth):
                out = Y[t * B:(t + 1) * B] if li + 1 == depth else Ya
                P.prox_dense_ffn(layers[li], xin, ws, y=out, stream=stream)
                if li + 1 < depth:
                    P.prox_rmsnorm(Ya, 1e-6, out=Xa[li % 2], stream=stream)
                    xin = Xa[li % 2]
        else:
            P.prox_dense_ffn(layers[layer_of(i)], X[t * B:(t + 1) * B], ws,
                             y=Y[t * B:(t + 1) * B], stream=stream)

    # the (layer, input, mask) triples of one rotation cycle, for timing Stage 2 alone; in the
    # chain each layer's input is the previous layer's normalised output
    cycle = nb_batches if chain else L * nb_batches
    s2_items = []
    with torch.cuda.stream(stream):
        for i in range(cycle):
            t = batch_of(i)
            if chain:
                xin = X[t * B:(t + 1) * B].clone()
                for li in range(depth):
                    idx = P.prox_build_mask(layers[li], xin, sp, s_in, ws, stream=stream)
                    s2_items.append((li, xin, idx))
                    y = P.prox_ffn_forward(layers[li], xin, sp, s_in, ws, stream=stream)
                    xin = P.prox_rmsnorm(y, 1e-6, stream=stream)
            else:
                xin = X[t * B:(t + 1) * B]
                idx = P.prox_build_mask(layers[layer_of(i)], xin, sp, s_in, ws, stream=stream)
                s2_items.append((layer_of(i), xin, idx))
    torch.cuda.synchronize()
    n_s2 = len(s2_items)

    def step_s2(i):
        li, xin, idx = s2_items[i % n_s2]
        P.prox_sparse_ffn(layers[li], xin, idx, ws, y=Ya, stream=stream)

    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for i in range(warm):
            step_fwd(i)
            step_dense(i)
            step_s2(i)
    torch.cuda.synchronize()
    st = P.prox_get_status(ws, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {P.prox_error_string(st)}")

    def graphs_for(fn, K, cyc):
        """Graphs replaying exactly K steps of fn, and the steps each one holds; every
        distinct graph is replayed once, untimed, before it is timed (graph upload)."""
        plan = plan_chunks(K, cyc)
        built = {}
        gs = []
        for n in plan:
            if n not in built:
                built[n] = capture(torch, stream, fn, n)
                with torch.cuda.stream(stream):
                    built[n].replay()
            gs.append(built[n])
        torch.cuda.synchronize()
        return gs, plan

    # launches per step, counted by the library while one step is recorded
    c0 = P.prox_launch_count()
    g_probe = capture(torch, stream, step_fwd, 1)
    launches_per_step = P.prox_launch_count() - c0
    del g_probe

    K = args.steps
    g_fwd, plan_fwd = graphs_for(step_fwd, K, cycle)
    with torch.cuda.stream(stream):   # bring the clocks up before the timed region
        for g in g_fwd[:2]:
            g.replay()
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
    t_fwd = max_over_ranks(timed_graph_replays(torch, stream, g_fwd, barrier, "timed_fwd"))
    # the spread: the same path replayed in chunks of about 1/20 of spread_ms each, for at
    # least spread_ms in total (outside the K-step measurement above)
    est = t_fwd / max(K, 1)
    per_chunk = max(1, int(args.spread_ms / 1000.0 / 20 / max(est, 1e-9)))
    per_chunk = min(per_chunk, 4 * cycle)
    g_sp = capture(torch, stream, step_fwd, per_chunk)
    with torch.cuda.stream(stream):
        g_sp.replay()
    chunk_t = []
    timed_graph_replays(torch, stream, [g_sp] * 20, barrier, "spread_fwd", per_graph=chunk_t)
    fwd_stats = step_stats(chunk_t, [per_chunk] * len(chunk_t))
    clocks = sampler.stop()
    del g_fwd, g_sp

    K2 = min(K * depth, 20000)
    g_s2, _ = graphs_for(step_s2, K2, n_s2)
    t_s2 = max_over_ranks(timed_graph_replays(torch, stream, g_s2, barrier, "timed_stage2"))
    del g_s2
    Kd = max(1, min(K, 5000 // depth))
    g_d, _ = graphs_for(step_dense, Kd, cycle)
    t_dense = max_over_ranks(timed_graph_replays(torch, stream, g_d, barrier, "timed_dense"))
    del g_d

    # end to end through the public API with host buffers: H2D of x, the path (all layers for
    # the stack), D2H of y, every step
    Ke = max(1, min(K, 3000 // depth))
    xh = torch.from_numpy(X_np).pin_memory()
    yh = torch.empty((B, d), dtype=torch.float32).pin_memory()

    def e2e_step(i):
        t = batch_of(i)
        if not chain:
            P.prox_ffn_forward_host(layers[layer_of(i)], xh[t * B:(t + 1) * B], sp, s_in, ws,
                                    y_host=yh, stream=stream)
            return
        with torch.cuda.stream(stream):
            xin = Xa[0]
            xin.copy_(xh[t * B:(t + 1) * B], non_blocking=True)
            for li in range(depth):
                P.prox_ffn_forward(layers[li], xin, sp, s_in, ws, y=Ya, stream=stream)
                if li + 1 < depth:
                    P.prox_rmsnorm(Ya, 1e-6, out=Xa[(li + 1) % 2], stream=stream)
                    xin = Xa[(li + 1) % 2]
            yh.copy_(Ya, non_blocking=True)
        stream.synchronize()

    for i in range(3):
        e2e_step(i)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(Ke):
        e2e_step(i)
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
        kept_sizes = []
        for t in range(nb_batches):
            kept = set()
            for r in X_np[t * B:(t + 1) * B]:
                kept |= set(np.argsort(-np.abs(r), kind="stable")[:k_in].tolist())
            kept_sizes.append(len(kept))
        union_sizes = [len(np.unique(it[2].cpu().numpy())) for it in s2_items]
        rows_in, rows_ch = statistics.mean(kept_sizes), statistics.mean(union_sizes)
    path_bytes = algorithmic_bytes(d, F, rows_in, rows_ch, B, cfg["row_bytes"]) * depth
    s2_bytes = stage2_bytes(d, rows_ch, B, cfg["row_bytes"])

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
    value = job_rate(world, B * K * depth, t_fwd)
    fused = B == 1 and launches_per_step == depth * (2 if chain else 1) - (1 if chain else 0)
    if fused:
        # one launch per layer: the fused kernel is the whole path, its bytes are the path's
        top_kernel = "fused_token_kernel"
        top_bytes = path_bytes / depth
        top_s = s_fwd / depth
        top_desc = ("fused_token_kernel (the whole single-token path in one launch: input "
                    "selection, Stage 1, top-k, Stage 2, the cross-block sum)")
    else:
        top_kernel = "stage2_kernel" if B == 1 else "stage2_tc_kernel"
        top_bytes = s2_bytes
        top_s = s_s2
        top_desc = (f"{top_kernel} (+ its fixed-order partial-sum reduce"
                    + (")" if B == 1 else
                       ", the batch's channel bitmap and the bf16 split of x)"))
    achieved = top_bytes / top_s / 1e9
    traffic, traffic_note = profiled_traffic(top_kernel, cfg["name"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, threads = cpu_oracle_rate(mats0, X_np, sp, s_in, args.cpu_seconds)
        rate1, n1, dt1, _ = cpu_oracle_rate(mats0, X_np, sp, s_in, args.cpu_seconds, threads=1)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "value_1core": rate1,
               "sample_1core": f"{n1} tokens in {dt1:.1f} s with the numerical libraries "
                               f"limited to one thread",
               "sample": f"{n} tokens (batch 1) of this workload, layer 0, through the fp64 "
                         f"numpy oracle in {dt:.1f} s (a token through one layer is the unit)"}

    if rank != 0:
        return
    us_layer = 1e6 * s_fwd / depth
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": warm, "ms_per_step": 1000.0 * s_fwd,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 Stage-2 weights" if cfg["fp8"] else "bf16", "data": "synthetic",
        "config": workload_config(cfg, world, T, k, k_in),
        "us_per_layer": us_layer,
        "us_per_step_chunks": fwd_stats,
        "spread_note": (f"20 chunks of {per_chunk} steps replayed after the {K} timed steps; "
                        "median/p10/p90 of the per-step time per chunk"),
        "hbm_gbs_path": path_bytes / s_fwd / 1e9,
        "path_frac": path_bytes / s_fwd / 1e9 / hbm_peak,
        "algorithmic_bytes_per_step": path_bytes,
        "dense_us_per_layer": 1e6 * s_dense / depth,
        "speedup_vs_dense": s_dense / s_fwd,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": top_desc,
                     "algorithmic_bytes_per_launch": top_bytes,
                     "us_per_launch": 1e6 * top_s,
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "traffic_note": traffic_note},
        "stage2_alone": {"us_per_layer": 1e6 * s_s2, "algorithmic_bytes": s2_bytes,
                         "achieved_gbs": s2_bytes / s_s2 / 1e9,
                         "frac": s2_bytes / s_s2 / 1e9 / hbm_peak,
                         "what": "prox_sparse_ffn over the masks the path builds (Stage 2 and "
                                 "the cross-block sum only)"},
        "e2e": {"value": job_rate(world, B * Ke * depth, t_e2e), "unit": UNIT,
                "h2d_bytes_per_step": B * d * 4, "d2h_bytes_per_step": B * d * 4,
                "api": ("prox_ffn_forward_host (pinned host x/y, synchronous per step)"
                        if not chain else
                        "pinned host x -> prox_ffn_forward + prox_rmsnorm through all layers "
                        "-> pinned host y, synchronous per step")},
        "gpu_launches": K * launches_per_step,
        "launches_per_step": launches_per_step,
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


def run_allocate(args):
    """Sparsity allocation with a measured cost model: the single-token path is timed at a few
    (k_in, k) points and the dense FFN once; prox_cost_model_fit turns those times into the
    cost model (microseconds), prox_choose_sparsity picks (input sparsity, sparsity) for each
    target effective sparsity, and the path is timed at that choice, so the achieved effective
    sparsity 1 - t / t_dense stands beside the predicted one. The byte cost model's choice is
    timed the same way. Rank 0 prints one JSON line."""
    import torch

    import free_sparse_swiglu_stage1_b300 as P
    import workloads as WL

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    cfg = resolve(args)
    if cfg["chain"] or cfg["batch"] != 1:
        raise SystemExit("--allocate times one layer at batch 1")
    d, F, L = cfg["d"], cfg["F"], cfg["layers"]
    layers = []
    for li in range(L):
        mats = WL.make_layer(cfg["key"], li)
        dev = {n: v.cuda() for n, v in mats.items() if n.startswith("w_")}
        layers.append(P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"]))
        del dev
    T = args.tokens
    X = torch.from_numpy(WL.make_tokens(cfg["key"], range(T))).cuda()
    Y = torch.empty((1, d), dtype=torch.float32, device="cuda")
    ws = P.prox_workspace(d, F, 1)
    stream = torch.cuda.Stream()
    K = args.steps

    def time_steps(fn):
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                fn(i)
        torch.cuda.synchronize()
        g = capture(torch, stream, fn, K)
        with torch.cuda.stream(stream):
            g.replay()
        return timed_graph_replays(torch, stream, [g], lambda: None, "allocate") / K * 1e6

    def path_us(s_in, s):
        return time_steps(lambda i: P.prox_ffn_forward(layers[i % L], X[(i // L) % T][None], s, s_in,
                                                       ws, y=Y, stream=stream))

    dense = time_steps(lambda i: P.prox_dense_ffn(layers[i % L], X[(i // L) % T][None], ws, y=Y,
                                                  stream=stream))
    pts = [(0.5, 0.7), (0.0, 0.7), (0.5, 0.4), (0.7, 0.9), (0.3, 0.55)]
    meas = []
    for s_in, s in pts:
        meas.append({"input_sparsity": s_in, "sparsity": s, "k_in": P.prox_k_for(s_in, d),
                     "k": P.prox_k_for(s, F), "us": path_us(s_in, s)})
    model = P.prox_cost_model_fit([m["k_in"] for m in meas], [m["k"] for m in meas],
                                  [m["us"] for m in meas], dense, 1e-6)
    byte_model = P.prox_cost_model_bytes(d, F)
    out = []
    for tgt in args.allocate:
        for name, cm in (("measured", model), ("bytes", byte_model)):
            try:
                s1, s2, pred = P.prox_choose_sparsity(cm, d, F, tgt)
            except P.ProxError as e:
                out.append({"target": tgt, "model": name, "error": str(e)})
                continue
            t = path_us(s1, s2)
            out.append({"target": tgt, "model": name, "input_sparsity": s1, "sparsity": s2,
                        "k_in": P.prox_k_for(s1, d), "k": P.prox_k_for(s2, F),
                        "predicted_effective": pred, "us": t, "achieved_effective": 1.0 - t / dense})
    if rank != 0:
        return
    print(json.dumps({"workload": cfg["name"], "d_model": d, "d_ff": F, "steps_per_point": K,
                      "dense_us": dense, "measurements": meas,
                      "fitted_model_us": {"in_cost": model.in_cost, "fixed_cost": model.fixed_cost,
                                          "ch_cost": model.ch_cost, "dense_cost": model.dense_cost},
                      "allocations": out}), flush=True)


def run_window(args):
    """The 32-layer stack with the proxy memory reduced to a sliding window of `args.window`
    device slots (split layers, proxies paged in from pinned host memory on the window's
    copy stream), against the same stack with resident layers. Steps are launched from the host
    (the window's slot state lives on the host), K steps timed with CUDA events on the compute
    stream. Rank 0 prints one JSON line."""
    import torch

    import free_sparse_swiglu_stage1_b300 as P
    import workloads as WL

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    cfg = resolve(args)
    if not cfg["chain"]:
        raise SystemExit("--window needs the 32-layer stack (--workload 4)")
    B, sp, s_in = cfg["batch"], cfg["sparsity"], cfg["input_sparsity"]
    d, F, depth = cfg["d"], cfg["F"], cfg["depth"]
    S = args.window
    full, split = [], []
    for li in range(depth):
        mats = WL.make_layer(cfg["key"], li)
        dev = {n: v.cuda() for n, v in mats.items() if n.startswith("w_")}
        lay = P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"])
        full.append(lay)
        split.append(P.prox_split_packed(lay, proxy_on_host=True))
        del dev
    win = P.ProxyWindow(split, S)
    T = max(B, args.tokens // B * B)
    X = torch.from_numpy(WL.make_tokens(cfg["key"], range(rank * T, (rank + 1) * T))).cuda()
    Xa = torch.empty((2, B, d), dtype=torch.float32, device="cuda")
    Ya = torch.empty((B, d), dtype=torch.float32, device="cuda")
    ws = P.prox_workspace(d, F, B)
    stream = torch.cuda.Stream()
    nb = T // B

    def step(i, windowed):
        t = i % nb
        xin = X[t * B:(t + 1) * B]
        for li in range(depth):
            desc = win.acquire(li, stream=stream) if windowed else full[li]
            P.prox_ffn_forward(desc, xin, sp, s_in, ws, y=Ya, stream=stream)
            if windowed:
                win.release(li, stream=stream)
            P.prox_rmsnorm(Ya, 1e-6, out=Xa[li % 2], stream=stream)
            xin = Xa[li % 2]

    def timed(windowed, K):
        for i in range(max(3, args.warmup)):
            step(i, windowed)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0 = win.stats()
        n0 = P.prox_launch_count()
        e0.record(stream)
        for i in range(K):
            step(i, windowed)
        e1.record(stream)
        torch.cuda.synchronize()
        c1 = win.stats()
        return (e0.elapsed_time(e1) / 1000.0, c1[0] - c0[0], c1[1] - c0[1],
                P.prox_launch_count() - n0)

    K = args.steps
    t_res, _, _, _ = timed(False, K)
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.3)
    t_win, copies, h2d, launches = timed(True, K)
    clocks = sampler.stop()
    st = P.prox_get_status(ws, stream=stream)
    if st != 0:
        raise RuntimeError(f"device status: {P.prox_error_string(st)}")
    pb = P.prox_proxy_bytes(d, F)
    units = K * B * depth
    if rank != 0:
        return
    line = {"metric": METRIC, "value": units / t_win, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": 1000.0 * t_win / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(workload_config(cfg, world, T, P.prox_k_for(sp, F), P.prox_k_for(s_in, d)),
                           proxy_window=S, launch="host-driven (no CUDA graph)"),
            "us_per_layer": 1e6 * t_win / (K * depth),
            "resident_us_per_layer": 1e6 * t_res / (K * depth),
            "window": {"slots": S, "proxy_bytes_per_layer": pb,
                       "proxy_device_bytes": S * pb, "proxy_device_bytes_resident": depth * pb,
                       "copies_per_step": copies / K, "h2d_bytes_per_step": h2d / K,
                       "h2d_gbs": h2d / t_win / 1e9},
            "gpu_launches": launches, "clocks": clocks, "e2e": None,
            "e2e_note": "the window's proxies come from host memory on every visit; the device "
                        "input and output stay resident"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.steps is None:
        args.steps = 400 if args.workload == CHAIN_WORKLOAD else 20000
    if args.impl == "reference":
        run_reference(args)
    elif args.window is not None:
        run_window(args)
    elif args.allocate is not None:
        run_allocate(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
