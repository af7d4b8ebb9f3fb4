#!/usr/bin/env python
"""Decode-step throughput of the packed two-D compressed KV cache on GB300.

One step = one decode step of the whole hot path over every layer: append and
compress one new token per sequence, score and select blocks, packed sparse
attention with un-rotation.  Inputs are synthetic (low rank plus outliers,
LLaMA-3.1-8B attention shapes) and resident in HBM; the step is captured once
in a CUDA graph and replayed.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3] [--impl reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the slow reference arm); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed decode-attn context tokens/s & HBM GB/s vs 8 TB/s roofline (1 GB300)"
UNIT = "context tokens/s"
D = 128


# Kernels each layer of a decode step launches: the fused path runs k_select
# (append + scoring), k_topk and k_attn; the separate path adds k_append_small
# in front of the same three.
LAUNCHES_PER_LAYER = {False: 3, True: 4}
# Untimed steps between the warm-up and the timed region while the clock
# sampler starts (each appends one token per layer, so capacity allows them).
CLOCK_SOAK_STEPS = 200


def max_over_ranks(x, dist, device):
    """The largest of the ranks' x (the job's time is its slowest rank's); x itself on one rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(units_per_rank, world, ms):
    """Whole-job throughput under weak scaling: every rank processes the same number of units (context
    tokens x layers) in one step, and the step takes ms on the slowest rank."""
    return units_per_rank * world / (ms * 1e-3)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c3")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dense-ref", action="store_true", help="also time the uncompressed reference kernel")
    ap.add_argument("--no-quest", action="store_true", help="skip the Quest comparator (uncompressed pages)")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling runs)")
    ap.add_argument("--bitmap", type=int, default=0, choices=[0, 1, 2, 4, 8],
                    help="bitmap pages with this element-group size instead of uint8 indices")
    ap.add_argument("--meta-channels", type=int, default=0,
                    help="variant: channel-compressed per-block keys keeping this many channels")
    ap.add_argument("--separate", action="store_true",
                    help="append and block selection as two launches (default: mk_append_select, one launch)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# algorithmic bytes (what the method must move per step)
# ----------------------------------------------------------------------------
def unit_bytes(wl, T, firsts):
    """Per (sequence, kv head) algorithmic bytes of one decode step at length T."""
    S, W, B, G = wl.n_sink, wl.window, wl.block, wl.group
    mid = max(0, T - S - W)
    nblk = (mid + B - 1) // B
    segs = wl.segments
    bounds = list(firsts) + [nblk]
    scored, always_bytes, r_scored = 0, 0, segs[0][1]
    for i, sg in enumerate(segs):
        r, always = sg[1], sg[2]
        lo, hi = min(bounds[i], nblk), min(bounds[i + 1] if i + 1 < len(segs) else nblk, nblk)
        n = max(0, hi - lo)
        if always:
            always_bytes += n * B * page_row(wl, r)
        else:
            scored += n
            r_scored = r
    if wl.topk_fixed:
        k = min(wl.topk_fixed, scored)
    else:
        k = min(max(1, (wl.retain_permille * scored + 999) // 1000), scored) if scored else 0
    dense = min(S, T) + (T - (S + mid))
    mc = getattr(wl, "meta_channels", 0)
    key_row = (5 * mc + 15) // 16 * 16 if mc else 2 * D * 2   # a block's key as the scoring reads it
    sel = nblk * key_row + G * D * 2 + D * D * 4
    attn = k * B * page_row(wl, r_scored) + always_bytes + dense * 2 * D * 2 + D * D * 4 + G * D * (4 + 2)
    r_new = segs[-1][1]
    app = (2 * D * 2 + 2 * D * D * 4 + 2 * D * 2 + 2 * D * 2 + page_row(wl, r_new) + 2 * 2 * D * 2 +
           (key_row if mc else 0))
    return {"append": app, "select": sel, "attn": attn}


def page_row(wl, r):
    """Packed bytes of one token (K and V): r bf16 values each plus r uint8
    indices each, or a bitmap of 128 / g bits each in the bitmap format."""
    g = getattr(wl, "elem_group", 0)
    return 2 * (2 * r + (D // g // 8 if g else r))


def segment_firsts(wl, T0):
    S, W, B = wl.n_sink, wl.window, wl.block
    nb0 = (max(0, T0 - S - W) + B - 1) // B
    out, prev = [], 0
    for i, sg in enumerate(wl.segments):
        beg = sg[0]
        b = 0 if i == 0 else min(max((max(0, beg * T0 // 1000 - S) + B - 1) // B, prev), nb0)
        out.append(b)
        prev = b
    return out


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def _host_ram_bytes():
    try:
        return os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 64 << 30


def _oracle_unit(job):
    """One worker process: builds one (layer, sequence, kv head) unit of the
    workload in the fp64 oracle (prefill), then times its decode steps (append
    one token, select, attend) for `seconds`, or exactly `steps` of them.
    Returns (seconds per decode step, steps timed)."""
    wl, (layer, seq, kvh), steps, seconds = job
    from compressed_kv_cache_vector_gb300 import synth
    from oracle import mosaickv_oracle as O
    T0 = wl.seq_lens[seq]
    n_extra = (steps if steps is not None else 4096) + 1
    sd = synth.seed_for(wl.name, 0, layer, seq, kvh)
    K = synth.bf16_values(synth.lowrank_outlier(T0 + n_extra, D, wl.decay, sd))
    V = synth.bf16_values(synth.lowrank_outlier(T0 + n_extra, D, wl.decay, sd + 1))
    Rk, _ = O.rotation_from_keys(K[:T0])
    Rv, _ = O.rotation_from_keys(V[:T0])
    st = O.Strategy(wl.n_sink, wl.window, wl.block, list(wl.segments), wl.topk_fixed, wl.retain_permille,
                    wl.meta_channels, wl.elem_group)
    oc = O.OracleCache(st, T0 + n_extra)
    oc.set_rotation(Rk, Rv)
    oc.append(K[:T0], V[:T0])
    q = synth.bf16_values(synth.query(1, wl.group, D, sd + 2)[0])
    t_total, n = 0.0, 0
    while True:
        t = oc.T
        t0 = time.perf_counter()
        oc.append(K[t:t + 1], V[t:t + 1])
        ids, _ = oc.select(q)
        oc.attention(q, ids)
        t_total += time.perf_counter() - t0
        n += 1
        if steps is not None and n >= steps:
            break
        if steps is None and (t_total >= seconds or n >= n_extra - 1):
            break
    return t_total / n, n


def oracle_sample(wl, steps=None, seconds=15.0):
    """Times the oracle's decode step on a sample of the workload's units, one
    single-threaded process per host core (spawned, never forked), each on its
    own (layer, sequence, kv head) unit, all at once.  The full step's time is
    extrapolated: every unit's mean step time, over the units the cores share.
    Returns (context tokens/s, description, seconds of the longest worker,
    processes used)."""
    import multiprocessing as mpr
    units = [(l, s, h) for l in range(wl.n_layers) for s in range(wl.n_seqs) for h in range(wl.n_kv_heads)]
    cores = os.cpu_count() or 1
    per_worker = 3600 * (max(wl.seq_lens) + 4096)         # oracle arrays of one unit, bytes
    n_proc = max(1, min(cores, len(units), int(0.5 * _host_ram_bytes() // per_worker)))
    pick = [units[(i * len(units)) // n_proc] for i in range(n_proc)]
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"                              # one thread per worker process
    try:
        with mpr.get_context("spawn").Pool(n_proc) as pool:
            res = pool.map(_oracle_unit, [(wl, u, steps, seconds) for u in pick])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    mean_step = sum(r[0] for r in res) / len(res)
    full_step = mean_step * len(units) / n_proc         # the cores share the units
    ctx = sum(wl.seq_lens) * wl.n_layers
    n_steps = sum(r[1] for r in res)
    desc = (f"{n_proc} single-threaded processes in parallel, each timing decode steps of its own "
            f"(layer, sequence, kv head) unit (fp64 numpy oracle; {n_steps} steps in all); the full step "
            f"of {len(units)} units extrapolated as mean step time x {len(units)} / {n_proc}")
    return ctx / full_step, desc, max(r[0] * r[1] for r in res), n_proc


# ----------------------------------------------------------------------------
# GPU workload
# ----------------------------------------------------------------------------
def build_gpu(wl, dev, rank, capacity_extra, quest=False):
    """The workload's cache on the GPU, built by bulk prefill of every layer.
    quest=True builds the Quest comparator instead: uncompressed pages
    (every channel kept), identity rotations, the same segments and blocks."""
    import torch
    from compressed_kv_cache_vector_gb300 import binding, synth
    from compressed_kv_cache_vector_gb300.build import build
    build()
    segments = [(sg[0], D, sg[2]) for sg in wl.segments] if quest else wl.segments
    cfg = binding.make_config(wl.n_q_heads, wl.n_kv_heads, wl.n_layers, wl.n_seqs,
                              max(wl.seq_lens) + capacity_extra, wl.n_sink, wl.window, wl.block,
                              segments, wl.topk_fixed, wl.retain_permille, 0 if quest else wl.meta_channels,
                              1 if quest else (2 if wl.elem_group else 0), 0 if quest else wl.elem_group)
    mk = binding.MosaicKV(cfg, dev)
    eye = np.eye(D, dtype=np.float32)
    seqs = list(range(wl.n_seqs))
    prefill_ms = mk.prefill_ms = []
    gram = torch.empty(D, D, dtype=torch.float32, device=dev)
    for l in range(wl.n_layers):
        ks, vs = [], []
        for s, T in enumerate(wl.seq_lens):
            kh, vh = [], []
            for h in range(wl.n_kv_heads):
                sd = synth.seed_for(wl.name, rank, l, s, h)
                k = synth.lowrank_outlier(T, D, wl.decay, sd, device=dev)
                v = synth.lowrank_outlier(T, D, wl.decay, sd + 1, device=dev)
                if quest:
                    mk.set_rotation(l, s, h, eye, eye)
                else:
                    Rk = binding.rotation_from_gram(binding.gram(k, T, D, gram).cpu().numpy())
                    Rv = binding.rotation_from_gram(binding.gram(v, T, D, gram).cpu().numpy())
                    mk.set_rotation(l, s, h, Rk, Rv)
                kh.append(k)
                vh.append(v)
            ks.append(torch.stack(kh, 1))
            vs.append(torch.stack(vh, 1))
            del kh, vh
        kcat, vcat = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
        del ks, vs
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        binding.record_event(e0)
        mk.append(l, seqs, list(wl.seq_lens), kcat, vcat)   # bulk prefill of the layer
        binding.record_event(e1)
        torch.cuda.synchronize()
        prefill_ms.append(e0.elapsed_time(e1))
        del kcat, vcat
    st, detail = mk.poll_error()
    if st != 0:
        raise RuntimeError(f"device error during cache build: {st}/{detail}")
    return mk


def _free_port():
    import socket
    so = socket.socket()
    so.bind(("127.0.0.1", 0))
    port = so.getsockname()[1]
    so.close()
    return port


def launch_ranks(a):
    """--gpus N outside a launcher: run this script as N ranks under
    torch.distributed.run (one process per GPU, rendezvous on 127.0.0.1) and
    return its exit code.  Our arm needs N visible GPUs; it exits with an error
    instead of running fewer ranks than asked."""
    if a.impl == "ours":
        import torch
        have = torch.cuda.device_count()
        if have < a.gpus:
            print(f"bench.py: --gpus {a.gpus} asked, {have} GPU(s) visible", file=sys.stderr)
            return 2
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={a.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    a = parse()
    if a.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(a))
    import torch
    from compressed_kv_cache_vector_gb300 import configs
    wl = configs.get(a.config)
    if a.layers:
        wl.n_layers = a.layers
        wl.name += f"-{a.layers}layer"
    if a.meta_channels:
        wl.meta_channels = a.meta_channels
        wl.name += f"-keys{a.meta_channels}ch"
    if a.bitmap:
        # Bitmap pages with element group g: each r rounded up to a multiple of g.
        g = a.bitmap
        wl.elem_group = g
        wl.segments = [(sg[0], (sg[1] + g - 1) // g * g) + tuple(sg[2:]) for sg in wl.segments]
        wl.name += f"-bitmap-g{g}-r{'-'.join(str(sg[1]) for sg in wl.segments)}"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if a.impl == "ours" else "gloo")

    base = {"metric": METRIC, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded low-rank-plus-outlier K/V, LLaMA-3.1-8B attention shapes)"}
    wcfg = {"workload": wl.name, "description": wl.description, "q_heads": wl.n_q_heads,
            "kv_heads": wl.n_kv_heads, "head_dim": D, "layers": wl.n_layers, "seqs_per_gpu": wl.n_seqs,
            "context_per_seq": wl.seq_lens[0] if len(set(wl.seq_lens)) == 1 else "mixed",
            "block": wl.block, "segments": wl.segments, "n_sink": wl.n_sink, "window": wl.window}

    if a.impl == "reference":
        if rank != 0:
            return
        cpu_v, desc, secs, n_proc = oracle_sample(wl, steps=a.warmup + a.steps)
        line = dict(base, impl="reference", value=cpu_v, n_gpus=world,
                    ms_per_step=1e3 * sum(wl.seq_lens) * wl.n_layers / cpu_v,
                    ms_per_step_kind=f"extrapolated: sampled units' mean step time x units / {n_proc} processes",
                    config=wcfg,
                    cpu_baseline={"value": cpu_v, "unit": UNIT, "cores": n_proc, "kind": "oracle",
                                  "sample": desc},
                    e2e={"value": cpu_v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                    dtype="f64")
        print(json.dumps(line), flush=True)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from compressed_kv_cache_vector_gb300 import binding, synth
    extra = 4 * (a.warmup + a.steps) + 32 + CLOCK_SOAK_STEPS
    mk = build_gpu(wl, dev, rank, extra)
    L, n_seq, Hq, Hkv = wl.n_layers, wl.n_seqs, wl.n_q_heads, wl.n_kv_heads
    seqs = list(range(n_seq))
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    k_in = [torch.randn(n_seq, Hkv, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    v_in = [torch.randn(n_seq, Hkv, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    q_in = [synth.query(n_seq, Hq, D, synth.seed_for(wl.name, "q", rank, l), device=dev) for l in range(L)]
    sel = [mk.alloc_select(n_seq) for _ in range(L)]
    outs = [torch.empty(n_seq, Hq, D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(L)]

    def step(instrument):
        for l in range(L):
            if instrument:
                binding.record_event(ev[l][0])
            if a.separate:
                mk.append(l, seqs, [1] * n_seq, k_in[l], v_in[l])
                if instrument:
                    binding.record_event(ev[l][1])
                mk.block_select(l, seqs, q_in[l], *sel[l])
            else:
                mk.append_select(l, seqs, k_in[l], v_in[l], q_in[l], *sel[l])
                if instrument:
                    binding.record_event(ev[l][1])
            if instrument:
                binding.record_event(ev[l][2])
            mk.decode_attn(l, seqs, *sel[l], out=outs[l])
            if instrument:
                binding.record_event(ev[l][3])

    # eager warm-up (also sets kernel attributes), then capture one step
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(True)
    torch.cuda.synchronize()
    # Two captures of the same step: `graph` (kernels back to back, so the
    # programmatic dependent launches overlap) for the timed value, and
    # `graph_ev` with event-record nodes between kernels for per-kernel times.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(False)
    torch.cuda.synchronize()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=s):
        step(True)
    torch.cuda.synchronize()
    # A third capture: only the layers' attention launches, back to back (each
    # over its layer's cache and selection, as left by the step), for the
    # dominant kernel's average launch duration without event nodes between
    # kernels.
    graph_attn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_attn, stream=s):
        for l in range(L):
            mk.decode_attn(l, seqs, *sel[l], out=outs[l])
    torch.cuda.synchronize()
    graph_sel = None
    if not a.separate:   # and only the selection calls (append + block selection), back to back
        graph_sel = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_sel, stream=s):
            for l in range(L):
                mk.append_select(l, seqs, k_in[l], v_in[l], q_in[l], *sel[l])
        torch.cuda.synchronize()
    mk.sync_state()
    T_start = [mk.seq_length(0, si) for si in seqs]

    # Clocks: nvidia-smi every 20 ms from the start of the warm-up (its own
    # start-up takes longer than the short timed region) to the end of the
    # timed regions; every sample is taken under the same load.
    clocks = Clocks(local)
    clocks.start()
    for _ in range(a.warmup):
        graph.replay()
    # A few more untimed steps (at most CLOCK_SOAK_STEPS, about 0.2 s) so that
    # the sampler's first readings fall under this load, not before it.
    t_soak = time.perf_counter() + 0.2
    n_soak = 0
    while n_soak < CLOCK_SOAK_STEPS and time.perf_counter() < t_soak:
        graph.replay()
        torch.cuda.synchronize()
        n_soak += 1
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    # Timed region A: K steps back to back (the reported value).
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(a.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    # Timed region B: the instrumented step, K more times, reading its event
    # nodes after each replay (per-kernel durations for the roofline).
    attn_ms, sel_ms, app_ms, span_ms = [], [], [], []
    for _ in range(a.steps):
        graph_ev.replay()
        torch.cuda.synchronize()
        span_ms.append(ev[0][0].elapsed_time(ev[L - 1][3]))
        for l in range(L):
            app_ms.append(ev[l][0].elapsed_time(ev[l][1]))
            sel_ms.append(ev[l][1].elapsed_time(ev[l][2]))
            attn_ms.append(ev[l][2].elapsed_time(ev[l][3]))
    # Timed region C: the attention-only graph, K times.
    torch.cuda.synchronize()
    e0.record()
    for _ in range(a.steps):
        graph_attn.replay()
    e1.record()
    torch.cuda.synchronize()
    attn_only_ms = e0.elapsed_time(e1) / (a.steps * L)
    # Timed region D: the selection-only graph, K times.
    sel_only_ms = time_graph(graph_sel, a.steps) / L if graph_sel is not None else None
    clk = clocks.stop()
    mk.sync_state()
    st, detail = mk.poll_error()
    if st != 0:
        raise RuntimeError(f"device error word set during the run: {st}/{detail}")
    ms = total_ms / a.steps
    ms = max_over_ranks(ms, dist, dev)

    # algorithmic bytes at the mean length of the timed steps
    T_mid = [t + a.warmup + n_soak + a.steps / 2 for t in T_start]
    firsts = [segment_firsts(wl, T0) for T0 in wl.seq_lens]
    per = {"append": 0, "select": 0, "attn": 0}
    for si, T in enumerate(T_mid):
        b = unit_bytes(wl, int(T), firsts[si])
        for k_ in per:
            per[k_] += b[k_] * Hkv
    step_bytes = sum(per.values()) * L
    ctx_tokens = sum(T_mid) * L * world
    value = weak_value(sum(T_mid) * L, world, ms)
    gbs = step_bytes * world / (ms * 1e-3) / 1e9

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except Exception:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    attn_avg = statistics.mean(attn_ms)
    sel_avg = statistics.mean(sel_ms)
    app_avg = statistics.mean(app_ms)
    achieved = per["attn"] / (attn_only_ms * 1e-3) / 1e9
    roofline = {"kernel": "k_attn (packed sparse attention + split-T combine + un-rotation)",
                "bound": "hbm", "achieved": achieved, "peak": peak, "peak_source": peak_src,
                "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                "alg_bytes_per_launch": per["attn"], "avg_launch_ms": attn_only_ms,
                "avg_launch_ms_how": f"CUDA events around {a.steps} replays of a graph of the {L} layers' "
                                     "attention launches back to back, divided by the launches"}
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            tr = json.load(f).get(wl.name, {}).get("k_attn")
        import hashlib
        src = open(os.path.join(ROOT, "compressed_kv_cache_vector_gb300", "csrc", "mk_attn.cu"), "rb").read()
        if tr and tr.get("src_sha256") == hashlib.sha256(src).hexdigest():
            roofline["traffic"] = tr["bytes_per_launch"]
    except Exception:
        pass
    if a.separate:
        phases = {
            "append_ms": app_avg, "select_ms": sel_avg, "attn_ms": attn_avg,
            "append_gbs": per["append"] / (app_avg * 1e-3) / 1e9,
            "select_gbs": per["select"] / (sel_avg * 1e-3) / 1e9,
        }
    else:
        phases = {
            "append_select_ms": app_avg + sel_avg, "attn_ms": attn_avg,
            "append_select_gbs": (per["append"] + per["select"]) / ((app_avg + sel_avg) * 1e-3) / 1e9,
        }
    phases.update({"graphs_ms_per_layer": {"step": ms / L, "append_select_only": sel_only_ms,
                                           "attn_only": attn_only_ms},
                   "attn_gbs_instrumented": per["attn"] / (attn_avg * 1e-3) / 1e9,
                   "step_span_ms": statistics.mean(span_ms), "alg_bytes_per_layer": per,
                   "launches_per_layer": LAUNCHES_PER_LAYER[a.separate],
                   "how": "instrumented graph: event-record nodes between the kernels, so a kernel cannot start "
                          "its prologue under the previous one (programmatic dependent launch overlap is lost); "
                          "each phase is timed alone and the phases add up to more than the step"})

    # end to end through the public API with host buffers (eager calls): each
    # step copies all layers' new k, v and q from one pinned host buffer in
    # one transfer, makes the per-layer calls, and reads all layers' outputs
    # back in one transfer.
    e2e = None
    if not a.no_e2e:
        per_layer = [k_in[0].numel(), v_in[0].numel(), q_in[0].numel()]
        n_in = sum(per_layer) * L
        hin = torch.empty(n_in, dtype=torch.bfloat16).pin_memory()
        din = torch.empty(n_in, dtype=torch.bfloat16, device=dev)
        dk, dv, dq = [], [], []
        off = 0
        for l in range(L):
            for src, dev_list in ((k_in[l], dk), (v_in[l], dv), (q_in[l], dq)):
                n = src.numel()
                hin[off:off + n].copy_(src.reshape(-1).cpu())
                dev_list.append(din[off:off + n].view(src.shape))
                off += n
        dout = torch.empty(L, n_seq, Hq, D, dtype=torch.bfloat16, device=dev)
        hout = torch.empty(L, n_seq, Hq, D, dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            din.copy_(hin, non_blocking=True)
            for l in range(L):
                if a.separate:
                    mk.append(l, seqs, [1] * n_seq, dk[l], dv[l])
                    mk.block_select(l, seqs, dq[l], *sel[l])
                else:
                    mk.append_select(l, seqs, dk[l], dv[l], dq[l], *sel[l])
                mk.decode_attn(l, seqs, *sel[l], out=dout[l])
            hout.copy_(dout, non_blocking=True)

        for _ in range(a.warmup):
            e2e_step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(a.steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / a.steps
        e2e_ms = max_over_ranks(e2e_ms, dist, dev)
        e2e = {"value": ctx_tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": hin.numel() * 2,
               "d2h_bytes_per_step": hout.numel() * 2, "ms_per_step": e2e_ms,
               "how": "eager C-ABI calls per layer (no graph); each step copies all layers' new k, v, q in from "
                      "pinned host memory and all outputs back, one transfer each way"}
        mk.sync_state()

    dense = None
    if a.dense_ref and rank == 0:
        dense = dense_reference(mk, wl, dev)
    quest = None
    if not a.no_quest and rank == 0 and not a.separate:
        del graph, graph_ev, graph_attn, graph_sel
        quest = quest_reference(wl, dev, rank, a.steps)
        quest["attn_ratio_quest_over_ours"] = quest["attn_ms_per_layer"] / attn_only_ms
        if sel_only_ms:
            quest["select_ratio_quest_over_ours"] = quest["select_ms_per_layer"] / sel_only_ms
        quest["step_ratio_quest_over_ours"] = quest["step_ms_per_layer"] / (ms / L)

    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cpu_v, desc, secs, n_proc = oracle_sample(wl, seconds=a.cpu_seconds)
        cpu = {"value": cpu_v, "unit": UNIT, "cores": n_proc, "kind": "oracle", "sample": desc,
               "seconds": secs}

    if rank != 0:
        return
    wcfg["l2"] = "inputs larger than L2: a step reads ~%.2f GB, the L2 holds 129 MB; no flush" % (step_bytes / 1e9)
    line = dict(base, value=value, ms_per_step=ms,
                config=wcfg,
                timing={"l2": "step reads ~%.2f GB across layers, far above the 129 MB L2, so no flush" %
                              (step_bytes / 1e9),
                        "how": "CUDA graph of one full step, replayed; CUDA events on the stream",
                        "untimed_soak_steps": n_soak,
                        "calls": ("mk_append_compress + mk_block_select + mk_decode_attn" if a.separate else
                                  "mk_append_select + mk_decode_attn") + " per layer"},
                hbm_gbs=gbs, alg_bytes_per_step=step_bytes, roofline=roofline, phases=phases,
                cpu_baseline=cpu, e2e=e2e, gpu_launches=LAUNCHES_PER_LAYER[a.separate] * L * a.steps, clocks=clk)
    if mk.prefill_ms:
        pm = sorted(mk.prefill_ms)[len(mk.prefill_ms) // 2]
        ntok = sum(wl.seq_lens) * wl.n_kv_heads
        line["prefill"] = {
            "kernel": "k_append_bulk (128-token tiles: tcgen05 rotation GEMM, top-r, pack, block min/max)",
            "ms_per_layer_median": pm, "vectors_per_s": 2 * ntok / (pm * 1e-3),
            "tensor_tflops": 2 * ntok * 3 * 2 * D * D / (pm * 1e-3) / 1e12,
            "hbm_read_gbs": 2 * ntok * D * 2 / (pm * 1e-3) / 1e9,
            "how": "CUDA events around the bulk mk_append_compress of each layer while building the cache"}
    if dense:
        line["dense_reference"] = dense
    if quest:
        line["quest_reference"] = quest
    print(json.dumps(line), flush=True)


def time_graph(graph, reps):
    """ms per replay of a captured graph: CUDA events around `reps` replays on
    the current stream, after one untimed replay."""
    import torch
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def capture_layer_graphs(mk, L, seqs, k_in, v_in, q_in, sel, outs, stream):
    """Three graphs over L layers: the whole decode step (append + selection,
    attention), the selection calls alone, the attention calls alone."""
    import torch
    graphs = {}
    for name in ("step", "select", "attn"):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                if name != "attn":
                    mk.append_select(l, seqs, k_in[l], v_in[l], q_in[l], *sel[l])
                if name != "select":
                    mk.decode_attn(l, seqs, *sel[l], out=outs[l])
        torch.cuda.synchronize()
        graphs[name] = g
    return graphs


def quest_reference(wl, dev, rank, steps):
    """The Quest comparator ([S] sec. 6.1, 6.3) on the same workload shape:
    uncompressed pages, identity rotations, the same block selection kernels
    and the same attention kernel reading whole rows.  Built for as few
    layers as make one pass over their selected pages larger than the L2
    (so no layer is read from L2 on its next turn)."""
    import copy
    import torch
    from compressed_kv_cache_vector_gb300 import synth
    qw = copy.deepcopy(wl)
    B = wl.block
    nblk = max(1, (max(wl.seq_lens) - wl.n_sink - wl.window) // B)
    k = max(1, (wl.retain_permille * nblk + 999) // 1000) if not wl.topk_fixed else wl.topk_fixed
    sel_bytes = k * B * 4 * D * wl.n_kv_heads * wl.n_seqs
    qw.n_layers = int(min(wl.n_layers, max(1, math.ceil(3 * 129e6 / sel_bytes))))
    qw.meta_channels = 0
    reps = max(4, steps)
    mk = build_gpu(qw, dev, rank, 4 * reps + 16, quest=True)
    L, n_seq = qw.n_layers, qw.n_seqs
    seqs = list(range(n_seq))
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + rank)
    k_in = [torch.randn(n_seq, qw.n_kv_heads, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    v_in = [torch.randn(n_seq, qw.n_kv_heads, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    q_in = [synth.query(n_seq, qw.n_q_heads, D, synth.seed_for(wl.name, "q", rank, l), device=dev) for l in range(L)]
    sel = [mk.alloc_select(n_seq) for _ in range(L)]
    outs = [torch.empty(n_seq, qw.n_q_heads, D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l in range(L):
            mk.append_select(l, seqs, k_in[l], v_in[l], q_in[l], *sel[l])
            mk.decode_attn(l, seqs, *sel[l], out=outs[l])
    torch.cuda.synchronize()
    graphs = capture_layer_graphs(mk, L, seqs, k_in, v_in, q_in, sel, outs, s)
    res = {name: time_graph(gr, reps) / L for name, gr in graphs.items()}
    st, detail = mk.poll_error()
    if st != 0:
        raise RuntimeError(f"device error in the Quest comparator: {st}/{detail}")
    out = {"layers": L, "step_ms_per_layer": res["step"], "select_ms_per_layer": res["select"],
           "attn_ms_per_layer": res["attn"], "selected_page_bytes_per_layer": sel_bytes,
           "how": "uncompressed pages (every channel, no rotation), same selection and attention kernels; "
                  "graphs of the layers' calls, CUDA events around replays"}
    mk.close()
    del mk
    torch.cuda.empty_cache()
    return out


def dense_reference(mk, wl, dev, reps=10):
    """Our own uncompressed decode attention on one layer's dense bf16 K/V."""
    import torch
    from compressed_kv_cache_vector_gb300 import synth
    n_seq, Hq, Hkv = wl.n_seqs, wl.n_q_heads, wl.n_kv_heads
    T = max(wl.seq_lens)
    K = torch.empty(n_seq, Hkv, T, D, dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    for s in range(n_seq):
        for h in range(Hkv):
            K[s, h] = synth.lowrank_outlier(T, D, wl.decay, synth.seed_for("dense", s, h), device=dev)
            V[s, h] = synth.lowrank_outlier(T, D, wl.decay, synth.seed_for("dense", s, h, 1), device=dev)
    q = synth.query(n_seq, Hq, D, 77, device=dev)
    out = torch.empty(n_seq, Hq, D, dtype=torch.bfloat16, device=dev)
    lens = list(wl.seq_lens)
    for _ in range(3):
        mk.dense_attn(lens, q, K, V, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        mk.dense_attn(lens, q, K, V, out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    byts = sum(lens) * Hkv * 2 * D * 2
    return {"ms_per_layer": ms, "gbs": byts / (ms * 1e-3) / 1e9, "bytes_per_layer": byts,
            "note": "K/V of one layer fit in L2 only when below 129 MB"}


if __name__ == "__main__":
    main()
