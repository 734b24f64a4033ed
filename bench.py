"""Decode-attention benchmark: one step = kv_append + gqa_decode_attn (fused:
gqa_decode_step) over a
seeded synthetic batch shaped like the PaLM-8B multi-query decode
(B=64, Hq=16, Hkv=1, D=256, 2048 cached positions) unless --workload says
otherwise.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-cpu-baseline]

Metric: KV-cache bytes the attention reads per second (only positions below
each sequence's length count), with decode sequence-steps per second beside
it.  Timing: W untimed steps, then exactly K steps between CUDA events on the
launching stream, each step reading a different copy of the cache (copies
together >= 4x L2) so reads come from HBM.  A step is one gqa_decode_step call
(the append fused into the attention kernel, plus the combine kernel); steps
are chained in CUDA graphs (one per rotation through the cache copies) and
the roofline uses the average step duration over the timed region.
Under torchrun every rank runs its own batch (weak scaling, no collective in
the data path); the barrier and the max over ranks stay.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV-cache read GB/s (fraction of GB300 HBM peak); decode-attn seq-steps/s"
DEFAULT_WORKLOAD = "palm8b_mqa"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(seed, rank):
    """Each rank draws its own batch: the ranks run independent problems
    (weak scaling, no data-path exchange)."""
    return seed + 1000 * rank


def over_ranks(ms_total, units, world, device):
    """Whole-job timing over the ranks: the slowest rank's elapsed time and
    the units (KV bytes of the timed steps) that all ranks processed.  With
    one rank, the inputs unchanged."""
    if world <= 1:
        return float(ms_total), float(units)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(ms_total)], dtype=torch.float64, device=device)
    uu = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    dist.all_reduce(uu, op=dist.ReduceOp.SUM)
    return float(tt.item()), float(uu.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ------------------------------------------------- DRAM traffic (from ncu)

def sources_digest():
    """sha256 over the CUDA sources and the C header (sorted by name): ties a
    stored ncu traffic figure to the exact kernels it was measured on."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(root, "grouped_query_kv_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join(root, "include", "kvattn.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(workload):
    """DRAM bytes (read + write) per launch of each kernel of one step, from
    the table in profiles/dram_traffic.md, when it was taken on the current
    sources; None otherwise."""
    root = os.path.dirname(os.path.abspath(__file__))
    path = os.path.join(root, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    digest = sources_digest()
    kernels = {}
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) != 5 or cells[0] != workload or cells[4] != digest:
            continue
        try:
            kernels[cells[1]] = int(cells[2]) + int(cells[3])
        except ValueError:
            continue
    return kernels or None


# ------------------------------------------------------------ clocks sampler

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
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
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle

def oracle_sample(w, seed, target_s, max_seqs=None, threads=None):
    """Time the oracle (all host cores, or `threads` of them) on whole
    sequences of the workload: as many sequences as fit in target_s (at most
    the whole batch), repeated until target_s of CPU work has run.  Returns
    (seconds, sequences, kv_bytes, threads, repetitions)."""
    import dataclasses

    import oracle
    from grouped_query_kv_gb300 import accounting
    from grouped_query_kv_gb300 import workloads as wl

    threads = threads or os.cpu_count() or 1
    lens_all = wl.attn_lens(w, seed)

    def inputs(nb):
        return _oracle_inputs(w, seed, nb, lens_all)

    def once(x):
        t = time.perf_counter()
        _oracle_call(w, x, threads)
        return time.perf_counter() - t

    x1 = inputs(1)
    dt1 = once(x1)
    nb = max(1, min(w.B if max_seqs is None else max_seqs,
                    int(math.ceil(target_s / max(dt1, 1e-6)))))
    x = inputs(nb) if nb > 1 else x1
    total, reps = 0.0, 0
    while total < target_s or reps == 0:
        total += once(x)
        reps += 1
    return total, nb, x[4] * reps, threads, reps


def reference_arm(a, w):
    """The reference arm is the CPU oracle as it stands, timed on this machine's
    host cores over a bounded sample of the workload each step (whole
    sequences, all heads), sized so that W + K steps take about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    per_step = min(3.0, 120.0 / max(1, a.steps + a.warmup))
    _, nb, _, threads, _ = oracle_sample(w, a.seed, per_step)
    times, by = [], 0
    for i in range(a.warmup + a.steps):
        dt, _, by, _ = _oracle_fixed(w, a.seed, nb, threads)
        if i >= a.warmup:
            times.append(dt)
    tot = sum(times)
    gbs = by * len(times) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B_sampled": nb, "B": w.B, "Hq": w.Hq,
                   "Hkv": w.Hkv, "D": w.D, "Lmax": w.Lmax, "window": w.window,
                   "T": w.T, "block_size": w.block_size},
        "seq_steps_per_s": nb * len(times) / tot,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "%d of %d sequences (all heads) per step; %s" %
                                   (nb, w.B, cpu_model())},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _oracle_inputs(w, seed, nb, lens_all):
    """The first nb sequences of the workload as the oracle takes them
    (bf16 bits; pools and a block table for a paged workload), with their
    algorithmic bytes."""
    import dataclasses

    from grouped_query_kv_gb300 import accounting
    from grouped_query_kv_gb300 import workloads as wl
    sub = dataclasses.replace(w, B=nb, lens=None, ragged=False)
    x = wl.make_inputs(sub, seed=seed, device="cpu", lens=lens_all[:nb])
    lens = x["attn_lens"].numpy()
    by = accounting.kv_bytes_read(lens, w.Hkv, w.D, window=w.window)
    if w.kv_dtype == "fp8":
        import oracle
        kc, ks = oracle.quantize_fp8(wl.bf16_bits(x["k_cache"]))
        vc, vs = oracle.quantize_fp8(wl.bf16_bits(x["v_cache"]))
        by = accounting.kv_bytes_read_fp8(lens, w.Hkv, w.D)
        return (wl.bf16_bits(x["q"]), kc, vc, lens, by, ("fp8", ks, vs))
    if w.block_size:
        pg = wl.make_paged(sub, x, seed=seed)
        return (wl.bf16_bits(x["q"]), wl.bf16_bits(pg["k_pool"]), wl.bf16_bits(pg["v_pool"]),
                lens, by, pg["block_table"].numpy())
    return tuple(wl.bf16_bits(x[n]) for n in ("q", "k_cache", "v_cache")) + (lens, by, None)


def _oracle_call(w, x, threads):
    import oracle
    q, k, v, lens, _, table = x
    if isinstance(table, tuple):
        oracle.gqa_decode_fp8(q, k, v, table[1], table[2], lens, w.scale, nthreads=threads)
    elif table is not None:
        oracle.gqa_decode_paged(q, k, v, table, lens, w.block_size, w.scale, nthreads=threads)
    elif w.T > 1:
        oracle.gqa_decode_multi(q, k, v, lens, w.scale, nthreads=threads)
    else:
        oracle.gqa_decode(q, k, v, lens, w.scale, nthreads=threads, window=w.window)


_FIXED_CACHE = {}


def _oracle_fixed(w, seed, nb, threads):
    from grouped_query_kv_gb300 import workloads as wl
    key = (w.name, seed, nb)
    if key not in _FIXED_CACHE:
        _FIXED_CACHE[key] = _oracle_inputs(w, seed, nb, wl.attn_lens(w, seed))
    x = _FIXED_CACHE[key]
    t = time.perf_counter()
    _oracle_call(w, x, threads)
    return time.perf_counter() - t, nb, x[4], threads


# ------------------------------------------------------------------ GPU arm

CHAIN_MAX = 1000          # steps per captured CUDA graph
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
# the other target shapes (and the built extensions), timed in the same run
PER_CONFIG = ["palm8b_mqa", "llama70b_gqa_ragged", "palm540b_long_mqa", "sweep_hkv32_b256",
              "sweep_hkv8_b256", "sweep_hkv1_b256", "local_gqa_w4096", "llama70b_spec4",
              "palm540b_spec4", "palm8b_spec4", "llama70b_paged64", "llama70b_paged16", "llama70b_fp8",
              "palm8b_fp8", "palm540b_fp8"]


class Setup:
    """One workload's device inputs, its rotation of cache copies (so that
    consecutive steps never hit in L2) and the step call."""

    def __init__(self, w, seed, dev, lib, stream):
        import torch

        import grouped_query_kv_gb300 as g
        from grouped_query_kv_gb300 import accounting
        from grouped_query_kv_gb300 import workloads as wl

        self.w, self.dev, self.lib, self.stream = w, dev, lib, stream
        props = torch.cuda.get_device_properties(dev)
        self.l2 = l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
        lens_host = wl.attn_lens(w, seed).tolist()
        read_bytes = accounting.kv_bytes_read(lens_host, w.Hkv, w.D, window=w.window)
        x = wl.make_inputs(w, seed=seed, device=dev)
        self.table = None
        self.fp8 = w.kv_dtype == "fp8"
        if w.block_size:
            # paged: the pools hold only the blocks the sequences use, scattered
            pg = wl.make_paged(w, x, seed=seed)
            del x["k_cache"], x["v_cache"]
            x["k_cache"], x["v_cache"], self.table = pg["k_pool"], pg["v_pool"], pg["block_table"]
            self.nblk, _, self.bs, _ = x["k_cache"].shape
            self.maxb = self.table.shape[1]
        if self.fp8:
            # the 8-bit cache: codes and per-row scales quantized on the GPU
            kc, ks = g.kv_quantize_fp8(x["k_cache"])
            vc, vs = g.kv_quantize_fp8(x["v_cache"])
            del x["k_cache"], x["v_cache"]
            x["k_cache"], x["v_cache"], x["k_scale"], x["v_scale"] = kc, vc, ks, vs
            self.cache_bytes = 2 * (kc.numel() + 4 * ks.numel())
            step_read = read_bytes * (w.D + 4) / (2 * w.D)
            names = ("k_cache", "v_cache", "k_scale", "v_scale")
        else:
            self.cache_bytes = 2 * x["k_cache"].numel() * 2
            step_read = read_bytes
            names = ("k_cache", "v_cache")
        free = torch.cuda.mem_get_info(dev)[0]
        self.ncopies = max(1, min(int(math.ceil(4 * l2 / step_read)),
                                  int(0.5 * free // self.cache_bytes)))
        self.caches = [tuple(x[n] for n in names)]
        for _ in range(1, self.ncopies):
            self.caches.append(tuple(x[n].clone() for n in names))
        self.x = x
        self.lens = x["attn_lens"]
        self.pos = x["append_pos"]
        self.out = torch.empty(tuple(x["q"].shape), dtype=torch.float32, device=dev)
        lh = self.lens.cpu().tolist()
        self.kv_bytes_bf16 = accounting.kv_bytes_read(lh, w.Hkv, w.D, window=w.window)
        self.kv_bytes = (accounting.kv_bytes_read_fp8(lh, w.Hkv, w.D) if self.fp8
                         else self.kv_bytes_bf16)
        self.sp = ctypes_void(stream.cuda_stream)

    def call(self, r, q=None, kn=None, vn=None, pos=None, lens=None, out=None, table=None):
        """One step on cache copy r through the C ABI: append this token's K/V
        and attend (fused kernel); T drafted tokens: their scoring pass; the
        8-bit cache: append, then attend.  Tensors default to the setup's own."""
        w, lib, c = self.w, self.lib, self.caches[r]
        P = lambda t: ctypes_void(t.data_ptr())  # noqa: E731
        q = P(self.x["q"] if q is None else q)
        kn = P(self.x["k_new"] if kn is None else kn)
        vn = P(self.x["v_new"] if vn is None else vn)
        pos = P(self.pos if pos is None else pos)
        lens = P(self.lens if lens is None else lens)
        out = P(self.out if out is None else out)
        sp = self.sp
        if self.fp8:
            rc = lib.gqa_decode_step_fp8(q, kn, vn, P(c[0]), P(c[1]), P(c[2]), P(c[3]), pos, out,
                                         w.B, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale), sp)
        elif self.table is not None:
            tp = P(self.table if table is None else table)
            rc = lib.gqa_decode_step_paged(q, kn, vn, P(c[0]), P(c[1]), tp, pos, out, w.B, w.Hq,
                                           w.Hkv, w.D, self.nblk, self.bs, self.maxb,
                                           float(w.scale), sp)
        elif w.T > 1:
            rc = lib.gqa_decode_attn_multi(q, P(c[0]), P(c[1]), lens, out, w.B, w.T, w.Hq, w.Hkv,
                                           w.D, w.Lmax, float(w.scale), sp)
        elif w.window is None:
            rc = lib.gqa_decode_step(q, kn, vn, P(c[0]), P(c[1]), pos, out, w.B, w.Hq, w.Hkv,
                                     w.D, w.Lmax, float(w.scale), sp)
        else:
            rc = lib.gqa_decode_step_window(q, kn, vn, P(c[0]), P(c[1]), pos, out, w.B, w.Hq,
                                            w.Hkv, w.D, w.Lmax, float(w.scale), int(w.window), sp)
        assert rc == 0, lib.kvattn_last_error()

    def launches_per_step(self):
        return 2

    def describe(self):
        w = self.w
        if self.fp8:
            return ("gqa_decode_step_fp8 (8-bit cache: E4M3 codes and one fp32 scale per row; "
                    "the quantized append fused into the attention kernel; kv_bytes_per_step "
                    "counts codes and scales)")
        if self.table is not None:
            return ("gqa_decode_step_paged (kv_append fused into the attention kernel, K/V "
                    "reached through the block table)")
        if w.T > 1:
            return ("gqa_decode_attn_multi (T new tokens scored in one pass over the cache, "
                    "which already holds their rows)")
        return "gqa_decode_step (kv_append fused into the attention kernel)"

    def free(self):
        import torch
        self.caches = self.x = self.out = self.lens = self.pos = self.table = None
        torch.cuda.synchronize(self.dev)
        torch.cuda.empty_cache()


def time_chained(S, steps, warmup):
    """Exactly `steps` steps, W untimed before them, chained in CUDA graphs of
    up to CHAIN_MAX steps (programmatic edges between their kernels, so a
    step's launch overlaps the previous step's tail).  Returns the elapsed
    milliseconds of the timed steps and the graph used most (for replays)."""
    import torch
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=S.stream):
                for i in range(n):
                    S.call(i % S.ncopies)
            graphs[n] = gr
        return graphs[n]

    L = max(1, min(steps, CHAIN_MAX))

    def run(k):
        for _ in range(k // L):
            graph_for(L).replay()
        if k % L:
            graph_for(k % L).replay()

    with torch.cuda.stream(S.stream):
        for r in range(S.ncopies):  # first calls allocate the workspace
            S.call(r)
    S.stream.synchronize()
    for n in {L, steps % L, min(warmup, L), warmup % L} - {0}:
        graph_for(n)
    torch.cuda.synchronize(S.dev)
    with torch.cuda.stream(S.stream):
        run(warmup)
    S.stream.synchronize()
    return run, graphs


def time_run(S, run, steps, before=None, after=None):
    """Events around exactly `steps` steps, with a barrier and a device
    synchronisation on both sides.  A short GPU sleep is queued ahead of the
    start event, so that the host has submitted the steps' graphs by the time
    the GPU reaches it: the timed region holds the steps' GPU work, not the
    submission latency of the first graph."""
    import torch
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if before:
        before()
    torch.cuda.synchronize(S.dev)
    with torch.cuda.stream(S.stream):
        torch.cuda._sleep(200000)  # ~0.1 ms at 2 GHz
        t0.record(S.stream)
        run(steps)
        t1.record(S.stream)
    torch.cuda.synchronize(S.dev)
    if after:
        after()
    return t0.elapsed_time(t1)


def kernel_alone(S, n):
    """The split-KV kernel timed by itself: events recorded just before and
    just after it inside each call (kvattn_set_kernel_events), steps issued
    one by one over the same cache rotation.  The records end the kernel's
    overlap with its neighbours, so this runs outside the timed region."""
    import torch

    import grouped_query_kv_gb300 as g
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    with torch.cuda.stream(S.stream):
        for b, a in evs:  # torch creates events on first record
            b.record(S.stream)
            a.record(S.stream)
        for r in range(3):
            S.call(r % S.ncopies)
    torch.cuda.synchronize(S.dev)
    try:
        with torch.cuda.stream(S.stream):
            for i, (b, a) in enumerate(evs):
                g.set_kernel_events(b, a)
                S.call(i % S.ncopies)
    finally:
        g.set_kernel_events(None, None)
    torch.cuda.synchronize(S.dev)
    us = sorted(1e3 * b.elapsed_time(a) for b, a in evs)
    return {"mean_us": sum(us) / len(us), "p10_us": us[len(us) // 10], "p50_us": us[len(us) // 2],
            "p90_us": us[(9 * len(us)) // 10], "launches": n}


def e2e_graphs(S, steps):
    """End to end through the public Python API with host buffers, the steps
    captured in CUDA graphs as a serving loop would run them: every step
    uploads its inputs from pinned host memory (one packed copy) and reads its
    output back into pinned host memory.  Uploads and downloads run on
    streams of their own with two buffer sets, so step i's upload and step
    i-1's download overlap the kernels around them.  Returns the timing and
    the bytes moved per step."""
    import torch

    import grouped_query_kv_gb300 as g
    w, dev, stream = S.w, S.dev, S.stream
    x = S.x
    if w.T > 1:
        send = [("q", x["q"]), ("lens", S.lens)]
    else:
        send = [("q", x["q"]), ("k_new", x["k_new"]), ("v_new", x["v_new"]), ("pos", S.pos)]
    if S.table is not None:
        send.append(("table", S.table))  # a paged server sends the block table with every step
    layout, nbuf = [], 0
    for name, t in send:
        nb = t.numel() * t.element_size()
        layout.append((name, nbuf, nb, t.dtype, tuple(t.shape)))
        nbuf += (nb + 255) // 256 * 256
    hbuf = torch.empty(nbuf, dtype=torch.uint8).pin_memory()
    for (name, o, nb, _, _), (_, t) in zip(layout, send):
        hbuf[o:o + nb].copy_(t.detach().cpu().contiguous().reshape(-1).view(torch.uint8))
    dbufs = [torch.empty(nbuf, dtype=torch.uint8, device=dev) for _ in range(2)]
    dviews = [{name: db[o:o + nb].view(dt).view(shp) for name, o, nb, dt, shp in layout}
              for db in dbufs]
    outs = [S.out, torch.empty_like(S.out)]
    houts = [torch.empty_like(S.out, device="cpu").pin_memory() for _ in range(2)]
    io = {"h2d": sum(nb for _, _, nb, _, _ in layout),
          "d2h": houts[0].numel() * houts[0].element_size()}
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)]
          for k in ("in_ready", "in_free", "out_ready", "out_free")}

    def step(i):
        s = i % 2
        v, o = dviews[s], outs[s]
        up.wait_event(ev["in_free"][s])          # step i-2's kernels are done with this set
        with torch.cuda.stream(up):
            dbufs[s].copy_(hbuf, non_blocking=True)
            ev["in_ready"][s].record(up)
        stream.wait_event(ev["in_ready"][s])
        stream.wait_event(ev["out_free"][s])     # step i-2's output has been read back
        c = S.caches[i % S.ncopies]
        if w.T > 1:
            g.gqa_decode_attn_multi(v["q"], c[0], c[1], v["lens"], w.scale, out=o, stream=stream)
        elif S.fp8:
            g.gqa_decode_step_fp8(v["q"], v["k_new"], v["v_new"], c[0], c[1], c[2], c[3],
                                  v["pos"], w.scale, out=o, stream=stream)
        elif S.table is not None:
            g.gqa_decode_step_paged(v["q"], v["k_new"], v["v_new"], c[0], c[1], v["table"],
                                    v["pos"], w.scale, out=o, stream=stream)
        else:
            g.gqa_decode_step(v["q"], v["k_new"], v["v_new"], c[0], c[1], v["pos"], w.scale,
                              out=o, stream=stream, window=w.window)
        ev["in_free"][s].record(stream)
        ev["out_ready"][s].record(stream)
        down.wait_event(ev["out_ready"][s])
        with torch.cuda.stream(down):
            houts[s].copy_(o, non_blocking=True)
            ev["out_free"][s].record(down)

    # eager: the host issues every copy and call (its issue time is reported)
    for i in range(6):
        step(i)
    torch.cuda.synchronize(dev)
    n_e = max(1, min(steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    h0 = time.perf_counter()
    for i in range(n_e):
        step(i)
    host_us = 1e6 * (time.perf_counter() - h0) / n_e
    e1.record(down)
    torch.cuda.synchronize(dev)
    eager_ms = e0.elapsed_time(e1) / n_e

    # graphs: the same steps captured (both side streams join the capture
    # through events recorded on the capturing stream)
    L = max(2, min(steps, 200))
    L += L % 2  # whole buffer-set pairs per graph
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for s in range(2):
            ev["in_free"][s].record(stream)
            ev["out_free"][s].record(stream)
        for i in range(L):
            step(i)
        for s in range(2):
            stream.wait_event(ev["out_free"][s])
            stream.wait_event(ev["in_free"][s])
    torch.cuda.synchronize(dev)
    gr.replay()
    torch.cuda.synchronize(dev)
    reps = max(1, int(math.ceil(steps / L)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        h0 = time.perf_counter()
        for _ in range(reps):
            gr.replay()
        ghost_us = 1e6 * (time.perf_counter() - h0) / (reps * L)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = e0.elapsed_time(e1) / (reps * L)
    return {"graph_ms": graph_ms, "graph_steps": reps * L, "graph_host_us": ghost_us,
            "eager_ms": eager_ms, "eager_steps": n_e, "eager_host_us": host_us, "io": io}


def config_line(S, ms_step, kern, peak):
    kv = S.kv_bytes
    d = {"us_per_step": 1e3 * ms_step, "gbs": kv / (ms_step / 1e3) / 1e9,
         "frac": kv / (ms_step / 1e3) / 1e9 / peak,
         "kernel_alone_us": kern["mean_us"],
         "kernel_alone_frac": kv / (kern["mean_us"] / 1e6) / 1e9 / peak,
         "kv_bytes_per_step": kv, "seq_steps_per_s": S.w.B / (ms_step / 1e3),
         "tokens_scored_per_s": S.w.B * S.w.T / (ms_step / 1e3),
         "rotating_copies": S.ncopies}
    if S.fp8:
        d["bf16_equivalent_gbs"] = S.kv_bytes_bf16 / (ms_step / 1e3) / 1e9
    return d


def gpu_arm(a, w):
    import torch
    import torch.distributed as dist

    import grouped_query_kv_gb300 as g
    from grouped_query_kv_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = g.lib()
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    S = Setup(w, rank_seed(a.seed, rank), dev, lib, stream)
    g.check_device_error(stream)

    # ---- warm-up, then exactly K timed steps (max over ranks)
    run, graphs = time_chained(S, a.steps, a.warmup)
    clocks = Clocks(local)

    def barrier():
        if world > 1:
            dist.barrier()
    clocks.start()
    ms_total = time_run(S, run, a.steps, before=barrier, after=barrier)
    clk = clocks.stop()
    g.check_device_error(stream)
    local_ms_step = ms_total / a.steps
    ms_total, job_bytes = over_ranks(ms_total, S.kv_bytes * a.steps, world, dev)
    ms_step = ms_total / a.steps
    value = job_bytes / (ms_total / 1e3) / 1e9

    # ---- spread of the step time, outside the timed region: events around
    # each replay of a chain of steps
    gsp = graphs[max(graphs)]
    reps = max(10, min(200, 4000 // max(graphs)))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for k in range(reps):
            gsp.replay()
            evs[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(1e3 * evs[k].elapsed_time(evs[k + 1]) / max(graphs) for k in range(reps))
    spread = {"p10": per[reps // 10], "p50": per[reps // 2], "p90": per[(9 * reps) // 10],
              "over": "%d replays of the %d-step chain (us per step)" % (reps, max(graphs))}

    # ---- the split-KV kernel alone (the dominant kernel of the step)
    kern = kernel_alone(S, 100)
    kern_gbs = S.kv_bytes / (kern["mean_us"] / 1e6) / 1e9
    step_gbs = S.kv_bytes / (local_ms_step / 1e3) / 1e9
    g.check_device_error(stream)

    # ---- end to end with host buffers
    e2e = e2e_graphs(S, a.e2e_steps)
    g.check_device_error(stream)
    e2e_ms, e2e_bytes = over_ranks(e2e["graph_ms"], S.kv_bytes, world, dev)
    e2e_val = e2e_bytes / (e2e_ms / 1e3) / 1e9
    eager_ms, _ = over_ranks(e2e["eager_ms"], S.kv_bytes, world, dev)

    traffic = stored_traffic(w.name)
    step_desc = S.describe()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "Lmax": w.Lmax, "window": w.window, "seq_len": int(S.lens.max().item()),
                   "kv_bytes_per_step": S.kv_bytes,
                   "l2": "inputs larger than L2: %d rotating cache copies, %.0f MB (%.1fx L2)"
                         % (S.ncopies, S.ncopies * S.cache_bytes / 1e6,
                            S.ncopies * S.cache_bytes / S.l2),
                   "T": w.T, "block_size": w.block_size, "kv_dtype": w.kv_dtype,
                   "step": step_desc + ", steps chained in CUDA graphs of up to %d steps"
                           % CHAIN_MAX,
                   "numerics": "bf16 in, fp32 accumulate and out",
                   "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world},
        "us_per_step_spread": spread,
        "seq_steps_per_s": world * w.B * a.steps / (ms_total / 1e3),
        "tokens_scored_per_s": world * w.B * w.T * a.steps / (ms_total / 1e3),
        "bf16_equivalent_gbs": world * S.kv_bytes_bf16 * a.steps / (ms_total / 1e3) / 1e9,
        "us_per_step": 1e3 * ms_step,
        "hbm_fraction": (S.kv_bytes / (local_ms_step / 1e3) / 1e9) / peak,
        "roofline": {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                     "frac": step_gbs / peak,
                     "frac_of_nominal": step_gbs / NOMINAL_HBM_GBS,
                     "traffic": traffic.get(_decode_kernel_name(traffic)) if traffic else None,
                     "traffic_by_kernel": traffic,
                     "kernel": "the split-KV attention kernel of %s: one launch per step, "
                               "back to back in the timed region, so its average launch "
                               "interval there is the step time (the combine runs beside its "
                               "tail and the next launch's prologue beside the combine)"
                               % step_desc.split(" (")[0],
                     "alone": {"achieved": kern_gbs, "frac": kern_gbs / peak,
                               "frac_of_nominal": kern_gbs / NOMINAL_HBM_GBS, "duration": kern,
                               "source": "CUDA events recorded just before and after the "
                                         "split-KV kernel inside each of %d steps issued one by "
                                         "one after the timed region (kvattn_set_kernel_events)"
                                         "; without a neighbour to overlap, its launch and "
                                         "prologue show in full" % kern["launches"]},
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "peak_source": "%s hbm_gbs (MEASURED_PEAKS.json)" % peak_kind
                     if peak_kind == "measured" else "fallback 6800 GB/s"},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": e2e["io"]["h2d"],
                "d2h_bytes_per_step": e2e["io"]["d2h"], "ms_per_step": e2e_ms,
                "steps": e2e["graph_steps"], "host_issue_us_per_step": e2e["graph_host_us"],
                "api": "grouped_query_kv_gb300.%s per step, with its upload (one packed copy "
                       "from pinned memory) and download on their own streams, double-buffered, "
                       "the steps captured in CUDA graphs" % step_desc.split(" (")[0],
                "eager": {"value": S.kv_bytes / (eager_ms / 1e3) / 1e9, "unit": "GB/s",
                          "ms_per_step": eager_ms, "steps": e2e["eager_steps"],
                          "host_issue_us_per_step": e2e["eager_host_us"],
                          "api": "the same steps issued one by one from Python"}},
        "gpu_launches": S.launches_per_step() * a.steps,
        "clocks": clk,
    }
    S.free()
    del S

    # ---- the other target shapes, each timed the same way in this run
    if not a.no_per_config and rank == 0 and world == 1:
        pcs = {}
        clocks_pc = Clocks(local)
        clocks_pc.start()
        for name in PER_CONFIG:
            if name == w.name or name not in wl.WORKLOADS:
                continue
            wp = wl.WORKLOADS[name]
            Sp = Setup(wp, a.seed, dev, lib, stream)
            est_ms = max(0.01, Sp.kv_bytes / 6.0e9)
            k = int(max(20, min(2000, 250.0 / est_ms)))
            runp, _ = time_chained(Sp, k, 5)
            msp = time_run(Sp, runp, k) / k
            kp = kernel_alone(Sp, 20)
            g.check_device_error(stream)
            pcs[name] = config_line(Sp, msp, kp, peak)
            pcs[name]["steps"] = k
            pcs[name]["step"] = Sp.describe()
            Sp.free()
            del Sp, runp
        line["per_config"] = pcs
        line["per_config_clocks"] = clocks_pc.stop()

    if rank == 0 and not a.no_cpu_baseline:
        dt, nb, by, threads, reps = oracle_sample(w, a.seed, a.cpu_seconds)
        line["cpu_baseline"] = {
            "value": by / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (all heads) x %d repetitions, %.1f s, "
                      "double precision; %s" % (nb, w.B, reps, dt, cpu_model())}
        dt1, nb1, by1, _, reps1 = oracle_sample(w, a.seed, a.cpu_seconds / 4, threads=1)
        line["cpu_baseline"]["single_thread"] = {
            "value": by1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
            "sample": "%d sequences x %d repetitions, %.1f s" % (nb1, reps1, dt1)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _decode_kernel_name(traffic):
    for k in traffic:
        if k.startswith("decode"):
            return k
    return next(iter(traffic))


def ctypes_void(v):
    import ctypes
    return ctypes.c_void_p(v)


def main():
    a = parse()
    from grouped_query_kv_gb300 import workloads as wl
    if a.workload not in wl.WORKLOADS:
        print("unknown workload %r; one of %s" % (a.workload, ", ".join(wl.CONFIG_ORDER)),
              file=sys.stderr)
        return 2
    w = wl.WORKLOADS[a.workload]
    if a.warmup < 3:
        a.warmup = 3
    if a.impl == "reference":
        return reference_arm(a, w)
    return gpu_arm(a, w)


if __name__ == "__main__":
    sys.exit(main())
