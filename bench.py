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

def gpu_arm(a, w):
    import torch
    import torch.distributed as dist

    import grouped_query_kv_gb300 as g
    from grouped_query_kv_gb300 import accounting
    from grouped_query_kv_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = g.lib()
    peak, peak_kind = measured_peaks()

    # ---- inputs: `ncopies` caches so consecutive steps never hit in L2 (the
    # steps of one round read at least 4x L2 between them)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    cache_bytes = 2 * w.B * w.Hkv * w.Lmax * w.D * 2
    read_bytes = accounting.kv_bytes_read(wl.attn_lens(w, rank_seed(a.seed, rank)).tolist(),
                                          w.Hkv, w.D, window=w.window)
    ncopies = max(1, int(math.ceil(4 * l2 / read_bytes)))
    ncopies = min(ncopies, max(1, int(0.5 * torch.cuda.mem_get_info(dev)[0] // cache_bytes)))
    x = wl.make_inputs(w, seed=rank_seed(a.seed, rank), device=dev)
    table = None
    if w.block_size:
        # paged: the pools hold only the blocks the sequences use, scattered
        pg = wl.make_paged(w, x, seed=rank_seed(a.seed, rank))
        del x["k_cache"], x["v_cache"]
        x["k_cache"], x["v_cache"], table = pg["k_pool"], pg["v_pool"], pg["block_table"]
        cache_bytes = 2 * x["k_cache"].numel() * 2
        ncopies = max(1, int(math.ceil(4 * l2 / read_bytes)))
        ncopies = min(ncopies, max(1, int(0.5 * torch.cuda.mem_get_info(dev)[0] // cache_bytes)))
        nblk, _, bs, _ = x["k_cache"].shape
        maxb = table.shape[1]
    fp8 = w.kv_dtype == "fp8"
    if fp8:
        # the 8-bit cache: codes and per-row scales quantized on the GPU
        kc, ks = g.kv_quantize_fp8(x["k_cache"])
        vc, vs = g.kv_quantize_fp8(x["v_cache"])
        del x["k_cache"], x["v_cache"]
        x["k_cache"], x["v_cache"] = kc, vc
        cache_bytes = 2 * (kc.numel() + 4 * ks.numel())
        ncopies = max(1, int(math.ceil(4 * l2 / (read_bytes * (w.D + 4) / (2 * w.D)))))
        ncopies = min(ncopies, max(1, int(0.5 * torch.cuda.mem_get_info(dev)[0] // cache_bytes)))
        caches = [(kc, vc, ks, vs)]
        for r in range(1, ncopies):
            caches.append((kc.clone(), vc.clone(), ks.clone(), vs.clone()))
    else:
        caches = [(x["k_cache"], x["v_cache"])]
        for r in range(1, ncopies):
            caches.append((x["k_cache"].clone(), x["v_cache"].clone()))
    lens = x["attn_lens"]
    pos = x["append_pos"]
    out = torch.empty(tuple(x["q"].shape), dtype=torch.float32, device=dev)
    kv_bytes = accounting.kv_bytes_read(lens.cpu().tolist(), w.Hkv, w.D, window=w.window)
    # bf16-equivalent bytes: what the same attention reads from a bf16 cache
    kv_bytes_bf16 = kv_bytes
    if fp8:
        kv_bytes = accounting.kv_bytes_read_fp8(lens.cpu().tolist(), w.Hkv, w.D)

    stream = torch.cuda.Stream(device=dev)
    sp = ctypes_void(stream.cuda_stream)
    P = lambda t: ctypes_void(t.data_ptr())  # noqa: E731
    q_p, kn_p, vn_p, pos_p, out_p = map(P, (x["q"], x["k_new"], x["v_new"], pos, out))

    lens_p = P(lens)
    table_p = P(table) if table is not None else None

    def call_step(r):
        # one decode step: append this token's K/V and attend (fused kernel);
        # for T drafted tokens, their scoring pass over the cache
        if fp8:
            c = caches[r]
            rc = lib.kv_append_fp8(P(c[0]), P(c[1]), P(c[2]), P(c[3]), kn_p, vn_p, pos_p, w.B,
                                   w.Hkv, w.D, w.Lmax, sp)
            assert rc == 0, lib.kvattn_last_error()
            rc = lib.gqa_decode_attn_fp8(q_p, P(c[0]), P(c[1]), P(c[2]), P(c[3]), lens_p, out_p,
                                         w.B, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale), sp)
        elif table is not None:
            rc = lib.gqa_decode_step_paged(q_p, kn_p, vn_p, P(caches[r][0]), P(caches[r][1]),
                                           table_p, pos_p, out_p, w.B, w.Hq, w.Hkv, w.D, nblk,
                                           bs, maxb, float(w.scale), sp)
        elif w.T > 1:
            rc = lib.gqa_decode_attn_multi(q_p, P(caches[r][0]), P(caches[r][1]), lens_p, out_p,
                                           w.B, w.T, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale), sp)
        elif w.window is None:
            rc = lib.gqa_decode_step(q_p, kn_p, vn_p, P(caches[r][0]), P(caches[r][1]), pos_p,
                                     out_p, w.B, w.Hq, w.Hkv, w.D, w.Lmax, float(w.scale), sp)
        else:
            rc = lib.gqa_decode_step_window(q_p, kn_p, vn_p, P(caches[r][0]), P(caches[r][1]),
                                            pos_p, out_p, w.B, w.Hq, w.Hkv, w.D, w.Lmax,
                                            float(w.scale), int(w.window), sp)
        assert rc == 0, lib.kvattn_last_error()

    with torch.cuda.stream(stream):
        for r in range(ncopies):           # first calls allocate the workspace
            call_step(r)
    stream.synchronize()
    g.check_device_error(stream)

    # one graph runs the ncopies steps back to back (programmatic edges between
    # their kernels, so a step's launch overlaps the previous step's tail);
    # single-step graphs make up the remainder, so exactly K steps are timed
    chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(chain, stream=stream):
        for r in range(ncopies):
            call_step(r)
    singles = []
    for r in range(ncopies):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            call_step(r)
        singles.append(gr)
    torch.cuda.synchronize(dev)

    def run_steps(k):
        for _ in range(k // ncopies):
            chain.replay()
        for r in range(k % ncopies):
            singles[r].replay()

    # ---- warm-up, then exactly K timed steps
    with torch.cuda.stream(stream):
        run_steps(a.warmup)
    stream.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0.record(stream)
        run_steps(a.steps)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    g.check_device_error(stream)
    ms_total = t0.elapsed_time(t1)
    local_ms_step = ms_total / a.steps
    ms_total, job_bytes = over_ranks(ms_total, kv_bytes * a.steps, world, dev)
    ms_step = ms_total / a.steps
    value = job_bytes / (ms_total / 1e3) / 1e9
    # average duration of one step's launch over the timed region
    achieved = kv_bytes / (local_ms_step / 1e3) / 1e9

    # ---- spread of the step time, outside the timed region: events around
    # each replay of the ncopies-step chain
    reps = max(20, min(400, 4000 // ncopies))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for k in range(reps):
            chain.replay()
            evs[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(1e3 * evs[k].elapsed_time(evs[k + 1]) / ncopies for k in range(reps))
    spread = {"p10": per[reps // 10], "p50": per[reps // 2], "p90": per[(9 * reps) // 10],
              "over": "%d replays of the %d-step chain (us per step)" % (reps, ncopies)}

    # ---- end to end through the public Python API with host buffers.  A
    # step's inputs go up from pinned host memory in ONE copy (the tensors
    # packed side by side at 256-byte offsets) and its output comes back in
    # one copy.  Uploads and downloads run on streams of their own with two
    # buffer sets, so step i's upload and step i-1's download overlap the
    # kernels of the steps around them, as a serving loop would run them.
    if w.T > 1:
        send = [("q", x["q"]), ("lens", lens)]
    elif fp8:
        send = [("q", x["q"]), ("k_new", x["k_new"]), ("v_new", x["v_new"]),
                ("pos", pos), ("lens", lens)]
    else:
        send = [("q", x["q"]), ("k_new", x["k_new"]), ("v_new", x["v_new"]), ("pos", pos)]
    if table is not None:
        send.append(("table", table))  # a paged server sends the block table with every step
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
    outs = [out, torch.empty_like(out)]
    houts = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
    io = {"h2d": sum(nb for _, _, nb, _, _ in layout),
          "d2h": houts[0].numel() * houts[0].element_size()}
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)]
          for k in ("in_ready", "in_free", "out_ready", "out_free")}
    n_e2e = max(1, a.e2e_steps)

    def e2e_step(i):
        s = i % 2
        v, o = dviews[s], outs[s]
        up.wait_event(ev["in_free"][s])          # step i-2's kernels are done with this set
        with torch.cuda.stream(up):
            dbufs[s].copy_(hbuf, non_blocking=True)
            ev["in_ready"][s].record(up)
        stream.wait_event(ev["in_ready"][s])
        stream.wait_event(ev["out_free"][s])     # step i-2's output has been read back
        r = i % ncopies
        c = caches[r]
        if w.T > 1:
            g.gqa_decode_attn_multi(v["q"], c[0], c[1], v["lens"], w.scale, out=o, stream=stream)
        elif fp8:
            g.kv_append_fp8(c[0], c[1], c[2], c[3], v["k_new"], v["v_new"], v["pos"],
                            stream=stream)
            g.gqa_decode_attn_fp8(v["q"], c[0], c[1], c[2], c[3], v["lens"], w.scale, out=o,
                                  stream=stream)
        elif table is not None:
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

    for i in range(6):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    h0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    host_us = 1e6 * (time.perf_counter() - h0) / n_e2e  # host time to issue one step
    e1.record(down)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    e2e_ms, e2e_bytes = over_ranks(e2e_ms, kv_bytes, world, dev)
    e2e_val = e2e_bytes / (e2e_ms / 1e3) / 1e9
    g.check_device_error(stream)

    traffic = stored_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "Lmax": w.Lmax, "window": w.window, "seq_len": int(lens.max().item()),
                   "kv_bytes_per_step": kv_bytes,
                   "l2": "inputs larger than L2: %d rotating cache copies, %.0f MB (%.1fx L2)"
                         % (ncopies, ncopies * cache_bytes / 1e6, ncopies * cache_bytes / l2),
                   "T": w.T, "block_size": w.block_size, "kv_dtype": w.kv_dtype,
                   "step": ("kv_append_fp8 then gqa_decode_attn_fp8 (8-bit cache: E4M3 codes and "
                            "one fp32 scale per row; kv_bytes_per_step counts codes and scales), "
                            "steps chained in CUDA graphs" if fp8 else
                            "gqa_decode_step_paged (kv_append fused into the attention kernel, "
                            "K/V reached through the block table), steps chained in CUDA graphs"
                            if table is not None else
                            "gqa_decode_attn_multi (T new tokens scored in one pass over the "
                            "cache, which already holds their rows), steps chained in CUDA graphs"
                            if w.T > 1 else
                            "gqa_decode_step (kv_append fused into the attention kernel), "
                            "steps chained in CUDA graphs"),
                   "numerics": "bf16 in, fp32 accumulate and out",
                   "parallelism": "replicas" if world == 1 else "dp%d (independent batches)" % world},
        "us_per_step_spread": spread,
        "seq_steps_per_s": world * w.B * a.steps / (ms_total / 1e3),
        "tokens_scored_per_s": world * w.B * w.T * a.steps / (ms_total / 1e3),
        "bf16_equivalent_gbs": world * kv_bytes_bf16 * a.steps / (ms_total / 1e3) / 1e9,
        "us_per_step": 1e3 * ms_step,
        "hbm_fraction": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": sum(traffic.values()) if traffic else None,
                     "traffic_by_kernel": traffic,
                     "kernel": ("kv_append_fp8 + gqa_decode_attn_fp8 (append, 8-bit split-KV "
                                "kernel, combine), " if fp8 else
                                "gqa_decode_step_paged (fused append + split-KV kernel over "
                                "the block table + combine), " if table is not None else
                                "gqa_decode_attn_multi (split-KV kernel + combine), " if w.T > 1
                                else "gqa_decode_step (fused append + split-KV kernel + combine), ")
                               +
                               "average over the timed steps",
                     "peak_source": "%s hbm_gbs (MEASURED_PEAKS.json)" % peak_kind
                     if peak_kind == "measured" else "fallback 6800 GB/s"},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": io["h2d"],
                "d2h_bytes_per_step": io["d2h"], "ms_per_step": e2e_ms,
                "host_issue_us_per_step": host_us,
                "api": "grouped_query_kv_gb300.%s (eager; one packed upload and one download per step on their own streams, double-buffered)"
                       % ("kv_append_fp8 + gqa_decode_attn_fp8" if fp8 else
                          "gqa_decode_step_paged" if table is not None else
                          "gqa_decode_attn_multi" if w.T > 1 else "gqa_decode_step")},
        "gpu_launches": (3 if fp8 else 2) * a.steps,
        "clocks": clk,
    }
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
