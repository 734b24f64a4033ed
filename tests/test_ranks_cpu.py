"""The N > 1 host path of bench.py on CPU: two gloo ranks, each with its own
batch, combine their timing as the whole-job contract asks (the slowest
rank's time, every rank's KV bytes).  No GPU: the path has no data-path
collective, so the reduction of the timing is all there is to cover."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from grouped_query_kv_gb300 import accounting  # noqa: E402
from grouped_query_kv_gb300 import workloads as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, units, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port,
                            rank=rank, world_size=world)
    try:
        got = bench.over_ranks(ms[rank], units[rank], world, torch.device("cpu"))
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%r %r\n" % got)
    finally:
        dist.destroy_process_group()


def test_over_ranks_two_gloo_ranks(tmp_path):
    world = 2
    ms = [12.5, 17.25]
    units = [3.0e9, 5.5e9]
    mp.start_processes(_rank_main, args=(world, _free_port(), ms, units, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        t, u = (float(v) for v in open(tmp_path / ("rank%d.txt" % r)).read().split())
        assert t == max(ms)
        assert u == sum(units)


def test_over_ranks_single_rank_is_identity():
    assert bench.over_ranks(3.5, 7.0, 1, None) == (3.5, 7.0)


def test_ranks_draw_independent_batches():
    # weak scaling: every rank gets a different, equally shaped problem
    w = wl.WORKLOADS["llama70b_gqa_ragged"]
    l0 = wl.attn_lens(w, bench.rank_seed(0, 0))
    l1 = wl.attn_lens(w, bench.rank_seed(0, 1))
    assert l0.shape == l1.shape
    assert not torch.equal(l0, l1)
    # the job's bytes are the sum of the ranks' own (ragged) bytes
    b0 = accounting.kv_bytes_read(l0.tolist(), w.Hkv, w.D)
    b1 = accounting.kv_bytes_read(l1.tolist(), w.Hkv, w.D)
    assert b0 != b1
