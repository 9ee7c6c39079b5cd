"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

The layer does not shard: N GPUs run N independent replicas, joined only by
the timing barrier and the max-over-ranks reduction of the elapsed time.
These tests run that plumbing without a GPU: the reduction returns the
slowest rank's time on every rank, and under torchrun only rank 0 prints the
reference arm's JSON line while the other rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    v = bench.max_over_ranks(w, float(10 * (r + 1)), "cpu")
    out.put((r, w, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 20.0), (1, 2, 20.0)]


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "4", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "tokens/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_streamed_replay_counts_and_comparison():
    """The stored oracle replay of the streamed workload parses into every
    run and layer, holds the policy's identities, and the comparison names the
    first counter that differs."""
    sys.path.insert(0, ROOT)
    import bench
    exp = bench.streamed_expected()
    assert set(exp) == {"independent", "chained_off", "chained_on"}
    for run, rows in exp.items():
        assert len(rows) == 4
        for l, (hits, misses, evictions, la_copies, la_hits) in enumerate(rows):
            assert hits + misses == 256 * 16                    # 256 one-token steps, top-16
            assert la_hits <= la_copies
            if run != "chained_on" or l == 0:                   # no lookahead: misses fill
                assert la_copies == 0                           # 64 empty slots, then evict
                assert evictions == misses - 64
    assert exp["independent"][0] == exp["chained_off"][0] == exp["chained_on"][0]  # layer 0 alike
    st = [dict(zip(bench.COUNT_KEYS, r)) for r in exp["chained_on"]]
    assert bench.replay_match(exp["chained_on"], st) == "equal"
    st[2]["lookahead_hits"] += 1
    v = bench.replay_match(exp["chained_on"], st)
    assert v.startswith("differs") and "layer 2 lookahead_hits" in v
    assert bench.replay_match(None, st) == "no stored replay"
