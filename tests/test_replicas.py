"""The N > 1 path on the CPU: replicas only.  Requests are independent, so
N GPUs run N copies of the serving loop, each with its own pool, tree and
queue; nothing but the job's timing crosses ranks.  Two gloo ranks (127.0.0.1)
each serve the same host-side few-shot trace through their own cache; both
replicas must end in exactly the state one process reaches alone, and the
benchmark's reduction must take the slowest rank's time and count every
rank's work."""
from __future__ import annotations

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _serve_replica():
    """One replica's host path (admission, prompt commit, finish) over a
    small few-shot trace; returns its cache statistics and tree dump."""
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from synth import traces
    from synth.model import SynthModel

    tr = traces.few_shot(n_questions=24, max_new=6, batch_salt=1)
    model = SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu")
    cache = ra.RadixCache(1 << 16)
    runner = wl.Runner(cache, model, None)
    runner.serve([runner.request(tr.warm, 0)])
    admitted, waiting = runner.serve([runner.request(tr.prompt(i), tr.max_new) for i in range(len(tr.questions))])
    assert not waiting
    return cache.stats(), cache.dump()


def _rank(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import json

    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        stats, dump = _serve_replica()
        everyone = [None] * world
        dist.all_gather_object(everyone, (stats, dump))
        dist.barrier()
        slowest = bench.slowest_rank(10.0 + rank, world, "cpu")
        rate = bench.whole_job_rate(1000.0, world, slowest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"same": all(e == everyone[0] for e in everyone), "stats": stats, "dump": dump,
                       "slowest": slowest, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_match_one_process_and_the_slowest_rank_counts(built, tmp_path):
    import json

    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    alone_stats, alone_dump = _serve_replica()
    for r in range(world):
        got = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert got["same"]
        assert got["stats"] == alone_stats and got["dump"] == alone_dump
        assert got["slowest"] == pytest.approx(10.0 + world - 1)
        assert got["rate"] == pytest.approx(1000.0 * world / ((10.0 + world - 1) / 1e3))
