"""The multi-rank host path with world_size 2 on CPU (gloo): every rank computes the same
owner plan, the owned sets partition the table, per-rank owner groups get distinct seeds,
and the step time reduces to the maximum over ranks."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import newton_schulz_orthogonalized_gb300 as nsm
        import synth
        shapes = synth.workload("split_moe").muon_shapes
        owner, load = nsm.assign_owners(shapes, world, "gram")
        plans = [None] * world
        dist.all_gather_object(plans, [int(o) for o in owner])
        mine = [i for i, o in enumerate(owner) if o == rank]
        owned = [None] * world
        dist.all_gather_object(owned, mine)
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_workload("llama7b", rank).seed)
        mx = bench.max_over_ranks(10.0 + rank, dist, torch.device("cpu"))
        out[rank] = {"plans_equal": all(p == plans[0] for p in plans),
                     "owned": owned, "n": len(shapes), "seeds": seeds, "max": mx}
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for r in range(world):
        res = out[r]
        assert res["plans_equal"]
        flat = sorted(i for part in res["owned"] for i in part)
        assert flat == list(range(res["n"]))          # every matrix owned exactly once
        assert len(set(res["seeds"])) == world          # independent owner groups
        assert res["max"] == 10.0 + world - 1           # slowest rank sets the step time
