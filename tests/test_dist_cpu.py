"""The multi-process side of bench.py on CPU ranks (gloo, world size 2): the
process group set-up, the barrier, the max over ranks that the whole-job
timing uses, and the reference arm printing on rank 0 only."""
import io
import json
import os
import socket
import sys
import types
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), BENCH_GLOO="1")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(w, float(10 + rank))
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), w, r)
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": m, "printed": buf.getvalue()}, f)


def test_two_gloo_ranks(tmp_path):
    pytest.importorskip("torch.distributed")
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(x["max"] == 10.0 + world - 1 for x in res)  # every rank sees the slowest rank's time
    assert res[1]["printed"] == ""                          # only rank 0 prints
    line = json.loads(res[0]["printed"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0


# ---------------------------------------------------------------- expert parallelism on CPU ranks

def test_expert_shards_cover_every_expert_once():
    sys.path.insert(0, ROOT)
    from bit_expert_ffn_gb300.model import expert_shards

    for E, world in ((512, 8), (16, 3), (33, 4), (7, 7), (1, 1)):
        sh = expert_shards(E, world)
        assert len(sh) == world and sh[0][0] == 0 and sh[-1][1] == E
        assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
        sizes = [e1 - e0 for e0, e1 in sh]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        expert_shards(4, 5)


def _ep_rank_main(rank, world, port, out_dir):
    """One expert shard on a CPU rank: this rank's experts' terms (and the shared expert on rank 0) from the
    oracle, summed over the ranks by the library's ep_all_reduce, against the whole layer."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import ep_all_reduce, expert_shards
    from helpers import host_layer

    dist.init_process_group("gloo", rank=rank, world_size=world)
    E, k, T = 16, 4, 6
    arena, wr, b, shared = host_layer(seed=5, layer=1, bits=2, H=256, I=128, E=E, Is=128, zipf=1.1)
    x = synth.verify_window(5, T, 256)
    ids, w = oracle.topk(oracle.router_logits(x, wr, b).astype(np.float32), k)
    e0, e1 = expert_shards(E, world)[rank]
    mine = (ids >= e0) & (ids < e1)
    part = oracle.moe_layer(2, x, ids, np.where(mine, w, 0.0), *arena, shared=shared if rank == 0 else None)
    out = torch.from_numpy(part)
    ep_all_reduce(out)
    full = oracle.moe_layer(2, x, ids, w, *arena, shared=shared)
    err = float(np.linalg.norm(out.numpy() - full) / np.linalg.norm(full))
    pairs = torch.tensor([int(mine.sum())], dtype=torch.int64)
    dist.all_reduce(pairs)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"ep{rank}.json"), "w") as f:
        json.dump({"err": err, "pairs": int(pairs.item()), "mine": int(mine.sum())}, f)


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_layer_on_gloo_ranks(tmp_path, world):
    pytest.importorskip("torch.distributed")
    mp.spawn(_ep_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"ep{r}.json")) for r in range(world)]
    assert all(r["err"] <= 1e-12 for r in res)       # every rank holds the whole layer
    assert all(r["pairs"] == 6 * 4 for r in res)      # each (token, slot) pair computed by exactly one shard
    assert all(r["mine"] > 0 for r in res)
