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
