"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1), the barrier,
max-over-ranks timing and the replica throughput (units of all ranks over the
slowest rank's time), and the reference arm's rank > 0 exit."""
import importlib.util
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    b = _bench()
    ws, r, local = b.dist_setup(None)
    b.barrier(ws)
    mx = b.max_over_ranks(1.5 + r, ws)                      # 1.5 on rank 0, 2.5 on rank 1
    value, ms_max = b.replica_value(10.0, 4.0 * (r + 1), ws)  # 10 units per rank, 4 / 8 ms
    b.barrier(ws)
    # the reference arm does its work on rank 0 only; other ranks return 0 at once
    ref_rc = None
    if r == 1:
        import types
        ref_rc = b.run_reference(types.SimpleNamespace(), None)
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump(dict(ws=ws, rank=r, local=local, mx=mx, value=value, ms_max=ms_max,
                       ref_rc=ref_rc), f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["ws"] == 2 and d["rank"] == r and d["local"] == r
        assert d["mx"] == 2.5                       # max over ranks, seen by both
        assert d["ms_max"] == 8.0
        assert d["value"] == pytest.approx(2 * 10.0 / 8e-3)  # both ranks' units / slowest time
    assert res[1]["ref_rc"] == 0
