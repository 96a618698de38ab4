"""The multi-rank report path of bench.py on CPU: two gloo ranks, each with its own
step time and token count, must agree on value = sum(tokens) / max(time)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        t_ms = [4.0, 5.5][r]                           # per-rank step time
        tokens = [1000, 3000][r]                       # per-rank tokens per step
        t_max = bench.reduce_max(t_ms, w)
        tok = bench.reduce_sum(tokens, w)
        out.put((r, t_max, tok, tok / (t_max / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_rank_report_reduction():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, t_max, tok, value in res:
        assert t_max == 5.5 and tok == 4000
        assert value == pytest.approx(4000 / 5.5e-3)
