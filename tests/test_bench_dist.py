"""The multi-rank path of bench.py without a GPU: two gloo ranks on the CPU.
Each rank times its own replica; the line must carry the slowest rank's time
and the whole job's tokens over it (weak scaling), which is what rank 0
prints."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    assert bench.dist_env() == (ws, rank, rank)
    local_ms = 2.0 + 3.0 * rank                 # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, ws, torch.device("cpu"))
    out[rank] = (ms, bench.whole_job_rate(16384, ws, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    for rank in range(ws):
        ms, value = res[rank]
        assert ms == 5.0
        assert value == pytest.approx(2 * 16384 / 5e-3 / 1e6)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_rate(1000, 1, 1.0) == pytest.approx(1.0)
