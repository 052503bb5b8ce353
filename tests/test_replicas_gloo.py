"""The N > 1 bench path on CPU: two gloo ranks, each an independent replica,
agree on the whole-job figure (the slowest rank's time, the units of both
ranks).  No GPU and no data-path collective are involved; the only
collective is the MAX reduction of the per-rank step times."""
import json
import os
import socket
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_rank = [3.0, 5.0][rank]  # rank 1 is the slower replica
        ms, value = bench.replica_aggregate(ms_rank, 96, world, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_units(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["ms"] == 5.0
        assert g["value"] == pytest.approx(2 * 96 / 0.005)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.replica_aggregate(4.0, 12288, 1)
    assert ms == 4.0 and value == pytest.approx(12288 / 0.004)
