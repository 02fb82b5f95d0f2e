"""Multi-replica aggregation on CPU: world_size 2 over gloo.

Each rank reports its own timed-region length and row count; the job's
figure is the summed rows over the slowest rank's time.  No data path
crosses ranks.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, rows, out_dir):
    import json
    import torch.distributed as dist
    from invariant_sequence_decode_gb300 import replicas
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert replicas.world() == (rank, world, rank)
        dist.barrier()
        agg = replicas.aggregate(elapsed[rank], rows[rank])
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(agg, f)
    finally:
        dist.destroy_process_group()


def test_single_replica_without_process_group():
    from invariant_sequence_decode_gb300 import replicas
    agg = replicas.aggregate(250.0, 40)
    assert agg == {"max_ms": 250.0, "rows": 40, "rows_per_s": 160.0, "world": 1}


def test_two_ranks_gloo(tmp_path):
    import json
    import torch.multiprocessing as mp
    elapsed = [120.0, 200.0]   # rank 1 is the slower replica
    rows = [40, 40]
    mp.start_processes(_rank_main, args=(2, _free_port(), elapsed, rows, str(tmp_path)), nprocs=2,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for agg in res:
        assert agg["world"] == 2
        assert agg["max_ms"] == 200.0
        assert agg["rows"] == 80
        assert agg["rows_per_s"] == pytest.approx(80 / 0.2)
    assert res[0] == res[1]
