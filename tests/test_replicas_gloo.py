"""The multi-process path of bench.py on CPU: world_size 2 over gloo.

The layer step does not shard (each GPU runs a whole replica with its own
weights, KV pool and batch), so the only cross-rank work is host-side: a
barrier around the timed region, the maximum of the ranks' step times, and
rank 0 alone printing.  These tests run that logic as two real processes."""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    r, w, local, pg = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank) and pg is not None
    # rank-dependent local step times: the job takes the slowest
    ms_local = 2.0 + 3.0 * rank
    ms, value = bench.replica_throughput(pg, w, 576, ms_local)
    bench.barrier(pg)
    # the reference arm runs on rank 0 only; the others leave without work or output
    buf = io.StringIO()
    if rank != 0:
        with redirect_stdout(buf):
            bench.run_reference(None, rank, w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms!r} {value!r} {buf.getvalue()!r}\n")
    pg.barrier()
    pg.destroy_process_group()


def test_replica_timing_takes_max_over_ranks_and_counts_all_tokens(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    rows = [open(tmp_path / f"rank{r}.txt").read().split(" ", 2) for r in range(world)]
    for ms, value, out in rows:
        assert float(ms) == 5.0                        # max(2.0, 5.0) on every rank
        assert float(value) == pytest.approx(world * 576 / 5e-3)
    assert rows[1][2].strip() == "''"                  # rank 1 printed nothing


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    r, w, local, pg = bench.dist_setup()
    assert (r, w, local, pg) == (0, 1, 0, None)
    assert bench.replica_throughput(None, 1, 100, 4.0) == (4.0, 100 / 4e-3)
