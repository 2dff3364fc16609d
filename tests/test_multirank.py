"""The multi-GPU host logic of bench.py on CPU: two gloo ranks agree on the
max-over-ranks time and on the whole-job throughput (weak scaling: each rank
decides its own batch; no collective on the decision path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import sys
    import torch.distributed as td
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    td.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]
    m = bench.max_over_ranks(local_ms, world, "cpu")
    v = bench.job_throughput(2048, world, 100, m)
    q.put((rank, m, v))
    td.barrier()
    td.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in out:
        assert m == 20.0
        assert v == pytest.approx(2048 * 2 * 100 / 0.020)


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(100, 1, 10, 1000.0) == pytest.approx(1000.0)


def _gather_rank(rank, world, port, q):
    import sys
    import torch
    import torch.distributed as td
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    td.init_process_group("gloo", rank=rank, world_size=world)
    from diffusion_decoding_token_gb300._binding import allgather_row_partials
    rows = 5
    mine = torch.arange(rows * 8, dtype=torch.float32).reshape(rows, 8) + 1000 * rank
    got = allgather_row_partials(mine)
    q.put((rank, got.numpy().tolist()))
    td.barrier()
    td.destroy_process_group()


def test_vocab_shard_exchange_orders_partials_by_rank():
    """The exchange of a vocabulary-sharded row pass: rank r's partial states
    land in slot r of every rank's [world, rows, 8] tensor (the merge takes
    the slices in vocabulary order)."""
    import numpy as np
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_gather_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    base = np.arange(40, dtype=np.float32).reshape(5, 8)
    for _, got in out:
        got = np.array(got)
        assert got.shape == (2, 5, 8)
        np.testing.assert_array_equal(got[0], base)
        np.testing.assert_array_equal(got[1], base + 1000)
