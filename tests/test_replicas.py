"""The multi-GPU path is independent replicas: check its bookkeeping with
two gloo ranks on the CPU (no data-path collective exists)."""

import os

import pytest
import torch.multiprocessing as mp


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from dense_decoder_layer_gb300 import replicas

    # rank r is slower by r ms and processed 512 tokens
    ms, tps = replicas.aggregate(10.0 + rank, 512)
    replicas.barrier()
    q.put((rank, ms, tps))
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_slowest_time_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tps in out:
        assert ms == pytest.approx(11.0)
        assert tps == pytest.approx(2 * 512 / 11.0e-3)


def test_single_process_aggregate():
    from dense_decoder_layer_gb300 import replicas

    ms, tps = replicas.aggregate(4.0, 100)
    assert ms == 4.0 and tps == pytest.approx(25000.0)
