"""The multi-GPU bench path runs independent replicas (no collective on the data path): each rank decodes tokens
of its own and the job's time is the slowest rank's. Its host-side logic runs here as two gloo ranks on the CPU."""
import multiprocessing as mp
import os
import socket


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(10.0 + 3.5 * rank, dist, "cpu")
    alone = bench.max_over_ranks(10.0 + 3.5 * rank, None, "cpu")
    out.put((rank, slowest, alone, bench.rank_token_seed(1, rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_time_is_the_slowest_rank_and_tokens_differ():
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
    assert [r[1] for r in res] == [13.5, 13.5]          # every rank reports the slowest rank's time
    assert [r[2] for r in res] == [10.0, 13.5]          # one process: its own
    assert res[0][3] != res[1][3]                        # each replica decodes tokens of its own
