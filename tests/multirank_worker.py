"""Worker of the two-rank gloo test (a module of its own so that spawned
processes can import it)."""
import os


def timing_rank(rank: int, world: int, port: int, local_ms: float, queue) -> None:
    import torch
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        job_ms = bench.max_over_ranks(local_ms, torch.device("cpu"))
        queue.put((rank, job_ms, bench.job_throughput(world, 2.0e9, 10, job_ms)))
    finally:
        dist.destroy_process_group()
