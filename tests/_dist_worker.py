"""Child process of tests/test_bench_dist.py: one gloo rank that runs bench.py's cross-rank pieces."""
import os


def run(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, local = bench.dist_info()
        slow = bench.slowest_rank(10.0 + 5.5 * rank, dist)    # the per-rank step time of bench.py
        dist.barrier()
        queue.put((rank, r, w, local, slow))
    finally:
        dist.destroy_process_group()
