"""One rank of a multi-process CPU test of bench.py's host logic (gloo)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_rank", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def timing_rank(rank, world, port, ms_by_rank, tokens, out):
    """Joins a gloo group on 127.0.0.1, reduces this rank's step time as
    bench.py does, and reports (rank, job ms, job tokens/s)."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = load_bench()
        dist.barrier()
        ms = bench.slowest_rank_ms(ms_by_rank[rank], world)
        out.put((rank, ms, bench.job_tokens_per_s(tokens, world, ms)))
    finally:
        dist.destroy_process_group()
