"""Rank worker for tests/test_multi_rank_cpu.py (run under torchrun, gloo on CPU).

Checks the benchmark's multi-rank host logic: process-group setup from the
torchrun environment, the barrier, and the max over ranks of a per-rank time.
Prints one line per rank: "rank <r> world <w> max <m>".
"""
import importlib.util
import pathlib
import sys

ROOT = pathlib.Path(__file__).resolve().parents[1]
spec = importlib.util.spec_from_file_location("bench", ROOT / "bench.py")
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)

world, rank, local = bench.dist_setup()
bench.barrier(world)
m = bench.max_over_ranks(1.5 + rank, world)   # per-rank "times" 1.5 and 2.5
bench.barrier(world)
print(f"rank {rank} world {world} max {m}", flush=True)
if world > 1:
    import torch.distributed as dist
    dist.destroy_process_group()
sys.exit(0)
