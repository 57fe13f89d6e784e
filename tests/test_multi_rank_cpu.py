"""Multi-rank host path of bench.py on CPU: two gloo ranks under torchrun
(127.0.0.1 rendezvous). The data path has no collective; these check the
barrier, the max over ranks of the step time, and that only rank 0 prints the
result line (the reference arm, which times the oracle)."""
import json
import os
import re
import socket
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(*args, timeout=240):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", *args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_two_gloo_ranks_barrier_and_max():
    r = _torchrun(str(ROOT / "tests" / "dist_ranks.py"))
    assert r.returncode == 0, r.stderr[-2000:]
    # the two ranks share stdout, so their lines may interleave
    found = sorted(re.findall(r"rank (\d) world (\d) max ([0-9.]+)", r.stdout))
    assert found == [("0", "2", "2.5"), ("1", "2", "2.5")], r.stdout


def test_reference_arm_prints_once_under_two_ranks():
    r = _torchrun("bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    out = re.findall(r"\{.*\}", r.stdout)
    assert len(out) == 1, r.stdout
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
