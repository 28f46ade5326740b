"""bench.py's multi-rank host logic with world size 2 on CPU (gloo), launched as the
driver launches it: torch.distributed.run, one process per rank, 127.0.0.1."""

import json
import os
import socket
import subprocess
import sys

from tests.conftest import ROOT


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=300):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    return [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]


def test_barrier_and_max_over_ranks_world_2(tmp_path):
    _torchrun([os.path.join("tests", "multirank_probe.py"), str(tmp_path)])
    lines = [json.load(open(tmp_path / f"rank_{r}.json", encoding="utf-8")) for r in (0, 1)]
    assert [l["rank"] for l in lines] == [0, 1]
    for l in lines:
        assert l["world"] == 2 and l["local"] == l["rank"]
        assert l["max"] == 11.5  # the larger of 1.5 (rank 0) and 11.5 (rank 1), on every rank


def test_reference_arm_world_2_prints_one_line_from_rank_0():
    lines = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
                       "--workload", "tiny"])
    assert len(lines) == 1, lines
    l = lines[0]
    assert l["impl"] == "reference" and l["n_gpus"] == 2 and l["steps"] == 2 and l["warmup"] == 3
    assert l["value"] > 0 and l["cpu_baseline"]["kind"] == "oracle"
    assert l["e2e"]["h2d_bytes_per_step"] == 0 and l["scaling"] == "weak"


def test_reference_arm_single_process_line_contract():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--workload", "tiny"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-4000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    l = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in l, k
    assert l["n_gpus"] == 1 and l["impl"] == "reference" and l["higher_is_better"] is True
    assert l["config"]["workload"] == "tiny" and l["cpu_baseline"]["value"] == l["value"]
    assert l["e2e"]["value"] == l["value"] and l["e2e"]["unit"] == l["unit"]
