"""The N > 1 host path on CPU (gloo, world size 2), as torchrun launches it.

The path is replicas only (every sequence's attention is independent; no
exchange step), so what N > 1 adds is host logic: the process group, the
barrier around the timed region, the maximum of the ranks' times, rank 0
alone printing the line, and the reference arm running on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, timeout=600):
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), *args]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_barrier_and_max_over_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    # each rank writes its own file (two ranks printing at once may interleave on stdout)
    script.write_text(
        "import json, sys\n"
        "import bench\n"
        "rank, world, local = bench.rank_info()\n"
        "dist = bench.dist_setup(world, local)\n"
        "bench.barrier(dist)\n"
        "m = bench.reduce_max(dist, 1.5 + 2.0 * rank)\n"
        "bench.barrier(dist)\n"
        "with open(sys.argv[1] + f'/rank{rank}.json', 'w') as f:\n"
        "    json.dump({'rank': rank, 'world': world, 'max': m}, f)\n")
    r = torchrun([str(script), str(tmp_path)])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{k}.json").read_text()) for k in range(2)]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    assert all(d["world"] == 2 and d["max"] == 3.5 for d in lines)


def test_reference_arm_prints_one_line_from_rank_zero():
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
                  "--ref-seqs", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["cpu_baseline"]["cores"] == 1
