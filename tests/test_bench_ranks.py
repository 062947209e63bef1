"""bench.py's multi-rank path on the CPU: two gloo ranks under torchrun.

The decode path does not shard (one GPU serves a whole step), so `bench.py
--gpus N` runs N independent replicas: one process per GPU, a barrier on each
side of the timed steps, the step time taken as the maximum over ranks, and
one JSON line printed by rank 0. These tests run that host logic with
world size 2 on the gloo backend (no GPU): the rank helpers themselves, and the
reference arm, which rank 0 alone runs and prints.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=REPO, env=env, capture_output=True, text=True, timeout=timeout)


def test_rank_helpers_reduce_the_max_over_two_gloo_ranks(tmp_path):
    worker = tmp_path / "worker.py"
    worker.write_text(textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {REPO!r})
        import bench
        world, rank, local = bench.dist_setup()
        bench.barrier(world)
        m = bench.max_over_ranks(float(10 * rank + 1), world)
        bench.barrier(world)
        with open({str(tmp_path)!r} + f"/rank{{rank}}.txt", "w") as f:  # a file per rank: no interleaving
            f.write(f"rank={{rank}} world={{world}} local={{local}} max={{m}}")
        import torch.distributed as dist
        dist.destroy_process_group()
    """))
    r = torchrun([str(worker)])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    got = [(tmp_path / f"rank{k}.txt").read_text() for k in range(2)]
    assert got == ["rank=0 world=2 local=0 max=11.0", "rank=1 world=2 local=1 max=11.0"], got


def test_reference_arm_prints_one_line_from_rank_zero():
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    out = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(out) == 1, r.stdout[-2000:]
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 3 and line["warmup"] == 3
    assert line["config"]["parallelism"] == "replicas x2"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_carries_the_contract_keys():
    """One rank, no torchrun: the line the driver parses, with every key of the contract."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3"], cwd=REPO,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1"), capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    out = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(out) == 1, r.stdout[-2000:]
    line = json.loads(out[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["scaling"] == "weak" and line["data"] == "synthetic"
    assert line["config"]["workload"] == "batched_gqa" and line["config"]["parallelism"] == "replicas x1"
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
