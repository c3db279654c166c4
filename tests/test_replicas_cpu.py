"""The N > 1 path of the benchmark on the CPU (gloo, world size 2): the
decode step does not shard, so N GPUs run N replicas and only the timing is
combined — the slowest rank's time (max over ranks) over all ranks' tokens.
These tests run that combination and the reference arm's rank handling under
torch.distributed.run with 127.0.0.1 rendezvous."""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, nproc=2, timeout=600):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run(cmd, capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def test_max_over_ranks_and_aggregate_with_gloo(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import json, os, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo")
        rank, ws = dist.get_rank(), dist.get_world_size()
        t = 0.5 + rank  # rank 1 is the slow one
        t_max = bench.max_over_ranks(t, ws, "cpu")
        out = {{"rank": rank, "t_max": t_max, "value": bench.aggregate_us_per_token(t_max, 100, ws)}}
        with open(os.path.join({str(tmp_path)!r}, f"r{{rank}}.json"), "w") as f:
            json.dump(out, f)
        dist.destroy_process_group()
    """))
    res = torchrun([str(script)])
    assert res.returncode == 0, res.stderr[-3000:]
    outs = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for o in outs:
        assert o["t_max"] == 1.5
        # 2 replicas x 100 tokens in 1.5 s (the slower rank's time)
        assert abs(o["value"] - 1.5e6 / 200) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25
    assert bench.aggregate_us_per_token(0.25, 50, 1) == 5000.0


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    res = torchrun([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                    "--gpus", "2", "--steps", "1", "--warmup", "1"])
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2  # the launch size; only rank 0 worked
