"""The benchmark's multi-rank path on CPU: world size 2 over gloo, launched the
way the N-GPU bench is launched (torch.distributed.run, rendezvous on
127.0.0.1).  Checks the barrier and max-over-ranks helpers, and that the
reference arm prints exactly one JSON line (rank 0) while the other rank exits
0 without work."""
import json
import os
import re
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, timeout=240):
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""          # CPU ranks (gloo) even on a GPU host
    env.pop("TGEMM_FORCE_CFG", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port())] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_barrier_and_max_over_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import bench
        world, rank, local = bench.dist_setup()
        assert world == 2
        bench.barrier(world)
        m = bench.max_over_ranks(1.5 + rank, world)
        bench.barrier(world)
        print(f"rank {{rank}} max {{m}}", flush=True)
        import torch.distributed as dist
        dist.destroy_process_group()
    """))
    r = torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-2000:]
    # The two ranks share stdout, so their lines may interleave.
    found = sorted(re.findall(r"rank (\d) max ([0-9.]+)", r.stdout))
    assert found == [("0", "2.5"), ("1", "2.5")], r.stdout


def test_reference_arm_prints_once_under_torchrun():
    r = torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--config", "c0",
                  "--steps", "1", "--warmup", "3", "--ref-rows", "2"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
