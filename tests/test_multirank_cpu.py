"""The N > 1 path of bench.py on CPU with the gloo backend, world size 2.

Decode attention shards by request (each rank owns its requests' pages, as the
kLLM article's request-level data parallelism does), so the only cross-rank
steps are the timing barrier and the max/sum reductions of the measured
numbers.  These run here over gloo; the reference arm runs under torchrun with
rank 0 alone printing its line."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import os, sys, json
sys.path.insert(0, os.environ["PFKV_ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
rank, ws = dist.get_rank(), dist.get_world_size()
bench.barrier(ws)
mx = bench.max_over_ranks(1.5 * (rank + 1), ws)
sm = bench.sum_over_ranks(10.0 * (rank + 1), ws)
with open(os.path.join(os.environ["PFKV_OUT"], f"rank{rank}.json"), "w") as f:
    json.dump({"rank": rank, "max": mx, "sum": sm}, f)
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout, out_dir=""):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, PFKV_ROOT=ROOT, PFKV_OUT=str(out_dir), CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def test_rank_reductions_over_gloo(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    r = _torchrun([str(script)], timeout=300, out_dir=tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    out = [json.load(open(tmp_path / f"rank{k}.json")) for k in range(2)]
    assert sorted(o["rank"] for o in out) == [0, 1]
    for o in out:
        assert o["max"] == 3.0 and o["sum"] == 30.0


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
                   "--oracle-requests", "1"], timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "long_splitkv_b8_h64kv8_p64"
