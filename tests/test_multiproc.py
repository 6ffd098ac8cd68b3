"""The benchmark's multi-rank host logic on CPU: two processes over gloo
(world size 2, rendezvous on 127.0.0.1).  Each rank runs an independent
replica, so the only cross-rank steps are the barrier around the timed region
and the max of the per-rank step times; the job's value is all ranks' tokens
over the slowest rank's time."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        bench.barrier(ws)
        # per-rank step times; the job takes the slowest
        ms = 10.0 + 5.0 * rank
        ms_max = bench.reduce_max(ms, ws)
        value = bench.aggregate(ms_max, tokens_per_rank_step=1000, world=ws)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ws": ws, "rank": r, "local": local, "ms_max": ms_max, "value": value}, f)
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_and_aggregate(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, x in enumerate(res):
        assert x["ws"] == 2 and x["rank"] == r and x["local"] == r
        assert x["ms_max"] == 15.0          # the slower rank's time on every rank
        # 2 ranks x 1000 tokens in 15 ms
        assert abs(x["value"] - 2 * 1000 / 0.015) < 1e-6


def test_single_rank_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate(2.0, 500, 1) == 500 / 0.002


def test_reference_arm_prints_on_rank_zero_only():
    """Under a 2-rank launch the reference arm (the CPU oracle) runs and
    prints on rank 0 only; the other rank exits 0 without work."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "causal_f32_n256", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "causal_f32_n256", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    # the fields the reference line carries besides the base contract's
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"] == "causal_f32_n256"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
