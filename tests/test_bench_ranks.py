"""The multi-rank host logic of bench.py on CPU: gloo process groups of two
ranks (the layer itself runs as independent replicas, so the only cross-rank
step is the max-over-ranks timing and rank 0 printing)."""
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    # rank r timed its region in 10 + r ms (mean 1 - r ms): the slowest rank decides both
    got = bench.max_over_ranks([10.0 + rank, 1.0 - rank], world, "cpu")
    torch.distributed.barrier()
    q.put((rank, got))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 1.0]


def test_replica_throughput_and_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]
    # two replicas of 8 tokens x 10 steps in 11 ms (max over ranks)
    assert abs(bench.replica_tokens_per_s(2, 8, 10, 11.0) - 2 * 8 * 10 / 0.011) < 1e-6


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_json_line_both_weight_formats():
    """Rank 0 of the reference arm prints one JSON line with the contract's keys
    (the oracle timed on the host cores), for both weight formats."""
    import json
    for extra in ([], ["--weights", "bfp8"]):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                            "tiny", "--steps", "1", "--warmup", "1", *extra],
                           env=dict(os.environ, RANK="0", WORLD_SIZE="1"), capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        lines = [l for l in r.stdout.splitlines() if l.strip()]
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
        assert d["higher_is_better"] is True and d["dtype"] == "f64"
        assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}
        assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
        assert ("block-FP8" in d["config"]["workload"]) == bool(extra)
