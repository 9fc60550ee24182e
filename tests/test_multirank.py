"""The benchmark's multi-rank path on CPU (gloo, world size 2): decode
attention shards by replica with no exchange on the data path, so the only
cross-rank steps are the slowest-rank time and the whole-job throughput, and
the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 1.0 + 0.5 * rank          # rank 1 is the slow replica
    got = bench.rank_max(dist, world, ms, "cpu")
    gbs = bench.aggregate_gbs(1e9, world, got)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
        json.dump({"ms": got, "gbs": gbs}, f)


def test_rank_max_and_aggregate_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    for rank in range(2):
        r = json.load(open(tmp_path / ("r%d.json" % rank)))
        assert r["ms"] == 1.5                      # every rank sees the slowest time
        assert abs(r["gbs"] - 2 * 1e9 / 1.5e-3 / 1e9) < 1e-9  # both ranks' bytes over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(None, 1, 3.25, "cpu") == 3.25
    assert bench.aggregate_gbs(2e9, 1, 2.0) == 1000.0


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--config", "tiny"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
