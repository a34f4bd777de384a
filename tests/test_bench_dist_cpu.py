"""bench.py's multi-process path on CPU: two gloo ranks launched the way the
driver launches the GPU run (torch.distributed.run, 127.0.0.1), checking the
barrier, the max-over-ranks time, the whole-job throughput and that the
reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_replicas(tmp_path):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", DIST_TEST_OUT=str(tmp_path))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "tests", "dist_worker.py")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [json.loads((tmp_path / ("rank%d.json" % i)).read_text()) for i in range(2)]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    for d in lines:
        assert d["world"] == 2
        assert d["ms_max"] == 2.5                       # the slower replica
        assert abs(d["tokens_s"] - 2 * 4096 / 2.5e-3) < 1e-6 * d["tokens_s"]
    assert lines[1]["ref_skipped"] is True
