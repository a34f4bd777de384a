"""The expert-parallel exchange over gloo on the CPU: 2 and 3 ranks, even and
uneven expert ranges, a rank that receives no rows.  Each rank's Y, dX and
routing-weight gradient must equal the single-process oracle layer on its
tokens, and its experts' LoRA gradients the oracle's sums over every rank's
tokens (the per-rank steps are the oracle's; what runs for real is the
exchange plan, the split sizes and the all-to-alls of the library's layer)."""
import json
import os
import socket
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from _ep_cases import CASES  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("case", sorted(CASES))
def test_expert_parallel_exchange_matches_the_oracle_layer(case, tmp_path):
    world = CASES[case]["world"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", EP_CASE=case, EP_TEST_OUT=str(tmp_path))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node=%d" % world, "--master-addr", "127.0.0.1", "--master-port",
           str(_free_port()), os.path.join(ROOT, "tests", "ep_worker.py")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    res = [json.loads((tmp_path / ("rank%d.json" % q)).read_text()) for q in range(world)]
    for q, e in enumerate(res):
        for n in ("Y", "dX", "dw", "dA_gu", "dB_gu", "dA_dn", "dB_dn"):
            assert e[n] < 1e-10, (case, q, n, e[n])
        # every row sent is received by its expert's rank
        assert sum(e["send"]) == CASES[case]["T"][q] * CASES[case]["k"]
    for q in range(world):
        assert [res[r]["send"][q] for r in range(world)] == res[q]["recv"]
    if CASES[case]["skew"]:
        assert sum(res[1]["recv"]) == 0     # rank 1's experts get no rows


def test_expert_ranges():
    from expert_routing_grouped_moe_gb300.ep import expert_ranges
    assert expert_ranges(8, 2) == [0, 4, 8]
    assert expert_ranges(7, 3) == [0, 2, 4, 7]
    assert expert_ranges(5, 5) == [0, 1, 2, 3, 4, 5]
    with pytest.raises(ValueError):
        expert_ranges(2, 3)
