"""One rank of the gloo test of the expert-parallel exchange (launched by
tests/test_ep_dist_cpu.py through torch.distributed.run).  The per-rank steps
are the oracle's (tests/_ep_cases.py); the exchange plan, the split sizes and
the all-to-alls are the library's expert-parallel layer over gloo.  Writes
the largest differences from the single-process oracle layer."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import oracle  # noqa: E402
from _ep_cases import CASES, OracleOps, full_params, local_params, rank_inputs  # noqa: E402
from expert_routing_grouped_moe_gb300.ep import (ExpertParallelLayer, TorchComm,  # noqa: E402
                                                 expert_ranges)


def main():
    case = os.environ["EP_CASE"]
    c = CASES[case]
    dist.init_process_group("gloo")
    comm = TorchComm()
    rank, world = comm.rank, comm.world
    assert world == c["world"]
    P = full_params(case)
    b = expert_ranges(c["E"], world)
    layer = ExpertParallelLayer(c["E"], c["k"], comm, OracleOps(local_params(P, b[rank],
                                                                             b[rank + 1])))
    X, ids, w, dY = rank_inputs(case, rank)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
    Y = layer.forward(t(X), t(ids), t(w)).numpy()
    g = layer.backward(t(dY))
    # the single-process oracle: this rank's tokens through all experts, and
    # the LoRA gradients of this rank's experts summed over every rank's tokens
    err = {"Y": float(np.max(np.abs(Y - oracle.layer_forward(X, ids, w, P))))}
    ref = oracle.layer_backward(X, ids, w, dY, P)
    err["dX"] = float(np.max(np.abs(g["dX"].numpy() - ref["dX"])))
    err["dw"] = float(np.max(np.abs(g["dw"].numpy() - ref["dw"])))
    allin = [rank_inputs(case, q) for q in range(world)]
    cat = lambda i: np.concatenate([a[i] for a in allin])  # noqa: E731
    ref_all = oracle.layer_backward(cat(0), cat(1), cat(2), cat(3), P)
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        err[n] = float(np.max(np.abs(g[n].numpy() - ref_all[n][b[rank]:b[rank + 1]])))
    err["E_loc"] = layer.E_loc
    err["send"], err["recv"] = layer._fw["send"], layer._fw["recv"]
    dist.destroy_process_group()
    with open(os.path.join(os.environ["EP_TEST_OUT"], "rank%d.json" % rank), "w") as fh:
        json.dump(err, fh)


if __name__ == "__main__":
    main()
