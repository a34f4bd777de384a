"""Failure detection on the GPU without a fault: a pipeline wait that never
completes gives up after its limit, the device status word reports
MOE_ERR_TIMEOUT, and the context stays usable for the next layer step."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import MoELoRALayer, _lib as L, synth
from _util import assert_close_bf16, oracle_params, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def test_bounded_wait_times_out_and_context_survives():
    assert L.moe_status() == L.MOE_OK
    L.moe_selftest_wait_timeout(20000)  # 20 ms on a barrier nothing arrives on
    assert L.moe_status() == L.MOE_ERR_TIMEOUT
    assert L.moe_status() == L.MOE_OK  # reading the word cleared it
    # the context still runs the layer correctly
    cfg = synth.CONFIGS["tiny"]
    wts = synth.layer_weights(cfg, 3, device="cuda")
    act = synth.layer_activations(cfg, 3, device="cuda")
    ids_np, w_np = oracle.router_topk(act["logits"].cpu().numpy(), cfg.k)
    layer = MoELoRALayer(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.r, cfg.alpha, wts,
                         shared_expert=cfg.shared, device="cuda")
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).cuda()
    Y = layer.forward(act["X"], ids, w)
    assert L.moe_status() == L.MOE_OK
    P = oracle_params(wts, cfg)
    assert_close_bf16(to64(Y), oracle.layer_forward(to64(act["X"]), ids_np, w_np, P), "Y")


def test_read_stream_probe_runs_and_reports_ok():
    """The read-stream probe (a measurement kernel) streams a buffer whose
    size is not a multiple of its 32 KB stage, and a buffer as GEMM-operand
    tiles, and leaves the status clean."""
    buf = torch.empty((64 << 20) + 48, dtype=torch.uint8, device="cuda")
    L.moe_probe_read_stream(buf, L.MOE_PROBE_LINEAR)
    tiles = torch.empty(300 * (128 * 4096), dtype=torch.uint8, device="cuda")
    L.moe_probe_read_stream(tiles, L.MOE_PROBE_TILES)
    torch.cuda.synchronize()
    assert L.moe_status() == L.MOE_OK
