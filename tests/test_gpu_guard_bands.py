"""Out-of-bounds writes, without a sanitizer: every output and workspace of a
full layer step sits between two 4 KB guard bands filled with a canary
byte, and every band must still hold it afterwards.  The step runs through
the C ABI (route, both permutes, forward, combine, backward with the full
weight gradients, combine of dX and dw) on ragged shapes, with the large
GEMMs on single CTAs and on CTA pairs, and in the gathered-row mode; the
results are also checked against the oracle so the buffers hold real work."""
import math

import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import _lib as L, synth
from _util import assert_close_bf16, oracle_params, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


class Guarded:
    """Device buffers with canary bands on both sides."""

    def __init__(self):
        self.bufs = []

    def __call__(self, name, shape, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        n = math.prod(shape)
        raw = torch.full((2 * GUARD + n * esz,), CANARY, dtype=torch.uint8, device=DEV)
        view = raw[GUARD:GUARD + n * esz].view(dtype).view(*shape)
        self.bufs.append((name, raw, n * esz))
        return view

    def check(self):
        torch.cuda.synchronize()
        for name, raw, nbytes in self.bufs:
            lo = raw[:GUARD]
            hi = raw[GUARD + nbytes:]
            assert bool(torch.all(lo == CANARY)), "%s: write before the buffer" % name
            assert bool(torch.all(hi == CANARY)), "%s: write past the end of the buffer" % name


def run_step(cfg, wts, act, ids_np, w_np, gather, full):
    g = Guarded()
    T, d, f, E, k, r = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.r
    K, G = cfg.slots, cfg.groups
    N = T * K
    i32, bf, f32 = torch.int32, torch.bfloat16, torch.float32
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
    w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(DEV)
    t = {n: g(n, (s,), i32) for n, s in (("counts", G), ("offsets", G + 1), ("tile_off", G + 1),
                                         ("sorted_src", N), ("dest_pos", N))}
    rws = g("route_ws", (max(16, L.moe_route_workspace_size(T, K, G)),), torch.uint8)
    L.moe_route(ids, E, cfg.shared, t["counts"], t["offsets"], t["tile_off"], t["sorted_src"],
                t["dest_pos"], rws)
    Xp = dYp = None
    if not gather:
        Xp = g("Xp", (N, d), bf)
        L.moe_permute(act["X"], K, t["dest_pos"], Xp)
    dims = L.make_dims(T, d, f, E, k, r, cfg.scale, cfg.shared)
    Yp = g("Yp", (N, d), bf)
    h = g("h", (N, 32 * ((f + 15) // 16)), f32)
    a = g("act", (2, N, f), bf)
    xa = g("xa_gu", (2, N, r), bf)
    xd = g("xa_dn", (2, N, r), bf)
    W = {n: wts[n] for n in ("W_gu", "A_gu", "B_gu", "W_dn", "A_dn", "B_dn")}
    L.moe_lora_grouped_mlp_fwd(dims, Xp, act["X"] if gather else None, t["counts"], t["offsets"],
                               t["tile_off"], t["sorted_src"], w, W["W_gu"], W["A_gu"],
                               W["B_gu"], W["W_dn"], W["A_dn"], W["B_dn"], Yp, h, a, xa, xd)
    Y = g("Y", (T, d), bf)
    L.moe_unpermute_combine(Yp, t["dest_pos"], k, cfg.shared, Y)
    if not gather:
        dYp = g("dYp", (N, d), bf)
        L.moe_permute(act["dY"], K, t["dest_pos"], dYp)
    dXp = g("dXp", (N, d), bf)
    dw_rows = g("dw_rows", (N,), f32)
    gr = {"dA_gu": g("dA_gu", (G, r, d), f32), "dB_gu": g("dB_gu", (G, 2 * f, r), f32),
          "dA_dn": g("dA_dn", (G, r, f), f32), "dB_dn": g("dB_dn", (G, d, r), f32)}
    dWgu = g("dW_gu", (G, 2 * f, d), f32) if full else None
    dWdn = g("dW_dn", (G, d, f), f32) if full else None
    bws = g("bwd_ws", (L.moe_mlp_bwd_workspace_size(dims),), torch.uint8)
    L.moe_lora_grouped_mlp_bwd(dims, dYp, act["dY"] if gather else None, Xp,
                               act["X"] if gather else None, t["counts"], t["offsets"],
                               t["tile_off"], t["sorted_src"], w, W["W_gu"], W["A_gu"],
                               W["B_gu"], W["W_dn"], W["A_dn"], W["B_dn"], h, a, xa, xd, dXp,
                               dw_rows, gr["dA_gu"], gr["dB_gu"], gr["dA_dn"], gr["dB_dn"], bws,
                               dW_gu=dWgu, dW_dn=dWdn)
    dX = g("dX", (T, d), bf)
    dw = g("dw", (T, k), f32)
    L.moe_unpermute_combine(dXp, t["dest_pos"], k, cfg.shared, dX, row_scalars=dw_rows,
                            slot_out=dw)
    assert L.moe_status() == L.MOE_OK
    g.check()
    return Y, dX, dw, gr


CASES = {
    # ragged d, f, r = 16 (single-CTA large GEMMs except gate_up)
    "ragged": synth.LayerConfig("ragged", T=1000, d=320, f=200, E=6, k=3, r=16, alpha=32),
    # >= 512 rows per group: every large GEMM on CTA pairs, ragged f
    "pairs": synth.LayerConfig("pairs", T=1100, d=256, f=136, E=4, k=2, r=24, alpha=48),
    # a shared expert and rank 8
    "shared": synth.LayerConfig("shared", T=300, d=192, f=72, E=8, k=2, r=8, alpha=16,
                                shared=True),
    # a shared expert of 2500 rows: its LoRA weight gradients are summed in
    # three parts of 1024 rows, through the workspace's partial sums
    "split": synth.LayerConfig("split", T=2500, d=128, f=64, E=7, k=1, r=8, alpha=16,
                               shared=True),
}


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_no_write_outside_any_buffer(name, gather):
    cfg = CASES[name]
    wts = synth.layer_weights(cfg, seed=3, device=DEV)
    act = synth.layer_activations(cfg, seed=3, device=DEV)
    ids_np, w_np = oracle.router_topk(act["logits"].cpu().numpy(), cfg.k)
    full = not gather
    Y, dX, dw, gr = run_step(cfg, wts, act, ids_np, w_np, gather, full)
    P = oracle_params(wts, cfg)
    X, dY = to64(act["X"]), to64(act["dY"])
    assert_close_bf16(to64(Y), oracle.layer_forward(X, ids_np, w_np, P), name + " Y")
    ref = oracle.layer_backward(X, ids_np, w_np, dY, P)
    assert_close_bf16(to64(dX), ref["dX"], name + " dX")
    assert_close_bf16(dw.cpu().numpy(), ref["dw"], name + " dw")
    for n in gr:
        assert_close_bf16(gr[n].cpu().numpy(), ref[n], name + " " + n)
