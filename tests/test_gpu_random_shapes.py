"""Seeded random layer shapes on the GPU against the fp64 oracle.

d, f and r are drawn as any multiple of 8 in range, E, k and T at random, with
or without a shared expert, in the permuted or the gathered-row mode, and
sometimes with an expert id repeated inside a token; the shapes in the
permuted-row mode also compute the full weight gradients.  Tiles, K slices, TMA
boxes, grid-mode passes and epilogue masks thus meet shapes that no
hand-written case picked.  Every element of Y, dX, dw and the four LoRA
gradients is compared."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import MoELoRALayer, _lib as L, synth
from _util import assert_close_bf16, oracle_params, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 41))
        r = 8 * int(rng.integers(1, 9))
        out.append(dict(
            name="rand%d" % i, d=8 * int(rng.integers(4, 48)), f=8 * int(rng.integers(2, 40)),
            r=r, E=E, k=int(rng.integers(1, min(E, 8) + 1)), T=int(rng.integers(1, 700)),
            shared=bool(rng.integers(0, 2)), gather=bool(rng.integers(0, 2)),
            dup_ids=bool(rng.integers(0, 3) == 0)))
    return out


SHAPES = _shapes(16, seed=2024)


@pytest.mark.parametrize("sh", SHAPES, ids=[s["name"] for s in SHAPES])
def test_random_shape_matches_oracle(sh):
    cfg = synth.LayerConfig(sh["name"], T=sh["T"], d=sh["d"], f=sh["f"], E=sh["E"], k=sh["k"],
                            r=sh["r"], alpha=2.0 * sh["r"], shared=sh["shared"])
    seed = 31 + int(sh["name"][4:])
    wts = synth.layer_weights(cfg, seed, device=DEV)
    act = synth.layer_activations(cfg, seed, device=DEV)
    if sh["dup_ids"]:
        rng = np.random.default_rng(seed)
        ids_np = rng.integers(0, cfg.E, size=(cfg.T, cfg.k)).astype(np.int32)
        w_np = synth.combine_weights(cfg.T, cfg.k, seed=seed).numpy()
    else:
        ids_np, w_np = oracle.router_topk(act["logits"].cpu().numpy(), cfg.k)
    full = not sh["gather"]  # the full weight gradients need the permuted rows
    layer = MoELoRALayer(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.r, cfg.alpha, wts,
                         shared_expert=cfg.shared, device=DEV, gather=sh["gather"],
                         full_grads=full)
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
    w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(DEV)
    Y = layer.forward(act["X"], ids, w).clone()
    g = {n: v.clone() for n, v in layer.backward(act["dY"]).items()}
    assert L.moe_status() == L.MOE_OK
    P = oracle_params(wts, cfg)
    X, dY = to64(act["X"]), to64(act["dY"])
    tag = sh["name"]
    assert_close_bf16(to64(Y), oracle.layer_forward(X, ids_np, w_np, P), tag + " Y")
    ref = oracle.layer_backward(X, ids_np, w_np, dY, P, full=full)
    assert_close_bf16(to64(g["dX"]), ref["dX"], tag + " dX")
    assert_close_bf16(g["dw"].cpu().numpy(), ref["dw"], tag + " dw")
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn") + (("dW_gu", "dW_dn") if full else ()):
        assert_close_bf16(g[n].cpu().numpy(), ref[n], tag + " " + n)
