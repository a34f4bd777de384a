"""GPU parity of the router and the grouped routing pass: bit-exact against the
oracle (the routing result is unique: stable order inside each expert)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import _lib as L, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def gpu_route(ids, E, shared=False):
    T, k = ids.shape
    K, G = k + int(shared), E + int(shared)
    N = T * K
    out = {"counts": torch.full((G,), -7, dtype=torch.int32, device=DEV),
           "offsets": torch.full((G + 1,), -7, dtype=torch.int32, device=DEV),
           "tile_off": torch.full((G + 1,), -7, dtype=torch.int32, device=DEV),
           "sorted_src": torch.full((N,), -7, dtype=torch.int32, device=DEV),
           "dest_pos": torch.full((N,), -7, dtype=torch.int32, device=DEV)}
    ws = torch.empty(L.moe_route_workspace_size(T, K, G), dtype=torch.uint8, device=DEV)
    L.moe_route(ids, E, shared, out["counts"], out["offsets"], out["tile_off"],
                out["sorted_src"], out["dest_pos"], ws)
    status = L.moe_status()
    return {k2: v.cpu().numpy().astype(np.int64) for k2, v in out.items()}, status


def check_route(ids_t, E, shared=False):
    got, status = gpu_route(ids_t, E, shared)
    assert status == L.MOE_OK
    ids = ids_t.cpu().numpy()
    if shared:
        ids = np.concatenate([ids, np.full((ids.shape[0], 1), E, dtype=ids.dtype)], 1)
    ref = oracle.route(ids, E + int(shared))
    for key in ("counts", "offsets", "sorted_src", "dest_pos"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    tiles = (ref["counts"] + 127) // 128
    np.testing.assert_array_equal(got["tile_off"], np.concatenate([[0], np.cumsum(tiles)]))


@pytest.mark.parametrize("name", ["tiny", "qwen3_30b_a3b", "gpt_oss_20b", "skewed_shared"])
def test_router_topk_matches_oracle(name):
    cfg = synth.CONFIGS[name]
    logits = synth.layer_activations(synth.scaled(cfg, T=min(cfg.T, 4096)), seed=3,
                                     device="cpu")["logits"]
    T = logits.shape[0]
    ids = torch.empty(T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, cfg.k, dtype=torch.float32, device=DEV)
    L.moe_router_topk(logits.to(DEV), cfg.k, ids, w)
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.router_topk(logits.numpy(), cfg.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_router_ties_lower_id_first():
    logits = torch.tensor([[1.0, 3.0, 3.0, 3.0, -np.inf, 0.5] * 6], dtype=torch.float32)
    ids = torch.empty(1, 5, dtype=torch.int32, device=DEV)
    w = torch.empty(1, 5, dtype=torch.float32, device=DEV)
    L.moe_router_topk(logits.to(DEV), 5, ids, w)
    ref_ids, ref_w = oracle.router_topk(logits.numpy(), 5)
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6)


@pytest.mark.parametrize("name", ["tiny", "qwen3_30b_a3b", "gpt_oss_20b", "skewed_shared"])
def test_route_layer_configs(name):
    cfg = synth.CONFIGS[name]
    logits = synth.layer_activations(cfg, seed=5, device="cpu")["logits"]
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV)
    L.moe_router_topk(logits.to(DEV), cfg.k, ids, w)
    check_route(ids, cfg.E, cfg.shared)


@pytest.mark.parametrize("T,E,k,dist", synth.ROUTE_SWEEP)
def test_route_sweep(T, E, k, dist):
    """Every point of the routing workload (T in 1K..1M, E in 8..128, top-2/4/8,
    uniform and Zipf ids), bit-exact against the oracle."""
    ids = synth.topk_ids(T, E, k, dist, seed=11, device=DEV)
    check_route(ids, E)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (1, 8, 8), (3, 2, 2), (1000, 4, 4), (4097, 3, 1000)])
def test_route_duplicate_ids_and_edges(T, k, E):
    g = torch.Generator().manual_seed(T * 7 + k)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    check_route(ids.to(DEV), E)
    check_route(ids.to(DEV), E, shared=True)


def test_route_all_to_one_expert():
    ids = torch.zeros(5000, 1, dtype=torch.int32, device=DEV)
    check_route(ids, 16)


def test_route_bad_ids_reported():
    E = 6
    g = torch.Generator().manual_seed(1)
    ids = torch.randint(0, E, (300, 3), generator=g, dtype=torch.int32)
    ids[5, 1] = -1
    ids[77, 0] = E
    ids[299, 2] = 1 << 20
    got, status = gpu_route(ids.to(DEV), E)
    assert status == L.MOE_ERR_BAD_IDS
    assert L.moe_status() == L.MOE_OK  # cleared by the read
    a = ids.numpy()
    loop = oracle.route_where_loop(a, E)   # bad ids match no expert
    valid = np.concatenate(loop)
    np.testing.assert_array_equal(got["counts"], [len(x) for x in loop])
    np.testing.assert_array_equal(got["sorted_src"][:valid.size], valid)
    assert np.all(got["sorted_src"][valid.size:] == -1)
    flat = a.reshape(-1)
    bad = (flat < 0) | (flat >= E)
    assert np.all(got["dest_pos"][bad] == -1)
    np.testing.assert_array_equal(got["sorted_src"][got["dest_pos"][~bad]],
                                  np.nonzero(~bad)[0])


@pytest.mark.parametrize("name", ["tiny", "qwen3_30b_a3b", "skewed_shared"])
def test_route_logits_equals_router_then_route(name):
    """The one-call router + routing gives the two calls' results bit for bit,
    and they are the oracle's."""
    cfg = synth.CONFIGS[name]
    logits = synth.layer_activations(cfg, seed=8, device="cpu")["logits"].to(DEV)
    T, k, E, shared = cfg.T, cfg.k, cfg.E, cfg.shared
    K, G = k + int(shared), E + int(shared)
    mk = lambda n: torch.full((n,), -7, dtype=torch.int32, device=DEV)  # noqa: E731
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    t = {n: mk(c) for n, c in (("counts", G), ("offsets", G + 1), ("tile_off", G + 1),
                               ("sorted_src", T * K), ("dest_pos", T * K))}
    ws = torch.empty(L.moe_route_workspace_size(T, K, G), dtype=torch.uint8, device=DEV)
    L.moe_route_logits(logits, k, shared, ids, w, t["counts"], t["offsets"], t["tile_off"],
                       t["sorted_src"], t["dest_pos"], ws)
    assert L.moe_status() == L.MOE_OK
    ref, _ = gpu_route(ids.clone(), E, shared)
    for key in ref:
        np.testing.assert_array_equal(t[key].cpu().numpy(), ref[key], err_msg=key)
    ids_ref, w_ref = oracle.router_topk(logits.cpu().numpy(), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    check_route(ids, E, shared)
