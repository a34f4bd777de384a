"""GPU parity of the row permute (bit-exact gather into expert-grouped sorted
layout) and the combine (weighted gather-reduce, bf16 tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import _lib as L, synth
from _util import assert_close_bf16, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def routed(ids, E, shared=False):
    T, k = ids.shape
    K, G = k + int(shared), E + int(shared)
    r = {"counts": torch.empty(G, dtype=torch.int32, device=DEV),
         "offsets": torch.empty(G + 1, dtype=torch.int32, device=DEV),
         "tile_off": torch.empty(G + 1, dtype=torch.int32, device=DEV),
         "sorted_src": torch.empty(T * K, dtype=torch.int32, device=DEV),
         "dest_pos": torch.empty(T * K, dtype=torch.int32, device=DEV)}
    ws = torch.empty(L.moe_route_workspace_size(T, K, G), dtype=torch.uint8, device=DEV)
    L.moe_route(ids, E, shared, r["counts"], r["offsets"], r["tile_off"], r["sorted_src"],
                r["dest_pos"], ws)
    return r, K, G


def expected_layout(ids_np, E, shared):
    """Host-side, from the oracle's routing: the source token of every
    permuted row (row p = sorted position p) and the permuted row of every
    flat index (its sorted position)."""
    T = ids_np.shape[0]
    if shared:
        ids_np = np.concatenate([ids_np, np.full((T, 1), E, dtype=ids_np.dtype)], 1)
    K = ids_np.shape[1]
    rt = oracle.route(ids_np, E + int(shared))
    return rt["sorted_src"] // K, rt["dest_pos"], T * K


@pytest.mark.parametrize("T,E,k,dist,shared,d", [
    (256, 8, 2, "uniform", False, 128), (300, 5, 3, "zipf", True, 64),
    (1 << 14, 128, 8, "uniform", False, 2048), (1 << 14, 32, 4, "zipf", False, 2048),
    (4096, 64, 4, "zipf", True, 2048)])
def test_permute_bit_exact(T, E, k, dist, shared, d):
    ids = synth.topk_ids(T, E, k, dist, seed=2, device=DEV)
    X = synth.hidden_rows(T, d, seed=2, device=DEV)
    r, K, G = routed(ids, E, shared)
    Xp = torch.full((T * K, d), 7.0, dtype=torch.bfloat16, device=DEV)
    L.moe_permute(X, K, r["dest_pos"], Xp)
    torch.cuda.synchronize()
    src_tok, _, N = expected_layout(ids.cpu().numpy(), E, shared)
    got = Xp.view(torch.int16).cpu().numpy()
    Xb = X.view(torch.int16).cpu().numpy()
    np.testing.assert_array_equal(got, Xb[src_tok])


@pytest.mark.parametrize("T,E,k,dist,shared,d,weighted", [
    (256, 8, 2, "uniform", False, 128, True), (300, 5, 3, "zipf", True, 64, True),
    (1 << 14, 128, 8, "uniform", False, 2048, True), (4096, 64, 4, "zipf", True, 2048, False)])
def test_combine(T, E, k, dist, shared, d, weighted):
    ids = synth.topk_ids(T, E, k, dist, seed=4, device=DEV)
    r, K, G = routed(ids, E, shared)
    N = T * K
    rows = synth.hidden_rows(N, d, seed=5, device=DEV)
    w = synth.combine_weights(T, k, seed=6, device=DEV) if weighted else None
    scal = torch.randn(N, generator=torch.Generator(DEV).manual_seed(3), device=DEV)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    slot = torch.empty(T, k, dtype=torch.float32, device=DEV)
    L.moe_unpermute_combine(rows, r["dest_pos"], k, shared, out, weights=w, row_scalars=scal,
                            slot_out=slot)
    torch.cuda.synchronize()
    _, prow, _ = expected_layout(ids.cpu().numpy(), E, shared)
    prow = prow.reshape(T, K)
    R = to64(rows)
    c = np.ones((T, K))
    if weighted:
        c[:, :k] = w.cpu().numpy()
    exp = np.einsum("tj,tjd->td", c, R[prow])
    assert_close_bf16(to64(out), exp, "combine")
    np.testing.assert_array_equal(slot.cpu().numpy(), scal.cpu().numpy()[prow[:, :k]])


@pytest.mark.parametrize("T,E,k,dist", [(1 << 18, 128, 8, "zipf"), (1 << 20, 128, 8, "uniform"),
                                         (1 << 20, 8, 2, "zipf")])
def test_permute_combine_full_size_sampled(T, E, k, dist):
    d = 2048
    ids = synth.topk_ids(T, E, k, dist, seed=8, device=DEV)
    X = synth.hidden_rows(T, d, seed=8, device=DEV)
    w = synth.combine_weights(T, k, seed=8, device=DEV)
    r, K, G = routed(ids, E)
    Xp = torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV)
    L.moe_permute(X, K, r["dest_pos"], Xp)
    Y = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    L.moe_unpermute_combine(Xp, r["dest_pos"], k, False, Y, weights=w)
    torch.cuda.synchronize()
    # properties that hold at any size: the round trip gives sum_j w_j * X[t]
    rng = np.random.default_rng(0)
    toks = rng.choice(T, size=64, replace=False)
    Xs = to64(X[torch.from_numpy(toks).to(DEV)])
    ws = w.cpu().numpy()[toks].astype(np.float64).sum(1, keepdims=True)
    assert_close_bf16(to64(Y[torch.from_numpy(toks).to(DEV)]), ws * Xs, "roundtrip")
    # and each sampled permuted row is the right token row, bit for bit
    src_tok, _, N = expected_layout(ids.cpu().numpy(), E, False)
    prows = rng.choice(N, size=256, replace=False)
    got = Xp[torch.from_numpy(prows).to(DEV)].view(torch.int16).cpu().numpy()
    ref = X.view(torch.int16)[torch.from_numpy(src_tok[prows]).to(DEV)].cpu().numpy()
    np.testing.assert_array_equal(got, ref)
