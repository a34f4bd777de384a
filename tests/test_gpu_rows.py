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
    rt = oracle_route(ids_np, E, shared)
    K = ids_np.shape[1] + int(shared)
    return rt["sorted_src"] // K, rt["dest_pos"], ids_np.shape[0] * K


def oracle_route(ids_np, E, shared):
    T = ids_np.shape[0]
    if shared:
        ids_np = np.concatenate([ids_np, np.full((T, 1), E, dtype=ids_np.dtype)], 1)
    return oracle.route(ids_np, E + int(shared))


def assert_within_one_bf16_ulp(got, exact, abs_terms, nterms, name):
    """A sum of fp32 terms rounded once to bf16: |got - exact| is at most one
    bf16 ulp of the exact value, plus the fp32 rounding of the nterms
    products and additions (2^-24 relative to the absolute terms each)."""
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    mag = np.maximum(np.abs(exact), 2.0 ** -126)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    bound = ulp + (2 * nterms) * 2.0 ** -24 * np.asarray(abs_terms, dtype=np.float64)
    err = np.abs(got - exact)
    bad = err > bound
    assert not bad.any(), "%s: %d elements beyond one bf16 ulp (worst %.3g ulp)" % (
        name, int(bad.sum()), float(np.max(err / ulp)))


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
    rt = oracle_route(ids.cpu().numpy(), E, shared)
    got = Xp.view(torch.int16).cpu().numpy()
    Xb = X.view(torch.int16).cpu().numpy()
    # the oracle's permute on the bf16 bit patterns: a pure gather
    np.testing.assert_array_equal(got, oracle.permute(Xb, rt["sorted_src"], K))


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
    rt = oracle_route(ids.cpu().numpy(), E, shared)
    prow = rt["dest_pos"].reshape(T, K)
    R = to64(rows)
    wn = w.cpu().numpy() if weighted else None
    exp = oracle.combine(R, rt["dest_pos"], K, wn)
    abs_terms = oracle.combine(np.abs(R), rt["dest_pos"], K,
                               None if wn is None else np.abs(wn))
    assert_close_bf16(to64(out), exp, "combine")
    assert_within_one_bf16_ulp(to64(out), exp, abs_terms, K, "combine")
    np.testing.assert_array_equal(slot.cpu().numpy(), scal.cpu().numpy()[prow[:, :k]])


@pytest.mark.parametrize("T,E,k,dist",
                         [p for p in synth.ROUTE_SWEEP if p[0] == 1 << 18]
                         + [(1 << 20, 128, 8, "uniform"), (1 << 20, 8, 2, "zipf"),
                            (1 << 20, 64, 4, "zipf")])
def test_permute_combine_full_size_sampled(T, E, k, dist):
    """Every (E, k, distribution) point of the routing workload at T = 256K, and
    three at 1M: sampled tokens' combine and permuted rows against the oracle."""
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
    # sampled tokens: the oracle's permute and combine on the sample's own
    # slots (rows gathered from the oracle's routing of the whole batch)
    rng = np.random.default_rng(0)
    rt = oracle.route(ids.cpu().numpy(), E)
    toks = np.sort(rng.choice(T, size=1024, replace=False))
    Xs = to64(X[torch.from_numpy(toks).to(DEV)])
    # the sample's slots, in token order: their sorted positions and sources,
    # with the sample's tokens renumbered 0..n-1
    pos = rt["dest_pos"].reshape(T, k)[toks].reshape(-1)
    local_src = (np.repeat(np.arange(toks.size), k) * k + np.tile(np.arange(k), toks.size))
    rows_s = oracle.permute(Xs, local_src, k)
    ws = w.cpu().numpy()[toks]
    exp = oracle.combine(rows_s, np.arange(toks.size * k), k, ws)
    abs_terms = oracle.combine(np.abs(rows_s), np.arange(toks.size * k), k, np.abs(ws))
    got_y = to64(Y[torch.from_numpy(toks).to(DEV)])
    assert_close_bf16(got_y, exp, "roundtrip")
    assert_within_one_bf16_ulp(got_y, exp, abs_terms, k, "roundtrip")
    # the sample's permuted rows and further random ones are the oracle's
    # permute of X, bit for bit
    prows = np.concatenate([pos, rng.choice(T * k, size=4096, replace=False)])
    got = Xp[torch.from_numpy(prows).to(DEV)].view(torch.int16).cpu().numpy()
    src_rows = rt["sorted_src"][prows]
    Xb_rows = X.view(torch.int16)[torch.from_numpy(np.unique(src_rows // k)).to(DEV)]
    lookup = {t: i for i, t in enumerate(np.unique(src_rows // k))}
    Xb = Xb_rows.cpu().numpy()
    ref = oracle.permute(Xb, np.array([lookup[t] * k for t in src_rows // k]), k)
    np.testing.assert_array_equal(got, ref)
