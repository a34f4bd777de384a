"""Pins for the oracle's routing and router (CPU only).

The routing pass of the Unsloth x NVIDIA article (section 'Optimisation 3')
replaces a per-expert where-loop; its result must be the loop's result.  The
oracle is pinned to that brute force, to hand-worked examples and to the
counting invariants.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


@pytest.mark.parametrize("case", _load("route_small.json")["cases"])
def test_route_golden(case):
    rt = oracle.route(np.array(case["ids"]), case["E"])
    for key in ("counts", "offsets", "sorted_src", "dest_pos"):
        assert rt[key].tolist() == case[key], key


def _random_ids(rng, T, k, E, distinct):
    if distinct:
        return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    return rng.integers(0, E, size=(T, k)).astype(np.int32)


@pytest.mark.parametrize("T,k,E,distinct", [
    (1, 1, 1, True), (1, 4, 4, True), (7, 2, 8, True), (64, 8, 128, True),
    (33, 3, 5, False), (100, 4, 3, False), (257, 2, 16, True), (5, 6, 2, False)])
def test_route_matches_where_loop(T, k, E, distinct):
    rng = np.random.default_rng(T * 1000 + k * 10 + E)
    ids = _random_ids(rng, T, k, E, distinct)
    rt = oracle.route(ids, E)
    loop = oracle.route_where_loop(ids, E)
    for e in range(E):
        seg = rt["sorted_src"][rt["offsets"][e]:rt["offsets"][e + 1]]
        assert seg.tolist() == loop[e].tolist()
        assert rt["counts"][e] == len(loop[e])


@pytest.mark.parametrize("seed", range(6))
def test_route_invariants(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 300))
    ids = _random_ids(rng, T, k, E, distinct=bool(seed % 2))
    rt = oracle.route(ids, E)
    N = T * k
    assert rt["counts"].sum() == N
    assert rt["offsets"][0] == 0 and rt["offsets"][-1] == N
    assert np.all(np.diff(rt["offsets"]) == rt["counts"])
    # permutation, inverse, grouping and stability
    assert sorted(rt["sorted_src"].tolist()) == list(range(N))
    assert np.all(rt["sorted_src"][rt["dest_pos"]] == np.arange(N))
    flat = ids.reshape(-1)
    keys = flat[rt["sorted_src"]]
    assert np.all(np.diff(keys) >= 0)
    same = np.diff(keys) == 0
    assert np.all(np.diff(rt["sorted_src"])[same] > 0)


def test_route_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 3]]), 3)


def _golden_logit(v):
    if v == "ln3":
        return np.float32(math.log(3.0))
    if v == "-inf":
        return np.float32(-np.inf)
    return np.float32(v)


@pytest.mark.parametrize("case", _load("router_small.json")["cases"])
def test_router_golden(case):
    logits = np.array([[_golden_logit(v) for v in row] for row in case["logits"]], dtype=np.float32)
    ids, w = oracle.router_topk(logits, case["k"])
    assert ids.tolist() == case["ids"]
    if "w" in case:
        np.testing.assert_allclose(w, np.array(case["w"]), rtol=1e-6, atol=1e-7)
    else:
        e3, em2 = math.exp(3.0), math.exp(-2.0)
        ref = np.array([[e3, e3, em2]]) / (2 * e3 + em2)
        np.testing.assert_allclose(w, ref, rtol=1e-6)


@pytest.mark.parametrize("seed", range(4))
def test_router_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T, E, k = 20, 9, 3
    # coarse values force ties
    logits = rng.integers(-3, 3, size=(T, E)).astype(np.float32)
    ids, w = oracle.router_topk(logits, k)
    for t in range(T):
        pairs = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        assert ids[t].tolist() == pairs[:k]
        p = np.exp(logits[t].astype(np.float64))
        p /= p.sum()
        ref = p[pairs[:k]] / p[pairs[:k]].sum()
        np.testing.assert_allclose(w[t], ref, rtol=1e-6)
        assert abs(float(w[t].sum()) - 1.0) < 1e-6
