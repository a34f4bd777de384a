"""Pins for the oracle's row permute and combine (CPU only).

permute is step 5 of the Unsloth x NVIDIA article's grouped routing
(section 'Optimisation 3'): the token rows sliced into expert order; combine
is its weighted inverse, the top-k mixture.  Pinned by a hand-worked example,
by the round trip through the routing, and by the layer: combining the
per-row expert outputs must give ``layer_forward``, which has its own pins.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold():
    with open(os.path.join(GOLD, "combine_small.json")) as fh:
        return json.load(fh)


def test_permute_combine_golden():
    g = _gold()
    rt = oracle.route(np.array(g["ids"]), g["E"])
    assert rt["sorted_src"].tolist() == g["sorted_src"]
    assert rt["dest_pos"].tolist() == g["dest_pos"]
    Xp = oracle.permute(np.array(g["X"]), rt["sorted_src"], g["K"])
    assert Xp.tolist() == g["Xp"]
    Y = oracle.combine(np.array(g["rows"]), rt["dest_pos"], g["K"], np.array(g["w"]))
    assert Y.tolist() == g["Y"]
    Yu = oracle.combine(np.array(g["rows"]), rt["dest_pos"], g["K"])
    assert Yu.tolist() == g["Y_unweighted"]


def test_combine_shared_slot_has_weight_one():
    # K = 3 slots, weights for the first 2: the third (shared) slot counts 1
    rows = np.arange(12, dtype=np.float64).reshape(6, 2)
    dest = np.array([5, 4, 3, 2, 1, 0])
    w = np.array([[0.5, 0.25], [0.0, 1.0]])
    Y = oracle.combine(rows, dest, 3, w)
    assert Y[0].tolist() == (0.5 * rows[5] + 0.25 * rows[4] + rows[3]).tolist()
    assert Y[1].tolist() == (rows[1] + rows[0]).tolist()


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (37, 3, 5, 1), (200, 8, 16, 2)])
def test_round_trip_returns_weighted_rows(T, k, E, seed):
    """combine(permute(X)) = (sum_j w[t,j]) X[t] for any routing, duplicate
    ids included: every slot's row is its token's row."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k))
    X = rng.standard_normal((T, 6))
    w = rng.random((T, k))
    rt = oracle.route(ids, E)
    Y = oracle.combine(oracle.permute(X, rt["sorted_src"], k), rt["dest_pos"], k, w)
    np.testing.assert_allclose(Y, w.sum(1, keepdims=True) * X, rtol=1e-14, atol=1e-14)


def test_permute_is_the_where_loop_slices():
    """Expert e's slice of the permuted rows holds, in order, the rows of the
    tokens the old per-expert loop finds for e."""
    rng = np.random.default_rng(7)
    T, k, E = 50, 4, 9
    ids = rng.integers(0, E, size=(T, k))
    X = rng.standard_normal((T, 3))
    rt = oracle.route(ids, E)
    Xp = oracle.permute(X, rt["sorted_src"], k)
    loop = oracle.route_where_loop(ids, E)
    for e in range(E):
        seg = Xp[rt["offsets"][e]:rt["offsets"][e + 1]]
        np.testing.assert_array_equal(seg, X[loop[e] // k])


def test_combine_of_expert_outputs_is_the_layer():
    """Combining each permuted row's expert output w * o (computed row group
    by row group) reproduces layer_forward, shared expert included."""
    rng = np.random.default_rng(11)
    T, d, f, E, k, r = 40, 8, 6, 5, 2, 3
    G = E + 1
    P = oracle.OracleParams(
        W_gu=rng.standard_normal((G, 2 * f, d)) / np.sqrt(d),
        A_gu=rng.standard_normal((G, r, d)) / np.sqrt(d),
        B_gu=rng.standard_normal((G, 2 * f, r)) * 0.1,
        W_dn=rng.standard_normal((G, d, f)) / np.sqrt(f),
        A_dn=rng.standard_normal((G, r, f)) / np.sqrt(f),
        B_dn=rng.standard_normal((G, d, r)) * 0.1, s=2.0, E=E, shared=True)
    X = rng.standard_normal((T, d))
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k))
    ids_sh = np.concatenate([ids, np.full((T, 1), E)], 1)
    K = k + 1
    rt = oracle.route(ids_sh, G)
    Xp = oracle.permute(X, rt["sorted_src"], K)
    out = np.zeros_like(Xp)
    for g in range(G):
        a, b = rt["offsets"][g], rt["offsets"][g + 1]
        if b > a:
            out[a:b] = oracle.expert_forward(Xp[a:b], P, g)["o"]
    Y = oracle.combine(out, rt["dest_pos"], K, w)
    np.testing.assert_allclose(Y, oracle.layer_forward(X, ids, w, P), rtol=1e-12, atol=1e-12)


def test_permute_rejects_out_of_range_positions():
    with pytest.raises(ValueError):
        oracle.permute(np.zeros((2, 2)), np.array([0, 4]), 2)
