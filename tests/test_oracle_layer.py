"""Pins for the oracle's split-LoRA SwiGLU expert layer (CPU only).

* hand-worked 1x1 example (gate/up order, SiLU, LoRA scale, combine weights)
* split LoRA == merged W + s B A (the associativity statement of the Unsloth
  'Faster MoE' docs, section 'Faster LoRA MoE training')
* central finite differences for every gradient
* reductions: B = 0 gives the base MoE, the shared expert equals an extra
  routed slot of weight 1, linearity in the routing weights
* the sampled (per-token / per-expert) evaluators agree with the full layer
"""
import copy
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_params(rng, G, d, f, r, s, E, shared, bscale=0.3):
    P = {
        "W_gu": rng.standard_normal((G, 2 * f, d)) / np.sqrt(d),
        "A_gu": rng.standard_normal((G, r, d)) / np.sqrt(d),
        "B_gu": rng.standard_normal((G, 2 * f, r)) * bscale,
        "W_dn": rng.standard_normal((G, d, f)) / np.sqrt(f),
        "A_dn": rng.standard_normal((G, r, f)) / np.sqrt(f),
        "B_dn": rng.standard_normal((G, d, r)) * bscale,
    }
    return oracle.OracleParams.from_arrays(P, s=s, E=E, shared=shared)


def _problem(seed, T=9, d=12, f=6, E=4, k=2, r=3, s=2.0, shared=False, dup=False):
    rng = np.random.default_rng(seed)
    G = E + (1 if shared else 0)
    P = _rand_params(rng, G, d, f, r, s, E, shared)
    X = rng.standard_normal((T, d))
    if dup:
        ids = rng.integers(0, E, size=(T, k))
    else:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k))
    w /= w.sum(1, keepdims=True)
    dY = rng.standard_normal((T, d))
    return P, X, ids.astype(np.int32), w, dY


def test_swiglu_golden():
    g = json.load(open(os.path.join(GOLD, "swiglu_1x1.json")))
    arr = {n: np.array([e[n] for e in g["experts"]], dtype=np.float64)
           for n in ("W_gu", "A_gu", "B_gu", "W_dn", "A_dn", "B_dn")}
    P = oracle.OracleParams.from_arrays(arr, s=g["s"], E=2)
    X = np.array([[g["x"]]])
    for e, ex in enumerate(g["experts"]):
        o = oracle.expert_forward(X, P, e)["o"][0, 0]
        assert o == pytest.approx(ex["o"], rel=1e-14)
    Y = oracle.layer_forward(X, np.array(g["ids"]), np.array(g["w"]), P)
    assert Y[0, 0] == pytest.approx(g["y"], rel=1e-14)
    # dw = dY . o for each slot (gradient of a linear function of w)
    gr = oracle.layer_backward(X, np.array(g["ids"]), np.array(g["w"]), np.ones((1, 1)), P)
    assert gr["dw"][0].tolist() == pytest.approx([ex["o"] for ex in g["experts"]], rel=1e-14)


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(-40.0)) < 1e-15
    assert oracle.dsilu(0.0) == pytest.approx(0.5)
    z = np.linspace(-6, 6, 25)
    fd = (oracle.silu(z + 1e-6) - oracle.silu(z - 1e-6)) / 2e-6
    np.testing.assert_allclose(oracle.dsilu(z), fd, rtol=1e-8, atol=1e-10)


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_lora_equals_merged(seed, shared):
    P, X, ids, w, _ = _problem(seed, shared=shared)
    Y = oracle.layer_forward(X, ids, w, P)
    Ym = oracle.layer_forward_merged(X, ids, w, P)
    np.testing.assert_allclose(Y, Ym, rtol=1e-12, atol=1e-12)


def test_zero_lora_b_is_base_moe():
    P, X, ids, w, _ = _problem(5)
    P0 = copy.deepcopy(P)
    P0.B_gu[:] = 0
    P0.B_dn[:] = 0
    P1 = copy.deepcopy(P)
    P1.A_gu[:] = 7.0  # ignored once B = 0
    P1.A_dn[:] = -3.0
    P1.B_gu[:] = 0
    P1.B_dn[:] = 0
    np.testing.assert_allclose(oracle.layer_forward(X, ids, w, P0),
                               oracle.layer_forward(X, ids, w, P1), rtol=0, atol=1e-13)
    P2 = copy.deepcopy(P0)
    P2.s = 123.0
    np.testing.assert_allclose(oracle.layer_forward(X, ids, w, P0),
                               oracle.layer_forward(X, ids, w, P2), rtol=0, atol=1e-13)


def test_shared_expert_is_extra_slot():
    P, X, ids, w, dY = _problem(7, shared=True)
    T = X.shape[0]
    Y = oracle.layer_forward(X, ids, w, P)
    ids2 = np.concatenate([ids, np.full((T, 1), P.E, dtype=np.int32)], axis=1)
    w2 = np.concatenate([w, np.ones((T, 1))], axis=1)
    P2 = copy.deepcopy(P)
    P2.shared = False
    P2.E = P.E + 1
    np.testing.assert_allclose(Y, oracle.layer_forward(X, ids2, w2, P2), rtol=1e-13, atol=1e-13)
    g1 = oracle.layer_backward(X, ids, w, dY, P)
    g2 = oracle.layer_backward(X, ids2, w2, dY, P2)
    for n in ("dX", "dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        np.testing.assert_allclose(g1[n], g2[n], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g1["dw"], g2["dw"][:, :-1], rtol=1e-12, atol=1e-12)


def test_linear_in_routing_weights():
    P, X, ids, w, _ = _problem(11)
    w2 = np.random.default_rng(3).random(w.shape)
    Ya = oracle.layer_forward(X, ids, w, P)
    Yb = oracle.layer_forward(X, ids, w2, P)
    Yab = oracle.layer_forward(X, ids, 2.0 * w - 0.5 * w2, P)
    np.testing.assert_allclose(Yab, 2.0 * Ya - 0.5 * Yb, rtol=1e-12, atol=1e-12)


def test_single_expert_k1_is_dense_mlp():
    # k = 1, w = 1, one expert: every token runs the same SwiGLU-LoRA MLP;
    # compare against evaluating the merged dense MLP row by row
    P, X, _, _, _ = _problem(13, E=1, k=1)
    T = X.shape[0]
    ids = np.zeros((T, 1), dtype=np.int32)
    Y = oracle.layer_forward(X, ids, np.ones((T, 1)), P)
    Wgu, Wdn = oracle.merged_weights(P)
    f = P.f
    for t in range(T):
        h = Wgu[0] @ X[t]
        act = [h[i] / (1 + np.exp(-h[i])) * h[f + i] for i in range(f)]
        np.testing.assert_allclose(Y[t], Wdn[0] @ np.array(act), rtol=1e-12, atol=1e-12)


def _loss(P, X, ids, w, dY):
    return float(np.sum(oracle.layer_forward(X, ids, w, P) * dY))


@pytest.mark.parametrize("shared,dup", [(False, False), (True, False), (False, True)])
def test_gradients_finite_difference(shared, dup):
    P, X, ids, w, dY = _problem(21 + shared + 2 * dup, shared=shared, dup=dup)
    gr = oracle.layer_backward(X, ids, w, dY, P)
    rng = np.random.default_rng(99)
    eps = 1e-5

    def check(name, base, grad, setter):
        for _ in range(3):
            V = rng.standard_normal(base.shape)
            Lp = _loss(*setter(base + eps * V))
            Lm = _loss(*setter(base - eps * V))
            fd = (Lp - Lm) / (2 * eps)
            an = float(np.sum(grad * V))
            assert fd == pytest.approx(an, rel=1e-6, abs=1e-8), name

    check("dX", X, gr["dX"], lambda v: (P, v, ids, w, dY))
    check("dw", w, gr["dw"], lambda v: (P, X, ids, v, dY))
    for pname, gname in (("A_gu", "dA_gu"), ("B_gu", "dB_gu"), ("A_dn", "dA_dn"), ("B_dn", "dB_dn")):
        def setter(v, pname=pname):
            Q = copy.deepcopy(P)
            setattr(Q, pname, v)
            return (Q, X, ids, w, dY)
        check(gname, getattr(P, pname), gr[gname], setter)


@pytest.mark.parametrize("shared,dup", [(False, False), (True, True)])
def test_full_weight_gradients_finite_difference(shared, dup):
    """dW_gu and dW_dn (full fine-tuning) against central differences of the
    loss in the expert weights themselves."""
    P, X, ids, w, dY = _problem(51 + shared, shared=shared, dup=dup)
    gr = oracle.layer_backward(X, ids, w, dY, P, full=True)
    rng = np.random.default_rng(7)
    eps = 1e-5
    for pname in ("W_gu", "W_dn"):
        base = getattr(P, pname)
        for _ in range(3):
            V = rng.standard_normal(base.shape)
            Qp, Qm = copy.deepcopy(P), copy.deepcopy(P)
            setattr(Qp, pname, base + eps * V)
            setattr(Qm, pname, base - eps * V)
            fd = (_loss(Qp, X, ids, w, dY) - _loss(Qm, X, ids, w, dY)) / (2 * eps)
            an = float(np.sum(gr["d" + pname] * V))
            assert fd == pytest.approx(an, rel=1e-6, abs=1e-8), pname


def test_full_and_lora_gradients_are_tied():
    """W_eff = W + s B A, so dB = s dW A^T and dA = s B^T dW for both
    projections: the full gradients must reproduce the LoRA gradients that
    the chain rule computes along a different path (through xa, u, v)."""
    P, X, ids, w, dY = _problem(61, T=13, E=5, k=3, shared=True)
    gr = oracle.layer_backward(X, ids, w, dY, P, full=True)
    for g in range(P.E + 1):
        for proj in ("gu", "dn"):
            dW = gr["dW_" + proj][g]
            A, B = getattr(P, "A_" + proj)[g], getattr(P, "B_" + proj)[g]
            np.testing.assert_allclose(gr["dB_" + proj][g], P.s * dW @ A.T, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(gr["dA_" + proj][g], P.s * B.T @ dW, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("shared", [False, True])
def test_sampled_evaluators_agree(shared):
    P, X, ids, w, dY = _problem(31, T=11, E=5, k=2, shared=shared)
    Y = oracle.layer_forward(X, ids, w, P)
    gr = oracle.layer_backward(X, ids, w, dY, P)
    for t in (0, 4, 10):
        np.testing.assert_allclose(oracle.token_forward(t, X, ids, w, P), Y[t], rtol=1e-12, atol=1e-12)
        dx, dw = oracle.token_backward_dx(t, X, ids, w, dY, P)
        np.testing.assert_allclose(dx, gr["dX"][t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dw, gr["dw"][t], rtol=1e-12, atol=1e-12)
    grf = oracle.layer_backward(X, ids, w, dY, P, full=True)
    for g in range(P.E + (1 if shared else 0)):
        eg = oracle.expert_lora_grads(g, X, ids, w, dY, P, full=True)
        for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn", "dW_gu", "dW_dn"):
            np.testing.assert_allclose(eg[n], grf[n][g], rtol=1e-12, atol=1e-12)


def test_empty_expert_has_zero_grads():
    P, X, _, w, dY = _problem(41, E=4, k=2)
    T = X.shape[0]
    ids = np.tile(np.array([[0, 2]], dtype=np.int32), (T, 1))
    gr = oracle.layer_backward(X, ids, w, dY, P)
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        assert np.all(gr[n][1] == 0) and np.all(gr[n][3] == 0)
        assert np.any(gr[n][0] != 0)
