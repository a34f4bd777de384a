"""GPU parity of the whole MoE-LoRA layer (forward and backward) against the
fp64 oracle: every element at sizes the oracle finishes in seconds (several
tiles, ragged tails), sampled tokens and experts at the full workloads, edge
cases, determinism and CUDA-graph capture."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import MoELoRALayer, _lib as L, synth
from _util import assert_close_bf16, oracle_params, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = {
    "tiny": synth.CONFIGS["tiny"],
    # ragged: d, f not multiples of the tile widths; several row tiles per expert
    "ragged": synth.LayerConfig("ragged", T=1024, d=320, f=200, E=6, k=3, r=16, alpha=32),
    "shared_small": synth.LayerConfig("shared_small", T=384, d=192, f=136, E=8, k=2, r=24,
                                      alpha=48, shared=True, zipf_bias=3.0, n_blocked=2),
    "rank64": synth.LayerConfig("rank64", T=256, d=256, f=128, E=4, k=2, r=64, alpha=128),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def make_inputs(cfg, seed, ids=None, w=None):
    wts = synth.layer_weights(cfg, seed, device=DEV)
    act = synth.layer_activations(cfg, seed, device=DEV)
    if ids is None:
        ids_np, w_np = oracle.router_topk(act["logits"].cpu().numpy(), cfg.k)
    else:
        ids_np, w_np = ids, w
    return wts, act, ids_np, w_np


def run(cfg, wts, act, ids_np, w_np, gather=False, full=False, rank_r_tokens=False):
    layer = MoELoRALayer(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.r, cfg.alpha, wts,
                         shared_expert=cfg.shared, device=DEV, gather=gather, full_grads=full,
                         rank_r_tokens=rank_r_tokens)
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
    w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(DEV)
    Y = layer.forward(act["X"], ids, w).clone()
    g = {k: v.clone() for k, v in layer.backward(act["dY"]).items()}
    assert L.moe_status() == L.MOE_OK
    return layer, Y, g


def group_rows(ids_np, cfg):
    """Oracle routing -> (group, token list, flat list, permuted row list)."""
    T = ids_np.shape[0]
    a = ids_np
    if cfg.shared:
        a = np.concatenate([a, np.full((T, 1), cfg.E, dtype=a.dtype)], 1)
    K = a.shape[1]
    rt = oracle.route(a, cfg.groups)
    out = []
    for g in range(cfg.groups):
        seg = rt["sorted_src"][rt["offsets"][g]:rt["offsets"][g + 1]]
        out.append((g, seg // K, seg, rt["offsets"][g] + np.arange(seg.size)))
    return out, T * K


@pytest.mark.parametrize("mode", ["gather", "permuted", "rank_r_tokens"])
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_full_parity(name, mode):
    """gather: GEMMs gather token rows from X / dY; permuted: permuted copies;
    rank_r_tokens: permuted copies, the LoRA-A products gather token rows."""
    cfg = SMALL[name]
    gather = mode == "gather"
    wts, act, ids_np, w_np = make_inputs(cfg, seed=7)
    layer, Y, g = run(cfg, wts, act, ids_np, w_np, gather=gather,
                      rank_r_tokens=mode == "rank_r_tokens")
    P = oracle_params(wts, cfg)
    X, dY = to64(act["X"]), to64(act["dY"])
    s = cfg.scale
    wfull = np.concatenate([w_np, np.ones((cfg.T, 1))], 1) if cfg.shared else w_np
    groups, N = group_rows(ids_np, cfg)
    # forward intermediates, group by group, in the permuted layout
    names = ("xa_gu", "act", "xa_dn", "Yp") + (() if gather else ("Xp",))
    bufs = {n: to64(getattr(layer, n)) for n in names}
    bufs["h"] = to64(layer.h_gate_up())
    for n in ("xa_gu", "act", "xa_dn"):  # hi + lo pairs carry ~16 significant bits
        bufs[n] = bufs[n][0] + bufs[n][1]
    for gi, tok, flat, prow in groups:
        if tok.size == 0:
            continue
        fw = oracle.expert_forward(X[tok], P, gi)
        wt = wfull.reshape(-1)[flat]
        if not gather:
            np.testing.assert_array_equal(bufs["Xp"][prow], X[tok])
        # fp32 accumulation of exact bf16 products: far inside the bf16 bounds
        tight = dict(rel_fro=1e-4, elem=1e-4)
        assert_close_bf16(bufs["xa_gu"][prow], s * fw["xa"], "xa_gu g%d" % gi, **tight)
        assert_close_bf16(bufs["h"][prow], fw["h"], "h g%d" % gi, **tight)
        # the saved act and xa_dn carry the routing weight of their row
        assert_close_bf16(bufs["act"][prow], wt[:, None] * fw["act"], "act g%d" % gi, **tight)
        assert_close_bf16(bufs["xa_dn"][prow], s * wt[:, None] * fw["xa_dn"], "xa_dn g%d" % gi,
                          **tight)
        assert_close_bf16(bufs["Yp"][prow], wt[:, None] * fw["o"], "Yp g%d" % gi)
    for n, b in bufs.items():  # one permuted row per routed (token, slot)
        assert b.shape[0] == N, n
    # layer outputs
    assert_close_bf16(to64(Y), oracle.layer_forward(X, ids_np, w_np, P), "Y")
    gr = oracle.layer_backward(X, ids_np, w_np, dY, P)
    assert_close_bf16(to64(g["dX"]), gr["dX"], "dX")
    assert_close_bf16(g["dw"].cpu().numpy(), gr["dw"], "dw")
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        assert_close_bf16(g[n].cpu().numpy(), gr[n], n)


@pytest.mark.parametrize("name", list(SMALL))
def test_full_weight_gradients_parity(name):
    """Full fine-tuning: dW_gu and dW_dn of every group against the oracle,
    next to unchanged LoRA gradients and dX."""
    cfg = SMALL[name]
    wts, act, ids_np, w_np = make_inputs(cfg, seed=17)
    layer, Y, g = run(cfg, wts, act, ids_np, w_np, full=True)
    P = oracle_params(wts, cfg)
    X, dY = to64(act["X"]), to64(act["dY"])
    gr = oracle.layer_backward(X, ids_np, w_np, dY, P, full=True)
    for n in ("dW_gu", "dW_dn", "dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        assert_close_bf16(g[n].cpu().numpy(), gr[n], n)
    assert_close_bf16(to64(g["dX"]), gr["dX"], "dX")
    counts = np.bincount(ids_np.reshape(-1), minlength=cfg.E)
    for e in np.nonzero(counts == 0)[0]:
        assert np.all(g["dW_gu"][e].cpu().numpy() == 0) and np.all(g["dW_dn"][e].cpu().numpy() == 0)


@pytest.mark.parametrize("name", ["qwen3_30b_a3b", "gpt_oss_20b", "skewed_shared"])
def test_full_weight_gradients_sampled_full_size(name):
    """dW_gu / dW_dn at the full workload sizes (single-CTA and pair tiles,
    d = f = 2880 against every tile width): the largest and the smallest
    non-empty expert, and the shared expert, against the per-expert oracle."""
    cfg = synth.CONFIGS[name]
    wts, act, ids_np, w_np = make_inputs(cfg, seed=1)
    layer, Y, g = run(cfg, wts, act, ids_np, w_np, full=True)
    counts = np.bincount(ids_np.reshape(-1), minlength=cfg.E)
    groups = [int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))]
    if cfg.shared:
        groups.append(cfg.E)
    P = oracle_params(wts, cfg, groups=groups)
    X, dY = to64(act["X"]), to64(act["dY"])
    for gi in groups:
        ref = oracle.expert_lora_grads(gi, X, ids_np, w_np, dY, P, full=True)
        for n in ("dW_gu", "dW_dn"):
            assert_close_bf16(g[n][gi].cpu().numpy(), ref[n], "%s[g%d]" % (n, gi))


EDGE = {
    # one token
    "one_token": (synth.LayerConfig("one_token", T=1, d=128, f=64, E=4, k=2, r=8, alpha=16),
                  lambda T, E, k, rng: np.array([[3, 1]])),
    # every token to one expert (the others empty)
    "all_to_one": (synth.LayerConfig("all_to_one", T=300, d=128, f=64, E=5, k=1, r=8, alpha=16),
                   lambda T, E, k, rng: np.full((T, 1), 2)),
    # many empty experts, counts not multiples of the tile
    "sparse": (synth.LayerConfig("sparse", T=40, d=64, f=64, E=16, k=2, r=16, alpha=32),
               lambda T, E, k, rng: np.stack([rng.choice([1, 6, 11], size=2, replace=False)
                                              for _ in range(T)])),
    # the same expert twice in one token (both rows count)
    "duplicates": (synth.LayerConfig("duplicates", T=200, d=128, f=72, E=3, k=3, r=8, alpha=16),
                   lambda T, E, k, rng: rng.integers(0, E, size=(T, k))),
    # exactly one full tile per expert
    "exact_tiles": (synth.LayerConfig("exact_tiles", T=256, d=128, f=128, E=4, k=2, r=16,
                                      alpha=32),
                    lambda T, E, k, rng: np.stack([[t % 4, (t + 1) % 4] for t in range(T)])),
    # many experts: the GEMMs keep only tile_off in shared memory (G + 1 > 224)
    "experts_300": (synth.LayerConfig("experts_300", T=600, d=128, f=64, E=300, k=4, r=8,
                                      alpha=16),
                    lambda T, E, k, rng: np.stack([rng.choice(E, size=k, replace=False)
                                                   for _ in range(T)])),
    # more: the tile scheduler searches global memory (G + 1 > 448)
    "experts_600": (synth.LayerConfig("experts_600", T=700, d=128, f=64, E=600, k=4, r=8,
                                      alpha=16),
                    lambda T, E, k, rng: np.stack([rng.choice(E, size=k, replace=False)
                                                   for _ in range(T)])),
    # two groups far above the mean (90 % of the tokens on expert 3, and the
    # shared expert): the LoRA weight gradients sum their rows in several
    # parts (1024 rows each here, six per group) and add the parts in order
    "split_groups": (synth.LayerConfig("split_groups", T=6000, d=64, f=48, E=15, k=1, r=8,
                                       alpha=16, shared=True),
                     lambda T, E, k, rng: np.where(rng.random((T, 1)) < 0.9, 3,
                                                   rng.integers(0, E, size=(T, 1)))),
}


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("name", list(EDGE))
def test_layer_edge_cases(name, gather):
    cfg, mk = EDGE[name]
    rng = np.random.default_rng(5)
    ids_np = mk(cfg.T, cfg.E, cfg.k, rng).astype(np.int32)
    w_np = synth.combine_weights(cfg.T, cfg.k, seed=9).numpy()
    wts, act, ids_np, w_np = make_inputs(cfg, seed=13, ids=ids_np, w=w_np)
    layer, Y, g = run(cfg, wts, act, ids_np, w_np, gather=gather)
    P = oracle_params(wts, cfg)
    X, dY = to64(act["X"]), to64(act["dY"])
    assert_close_bf16(to64(Y), oracle.layer_forward(X, ids_np, w_np, P), "Y")
    gr = oracle.layer_backward(X, ids_np, w_np, dY, P)
    assert_close_bf16(to64(g["dX"]), gr["dX"], "dX")
    assert_close_bf16(g["dw"].cpu().numpy(), gr["dw"], "dw")
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
        assert_close_bf16(g[n].cpu().numpy(), gr[n], n)
        empty = [e for e in range(cfg.E) if not np.any(ids_np == e)]
        assert np.all(g[n].cpu().numpy()[empty] == 0), n


@pytest.mark.parametrize("name,gather", [("qwen3_30b_a3b", False), ("qwen3_30b_a3b", True),
                                         ("gpt_oss_20b", False), ("skewed_shared", False)])
def test_layer_full_size_sampled(name, gather):
    cfg = synth.CONFIGS[name]
    wts, act, ids_np, w_np = make_inputs(cfg, seed=1)
    layer, Y, g = run(cfg, wts, act, ids_np, w_np, gather=gather)
    rng = np.random.default_rng(3)
    # 40 random tokens plus the first and the last, and the rows of the
    # largest, the smallest non-empty, an empty, the shared and four random
    # experts (every tile shape the full-size kernels meet: ragged tails,
    # pair tiles with an idle half, experts spanning several tiles)
    toks = sorted(set(rng.choice(cfg.T, size=40, replace=False).tolist() + [0, cfg.T - 1]))
    counts = np.bincount(ids_np.reshape(-1), minlength=cfg.E)
    sample_groups = [int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))]
    empties = np.nonzero(counts == 0)[0]
    if empties.size:
        sample_groups.append(int(empties[0]))
    if cfg.shared:
        sample_groups.append(cfg.E)
    others = [e for e in np.nonzero(counts > 0)[0].tolist() if e not in sample_groups]
    sample_groups += [int(e) for e in rng.choice(others, size=min(4, len(others)), replace=False)]
    need = set(sample_groups)
    for t in toks:
        need.update(int(e) for e in ids_np[t])
    if cfg.shared:
        need.add(cfg.E)
    P = oracle_params(wts, cfg, groups=sorted(need))
    X, dY = act["X"], act["dY"]
    tsel = torch.tensor(toks, device=DEV)
    Xs, dYs = to64(X[tsel]), to64(dY[tsel])
    Xh = {t: Xs[i] for i, t in enumerate(toks)}
    Yg, dXg, dwg = to64(Y[tsel]), to64(g["dX"][tsel]), g["dw"][tsel].cpu().numpy()
    for i, t in enumerate(toks):
        Xrow = {t: Xh[t]}          # the per-token oracle reads row t only
        dYrow = {t: dYs[i]}
        assert_close_bf16(Yg[i], oracle.token_forward(t, Xrow, ids_np, w_np, P), "Y[%d]" % t)
        dx, dw = oracle.token_backward_dx(t, Xrow, ids_np, w_np, dYrow, P)
        assert_close_bf16(dXg[i], dx, "dX[%d]" % t)
        assert_close_bf16(dwg[i], dw, "dw[%d]" % t)
    Xall, dYall = to64(X), to64(dY)
    for gi in sample_groups:
        ref = oracle.expert_lora_grads(gi, Xall, ids_np, w_np, dYall, P)
        for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
            got = g[n][gi].cpu().numpy()
            if not np.any(ref[n]):
                assert np.all(got == 0), (n, gi)
            else:
                assert_close_bf16(got, ref[n], "%s[g%d]" % (n, gi))


@pytest.mark.parametrize("name", ["ragged", "split_groups"])
def test_layer_deterministic_and_graph_capturable(name):
    if name in SMALL:
        cfg = SMALL[name]
        wts, act, ids_np, w_np = make_inputs(cfg, seed=21)
    else:
        cfg, mk = EDGE[name]
        ids_np = mk(cfg.T, cfg.E, cfg.k, np.random.default_rng(5)).astype(np.int32)
        w_np = synth.combine_weights(cfg.T, cfg.k, seed=9).numpy()
        wts, act, ids_np, w_np = make_inputs(cfg, seed=21, ids=ids_np, w=w_np)
    layer, Y1, g1 = run(cfg, wts, act, ids_np, w_np)
    ids = torch.from_numpy(ids_np).to(DEV)
    w = torch.from_numpy(w_np).to(DEV)
    Y2 = layer.forward(act["X"], ids, w).clone()
    g2 = {k: v.clone() for k, v in layer.backward(act["dY"]).items()}
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    for n in g1:
        assert torch.equal(g1[n].view(torch.int32) if g1[n].dtype == torch.float32
                           else g1[n].view(torch.int16),
                           g2[n].view(torch.int32) if g2[n].dtype == torch.float32
                           else g2[n].view(torch.int16)), n
    # the whole fwd + bwd step, captured without any host synchronisation
    for buf in (layer.Y, layer.dX, layer.dw, *layer.grads.values()):
        buf.zero_()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer.step(act["X"], ids, w, act["dY"])
    torch.cuda.current_stream().wait_stream(s)
    for buf in (layer.Y, layer.dX, layer.dw, *layer.grads.values()):
        buf.fill_(3.0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.Y.view(torch.int16), Y1.view(torch.int16))
    assert torch.equal(layer.dX.view(torch.int16), g1["dX"].view(torch.int16))
    for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn", "dw"):
        got = layer.grads[n] if n != "dw" else layer.dw
        assert torch.equal(got, g1[n]), n
