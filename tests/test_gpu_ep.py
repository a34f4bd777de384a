"""Expert parallelism on one GPU: the two index kernels bit-exact, and the
expert-parallel layer with two or three ranks simulated in one process
(threads, each rank's steps through the library; the all-to-all is a host
loopback that copies slices once every rank has posted its buffer, so no
kernel ever waits on another) against the fp64 oracle layer."""
import threading

import numpy as np
import pytest
import torch

import oracle
from expert_routing_grouped_moe_gb300 import _lib as L, synth
from expert_routing_grouped_moe_gb300.ep import CudaOps, ExpertParallelLayer, expert_ranges
from _util import assert_close_bf16, oracle_params, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


# ------------------------------------------------------------- index kernels

@pytest.mark.parametrize("T,k,shared", [(1, 1, False), (300, 3, True), (4096, 8, False)])
def test_ep_row_weights_bit_exact(T, k, shared):
    E = 16
    ids = synth.topk_ids(T, E, k, "zipf", seed=3, device=DEV)
    w = synth.combine_weights(T, k, seed=3, device=DEV)
    K, G = k + int(shared), E + int(shared)
    t = {n: torch.empty(s, dtype=torch.int32, device=DEV) for n, s in
         (("counts", G), ("offsets", G + 1), ("tile_off", G + 1), ("sorted_src", T * K),
          ("dest_pos", T * K))}
    ws = torch.empty(L.moe_route_workspace_size(T, K, G), dtype=torch.uint8, device=DEV)
    L.moe_route(ids, E, shared, t["counts"], t["offsets"], t["tile_off"], t["sorted_src"],
                t["dest_pos"], ws)
    row_w = torch.full((T * K,), -1.0, device=DEV)
    L.moe_ep_row_weights(w, t["dest_pos"], shared, row_w)
    torch.cuda.synchronize()
    a = ids.cpu().numpy()
    if shared:
        a = np.concatenate([a, np.full((T, 1), E)], 1)
    rt = oracle.route(a, G)
    wf = np.concatenate([w.cpu().numpy(), np.ones((T, 1), np.float32)], 1) if shared \
        else w.cpu().numpy()
    exp = np.empty(T * K, np.float32)
    exp[rt["dest_pos"]] = wf.reshape(-1)
    np.testing.assert_array_equal(row_w.cpu().numpy(), exp)


@pytest.mark.parametrize("P,E_loc,empty_frac", [(1, 1, 0.0), (2, 4, 0.3), (8, 128, 0.5),
                                                (16, 1024, 0.9)])
def test_ep_segment_ids_bit_exact(P, E_loc, empty_frac):
    rng = np.random.default_rng(P * 1000 + E_loc)
    c = rng.integers(0, 40, size=(P, E_loc)).astype(np.int32)
    c[rng.random((P, E_loc)) < empty_frac] = 0
    n = int(c.sum())
    ids = torch.full((max(n, 1),), -1, dtype=torch.int32, device=DEV)[:n]
    L.moe_ep_segment_ids(torch.from_numpy(c).to(DEV), ids)
    assert L.moe_status() == L.MOE_OK
    exp = np.repeat(np.tile(np.arange(E_loc), P), c.reshape(-1))
    np.testing.assert_array_equal(ids.cpu().numpy(), exp)


def test_ep_segment_ids_count_mismatch_is_reported():
    c = torch.tensor([[3, 0], [1, 2]], dtype=torch.int32, device=DEV)
    ids = torch.full((5,), -1, dtype=torch.int32, device=DEV)   # the counts sum to 6
    L.moe_ep_segment_ids(c, ids)
    assert L.moe_status() == L.MOE_ERR_BAD_IDS
    assert torch.all(ids == -1)


# ------------------------------------------------------------------ the layer

class _Loopback:
    """All-to-all among `world` threads of one process: each rank posts its
    buffer and split sizes, waits for all, copies its pieces, waits again."""

    def __init__(self, world):
        self.world = world
        self.bar = threading.Barrier(world, timeout=300)
        self.box = [None] * world

    def comm(self, rank):
        group = self

        class _Comm:
            def __init__(self):
                self.rank, self.world = rank, group.world

            def all_to_all(self, out, inp, out_splits, in_splits):
                group.box[rank] = (inp, list(in_splits))
                group.bar.wait()
                off = 0
                for src in range(group.world):
                    buf, sp = group.box[src]
                    start, n = sum(sp[:rank]), sp[rank]
                    assert n == out_splits[src]
                    if n:
                        out[off:off + n].copy_(buf[start:start + n])
                    off += n
                group.bar.wait()
        return _Comm()


def _run_ranks(world, fn):
    errs = [None] * world

    def body(q):
        try:
            fn(q)
        except BaseException as e:  # noqa: BLE001 (re-raised below)
            errs[q] = e
    th = [threading.Thread(target=body, args=(q,)) for q in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for e in errs:
        if e is not None:
            raise e


@pytest.mark.parametrize("world,cfg", [
    (2, synth.LayerConfig("ep_small", T=300, d=128, f=64, E=8, k=2, r=16, alpha=32)),
    (3, synth.LayerConfig("ep_ragged", T=257, d=320, f=200, E=7, k=3, r=8, alpha=16)),
    (2, synth.LayerConfig("ep_qwen3_like", T=512, d=2048, f=768, E=128, k=8, r=64,
                          alpha=128)),
])
def test_expert_parallel_layer_matches_oracle(world, cfg):
    wts = synth.layer_weights(cfg, seed=21, device=DEV)
    b = expert_ranges(cfg.E, world)
    lb = _Loopback(world)
    inputs, outs = [], [None] * world
    for q in range(world):
        act = synth.layer_activations(cfg, seed=40 + q, device=DEV)
        ids_np, w_np = oracle.router_topk(act["logits"].cpu().numpy(), cfg.k)
        inputs.append((act, ids_np, w_np))

    def rank_fn(q):
        act, ids_np, w_np = inputs[q]
        local = {n: t[b[q]:b[q + 1]] for n, t in wts.items()}
        ops = CudaOps(cfg.d, cfg.f, b[q + 1] - b[q], cfg.r, cfg.alpha, local, DEV)
        layer = ExpertParallelLayer(cfg.E, cfg.k, lb.comm(q), ops)
        ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
        w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(DEV)
        Y = layer.forward(act["X"], ids, w)
        g = layer.backward(act["dY"])
        torch.cuda.synchronize()
        outs[q] = (Y.clone(), {n: v.clone() for n, v in g.items()})

    _run_ranks(world, rank_fn)
    assert L.moe_status() == L.MOE_OK
    P = oracle_params(wts, cfg)
    cat = lambda f: np.concatenate([f(q) for q in range(world)])  # noqa: E731
    Xall = cat(lambda q: to64(inputs[q][0]["X"]))
    dYall = cat(lambda q: to64(inputs[q][0]["dY"]))
    ref_all = oracle.layer_backward(Xall, cat(lambda q: inputs[q][1]),
                                    cat(lambda q: inputs[q][2]), dYall, P)
    t0 = 0
    for q in range(world):
        act, ids_np, w_np = inputs[q]
        Y, g = outs[q]
        T = act["X"].shape[0]
        tag = "%s rank %d" % (cfg.name, q)
        assert_close_bf16(to64(Y), oracle.layer_forward(to64(act["X"]), ids_np, w_np, P),
                          tag + " Y")
        assert_close_bf16(to64(g["dX"]), ref_all["dX"][t0:t0 + T], tag + " dX")
        assert_close_bf16(g["dw"].cpu().numpy(), ref_all["dw"][t0:t0 + T], tag + " dw")
        for n in ("dA_gu", "dB_gu", "dA_dn", "dB_dn"):
            assert_close_bf16(g[n].cpu().numpy(), ref_all[n][b[q]:b[q + 1]], tag + " " + n)
        t0 += T
