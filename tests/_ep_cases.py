"""Seeded inputs and oracle-backed per-rank steps for the expert-parallel
tests (test infrastructure: the oracle computes every step here).

``OracleOps`` implements the per-rank interface of
``expert_routing_grouped_moe_gb300.ep`` (route / permute / row weights /
combine on the token side, the local experts' MLP on the expert side) with
the oracle, so the exchange plan and its collectives can run over gloo on the
CPU and be compared with the single-process oracle layer."""
import numpy as np
import torch

import oracle

CASES = {
    # world, E, k, tokens per rank, d, f, r; "skew" sends most rows to rank 0
    "even2": dict(world=2, E=6, k=2, T=(40, 57), d=16, f=12, r=4, skew=False),
    "uneven3": dict(world=3, E=7, k=3, T=(30, 1, 45), d=8, f=16, r=8, skew=False),
    "skew2": dict(world=2, E=4, k=1, T=(33, 20), d=16, f=8, r=4, skew=True),
}


def full_params(case, seed=5):
    c = CASES[case]
    rng = np.random.default_rng(seed)
    E, d, f, r = c["E"], c["d"], c["f"], c["r"]
    return oracle.OracleParams(
        W_gu=rng.standard_normal((E, 2 * f, d)) / np.sqrt(d),
        A_gu=rng.standard_normal((E, r, d)) / np.sqrt(d),
        B_gu=rng.standard_normal((E, 2 * f, r)) * 0.1,
        W_dn=rng.standard_normal((E, d, f)) / np.sqrt(f),
        A_dn=rng.standard_normal((E, r, f)) / np.sqrt(f),
        B_dn=rng.standard_normal((E, d, r)) * 0.1, s=2.0, E=E)


def local_params(P, lo, hi):
    return oracle.OracleParams(W_gu=P.W_gu[lo:hi], A_gu=P.A_gu[lo:hi], B_gu=P.B_gu[lo:hi],
                               W_dn=P.W_dn[lo:hi], A_dn=P.A_dn[lo:hi], B_dn=P.B_dn[lo:hi],
                               s=P.s, E=hi - lo)


def rank_inputs(case, rank):
    """X [T,d], ids [T,k] (distinct per token), w [T,k], dY [T,d] of one rank."""
    c = CASES[case]
    rng = np.random.default_rng(100 + rank)
    T, E, k, d = c["T"][rank], c["E"], c["k"], c["d"]
    if c["skew"]:
        ids = np.zeros((T, k), dtype=np.int64)       # every row to expert 0 (rank 0)
    else:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k)) + 0.1
    w /= w.sum(1, keepdims=True)
    return rng.standard_normal((T, d)), ids, w, rng.standard_normal((T, d))


class OracleOps:
    """The per-rank steps of expert parallelism computed by the oracle, on
    float64 / int64 CPU tensors."""

    def __init__(self, P_local):
        self.P = P_local
        self._saved = None

    @staticmethod
    def _np(t):
        return t.detach().cpu().numpy()

    def route(self, ids, E):
        rt = oracle.route(self._np(ids), E)
        return {n: torch.from_numpy(np.asarray(v, dtype=np.int64)) for n, v in rt.items()}

    def permute(self, rows, K, dest_pos):
        dp = self._np(dest_pos)
        sorted_src = np.empty_like(dp)
        sorted_src[dp] = np.arange(dp.size)
        return torch.from_numpy(oracle.permute(self._np(rows), sorted_src, K))

    def row_weights(self, w, dest_pos):
        out = np.empty(w.numel())
        out[self._np(dest_pos)] = self._np(w).reshape(-1)
        return torch.from_numpy(out)

    def combine(self, rows, dest_pos, k, row_scalars=None):
        dp = self._np(dest_pos)
        Y = oracle.combine(self._np(rows), dp, k)
        slot = None
        if row_scalars is not None:
            slot = torch.from_numpy(self._np(row_scalars)[dp].reshape(-1, k))
        return torch.from_numpy(Y), slot

    def local_forward(self, rows, counts, row_w):
        c = self._np(counts)
        P_ranks, E_loc = c.shape
        seg = np.repeat(np.tile(np.arange(E_loc), P_ranks), c.reshape(-1))
        x, wr = self._np(rows), self._np(row_w)
        self._saved = (x, seg[:, None], wr[:, None])
        if x.shape[0] == 0:
            return torch.zeros(0, x.shape[1], dtype=torch.float64)
        return torch.from_numpy(oracle.layer_forward(x, seg[:, None], wr[:, None], self.P))

    def local_backward(self, dy_rows):
        x, seg, wr = self._saved
        names = ("dA_gu", "dB_gu", "dA_dn", "dB_dn")
        if x.shape[0] == 0:
            return (torch.zeros(0, x.shape[1], dtype=torch.float64),
                    torch.zeros(0, dtype=torch.float64),
                    {n: torch.zeros(getattr(self.P, n[1:]).shape, dtype=torch.float64)
                     for n in names})
        g = oracle.layer_backward(x, seg, wr, self._np(dy_rows), self.P)
        return (torch.from_numpy(g["dX"]), torch.from_numpy(g["dw"][:, 0]),
                {n: torch.from_numpy(g[n]) for n in names})
