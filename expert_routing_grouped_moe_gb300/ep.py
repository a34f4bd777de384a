"""Expert-parallel MoE-LoRA layer: the experts split into contiguous ranges
over the ranks of a process group, token rows sent to the rank that owns
their expert and the results sent back (one all-to-all each way per pass).

The Unsloth x NVIDIA article's closing section points multi-GPU training at
sharding the experts and the data across GPUs; this module is that exchange
for the grouped layer of the article's routing section.  Rank q owns experts
[e_q, e_{q+1}) with e_q = floor(q E / P), their frozen weights and their LoRA
adapters; the LoRA gradients of an expert stay on its rank.

One pass on rank r (every step a library call or a collective):

  1. route its own tokens over all E experts (moe_route) and permute its rows
     into sorted order (moe_permute); the rows for rank q's experts are then
     the contiguous slice [offsets[e_q], offsets[e_{q+1}]);
  2. send every rank the counts of its experts (a fixed-size all-to-all), read
     the count matrix on the host once (the only host synchronisation: the
     all-to-all of rows needs its split sizes), and send the rows and their
     routing weights (moe_ep_row_weights) with an all-to-all of uneven splits;
  3. on the expert side, label the received rows with their local expert
     (moe_ep_segment_ids), regroup them by expert (moe_route, moe_permute with
     K = 1), run the grouped split-LoRA MLP with the received weights, and put
     the results back in received order (moe_unpermute_combine with K = 1);
  4. send the results back with the reverse all-to-all and combine them per
     token (moe_unpermute_combine).

The backward moves dY the same way, runs the grouped backward on the expert
side and returns dX rows and routing-weight gradients.  A shared expert is
not supported here (it would be replicated on every rank instead).

`ops` supplies the per-rank steps and `comm` the all-to-all, so the same
exchange plan runs over NCCL on GPUs (CudaOps, TorchComm) and can be checked
with other implementations of the two interfaces.
"""
from __future__ import annotations

import torch

from . import _lib as L


def expert_ranges(E: int, world: int):
    """Boundaries e_0 = 0 < ... < e_P = E of the contiguous expert ranges."""
    if not 1 <= world <= E:
        raise ValueError("need 1 <= world size <= E")
    return [(q * E) // world for q in range(world + 1)]


class TorchComm:
    """All-to-all of uneven splits over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all(self, out, inp, out_splits, in_splits):
        self.dist.all_to_all_single(out, inp, list(out_splits), list(in_splits), group=self.group)


class CudaOps:
    """The per-rank steps of expert parallelism on this GPU, through the C ABI.

    Source side: route / permute / row weights / combine over all E experts.
    Expert side: the grouped split-LoRA MLP of the E_loc local experts on the
    rows received from every rank, with its saved intermediates kept between
    forward and backward."""

    def __init__(self, d, f, E_loc, r, alpha, local_weights: dict, device):
        self.d, self.f, self.E_loc, self.r = d, f, E_loc, r
        self.scale = alpha / r
        self.dev = torch.device(device)
        self.w = {n: local_weights[n].contiguous() for n in
                  ("W_gu", "A_gu", "B_gu", "W_dn", "A_dn", "B_dn")}
        for n, t in self.w.items():
            if t.shape[0] != E_loc:
                raise ValueError("%s holds %d experts, expected %d" % (n, t.shape[0], E_loc))
        self._saved = None

    # -------------------------------------------------------------- helpers
    def _i32(self, *shape):
        return torch.empty(*shape, dtype=torch.int32, device=self.dev)

    def _route(self, ids, E):
        T, k = ids.shape
        t = {"counts": self._i32(E), "offsets": self._i32(E + 1), "tile_off": self._i32(E + 1),
             "sorted_src": self._i32(T * k), "dest_pos": self._i32(T * k)}
        ws = torch.empty(max(16, L.moe_route_workspace_size(T, k, E)), dtype=torch.uint8,
                         device=self.dev)
        L.moe_route(ids, E, False, t["counts"], t["offsets"], t["tile_off"], t["sorted_src"],
                    t["dest_pos"], ws)
        return t

    # ---------------------------------------------------------- source side
    def route(self, ids, E):
        return self._route(ids, E)

    def permute(self, rows, K, dest_pos):
        out = torch.empty(rows.shape[0] * K, rows.shape[1], dtype=rows.dtype, device=self.dev)
        L.moe_permute(rows, K, dest_pos, out)
        return out

    def row_weights(self, w, dest_pos):
        out = torch.empty(w.numel(), dtype=torch.float32, device=self.dev)
        L.moe_ep_row_weights(w, dest_pos, False, out)
        return out

    def combine(self, rows, dest_pos, k, row_scalars=None):
        T = dest_pos.numel() // k
        out = torch.empty(T, rows.shape[1], dtype=rows.dtype, device=self.dev)
        slot = None if row_scalars is None else torch.empty(T, k, dtype=torch.float32,
                                                             device=self.dev)
        L.moe_unpermute_combine(rows, dest_pos, k, False, out, row_scalars=row_scalars,
                                slot_out=slot)
        return out, slot

    # ---------------------------------------------------------- expert side
    def local_forward(self, rows, counts, row_w):
        """Rows received rank-major / expert-minor (counts [P, E_loc]) with their
        routing weights -> w * expert(row) in the same (received) order."""
        n = rows.shape[0]
        d, f, r, E = self.d, self.f, self.r, self.E_loc
        if n == 0:
            self._saved = None
            return torch.empty(0, d, dtype=torch.bfloat16, device=self.dev)
        seg = self._i32(n, 1)
        L.moe_ep_segment_ids(counts, seg)
        t = self._route(seg, E)                      # regroup by local expert (K = 1)
        Xl = self.permute(rows, 1, t["dest_pos"])
        dims = L.make_dims(n, d, f, E, 1, r, self.scale, False)
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        Yl = torch.empty(n, d, **bf)
        h = torch.empty(n, 32 * ((f + 15) // 16), dtype=torch.float32, device=self.dev)
        act = torch.empty(2, n, f, **bf)
        xa_gu = torch.empty(2, n, r, **bf)
        xa_dn = torch.empty(2, n, r, **bf)
        w = self.w
        L.moe_lora_grouped_mlp_fwd(dims, Xl, None, t["counts"], t["offsets"], t["tile_off"],
                                   t["sorted_src"], row_w.view(n, 1), w["W_gu"], w["A_gu"],
                                   w["B_gu"], w["W_dn"], w["A_dn"], w["B_dn"], Yl, h, act,
                                   xa_gu, xa_dn)
        self._saved = dict(dims=dims, t=t, Xl=Xl, h=h, act=act, xa_gu=xa_gu, xa_dn=xa_dn,
                           row_w=row_w.view(n, 1))
        out, _ = self.combine(Yl, t["dest_pos"], 1)  # back to received order
        return out

    def local_backward(self, dy_rows):
        """dY rows in received order -> (dX rows, routing-weight gradient per
        row, both in received order; LoRA gradients of the local experts)."""
        E, d, f, r = self.E_loc, self.d, self.f, self.r
        f32 = dict(dtype=torch.float32, device=self.dev)
        grads = {"dA_gu": torch.zeros(E, r, d, **f32), "dB_gu": torch.zeros(E, 2 * f, r, **f32),
                 "dA_dn": torch.zeros(E, r, f, **f32), "dB_dn": torch.zeros(E, d, r, **f32)}
        n = dy_rows.shape[0]
        if n == 0 or self._saved is None:
            return (torch.empty(0, d, dtype=torch.bfloat16, device=self.dev),
                    torch.empty(0, **f32), grads)
        sv, t, w = self._saved, self._saved["t"], self.w
        dYl = self.permute(dy_rows, 1, t["dest_pos"])
        dXl = torch.empty(n, d, dtype=torch.bfloat16, device=self.dev)
        dw_l = torch.empty(n, **f32)
        ws = torch.empty(L.moe_mlp_bwd_workspace_size(sv["dims"]), dtype=torch.uint8,
                         device=self.dev)
        L.moe_lora_grouped_mlp_bwd(sv["dims"], dYl, None, sv["Xl"], None, t["counts"],
                                   t["offsets"], t["tile_off"], t["sorted_src"], sv["row_w"],
                                   w["W_gu"], w["A_gu"], w["B_gu"], w["W_dn"], w["A_dn"],
                                   w["B_dn"], sv["h"], sv["act"], sv["xa_gu"], sv["xa_dn"], dXl,
                                   dw_l, grads["dA_gu"], grads["dB_gu"], grads["dA_dn"],
                                   grads["dB_dn"], ws)
        dx, dw = self.combine(dXl, t["dest_pos"], 1, row_scalars=dw_l)
        return dx, dw.view(n), grads


class ExpertParallelLayer:
    """One rank's view of the expert-parallel layer (see the module notes).

    T tokens on this rank, top-k of E experts; this rank owns experts
    [e_rank, e_rank+1).  forward(X, ids, w) -> Y [T,d];
    backward(dY) -> {dX, dw, dA_gu, dB_gu, dA_dn, dB_dn} (LoRA gradients of
    the local experts only)."""

    def __init__(self, E, k, comm, ops):
        self.E, self.k = E, k
        self.comm, self.ops = comm, ops
        self.P, self.rank = comm.world, comm.rank
        self.bounds = expert_ranges(E, self.P)
        self.E_loc = self.bounds[self.rank + 1] - self.bounds[self.rank]
        self._fw = None

    def plan(self, counts_host, recv_counts_host):
        """Row split sizes of the dispatch: to each rank (from this rank's
        per-expert counts) and from each rank (from the received count matrix
        [P, E_loc]).  The combine uses them reversed."""
        b = self.bounds
        send = [int(sum(counts_host[b[q]:b[q + 1]])) for q in range(self.P)]
        recv = [int(sum(row)) for row in recv_counts_host]
        return send, recv

    def forward(self, X, ids, w):
        ops, comm, k, P = self.ops, self.comm, self.k, self.P
        t = ops.route(ids, self.E)
        Xp = ops.permute(X, k, t["dest_pos"])
        wp = ops.row_weights(w, t["dest_pos"])
        # counts of this rank's rows for every rank's experts -> count matrix
        # of the rows this rank will receive, [P, E_loc]
        recv_counts = torch.empty(P * self.E_loc, dtype=t["counts"].dtype,
                                  device=t["counts"].device)
        comm.all_to_all(recv_counts, t["counts"], [self.E_loc] * P,
                        [self.bounds[q + 1] - self.bounds[q] for q in range(P)])
        host = torch.cat([t["counts"].reshape(-1), recv_counts]).cpu().tolist()
        counts_h, recv_h = host[:self.E], host[self.E:]
        recv_h = [recv_h[i * self.E_loc:(i + 1) * self.E_loc] for i in range(P)]
        send, recv = self.plan(counts_h, recv_h)
        n_recv = sum(recv)
        rows = Xp.new_empty((n_recv, Xp.shape[1]))
        comm.all_to_all(rows, Xp, recv, send)
        row_w = wp.new_empty((n_recv,))
        comm.all_to_all(row_w, wp, recv, send)
        out_rows = ops.local_forward(rows, recv_counts.view(P, self.E_loc), row_w)
        Yp = Xp.new_empty(Xp.shape)
        comm.all_to_all(Yp, out_rows, send, recv)
        Y, _ = ops.combine(Yp, t["dest_pos"], k)
        self._fw = dict(t=t, send=send, recv=recv, n_recv=n_recv)
        return Y

    def backward(self, dY):
        if self._fw is None:
            raise RuntimeError("backward before forward")
        ops, comm, k, fw = self.ops, self.comm, self.k, self._fw
        t = fw["t"]
        dYp = ops.permute(dY, k, t["dest_pos"])
        rows = dYp.new_empty((fw["n_recv"], dYp.shape[1]))
        comm.all_to_all(rows, dYp, fw["recv"], fw["send"])
        dx_rows, dw_rows, grads = ops.local_backward(rows)
        dXp = dYp.new_empty(dYp.shape)
        comm.all_to_all(dXp, dx_rows, fw["send"], fw["recv"])
        dwp = dw_rows.new_empty((dYp.shape[0],))
        comm.all_to_all(dwp, dw_rows, fw["send"], fw["recv"])
        dX, dw = ops.combine(dXp, t["dest_pos"], k, row_scalars=dwp)
        return {"dX": dX, "dw": dw, **grads}
