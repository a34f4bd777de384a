"""MoE-LoRA expert layer object: owns the device buffers, calls the C ABI.

``MoELoRALayer`` is a convenience wrapper over the library's calls for one
layer shape: it allocates every buffer once (torch device memory), then
``forward`` runs route -> grouped split-LoRA SwiGLU MLP -> combine and
``backward`` runs the grouped backward -> combine of dX and of the
routing-weight gradient.  With ``gather=False`` (default) the token rows are
first permuted into Xp / dYp by moe_permute and the GEMMs read them with TMA;
with ``gather=True`` the GEMMs copy token rows straight from X and dY
(sorted_src picks them), which saves the two [N, d] permuted buffers but is
slower on GB300.  All arithmetic happens in the CUDA library; this module
only sequences calls and owns memory.
"""
from __future__ import annotations

import torch

from . import _lib as L

# Kernel launches issued by one forward / one backward in the default
# (permuted) mode: route 2 or 3 (L.moe_route_kernel_count), permute 1,
# forward GEMMs 4, combine 1; backward: permute 1, GEMMs 4 + weight-gradient
# GEMMs 4, partial-sum 1, combine 1.  The gather mode issues no permute.
LAUNCHES_FWD = 6   # besides the route's
LAUNCHES_BWD = 11


class MoELoRALayer:
    def __init__(self, T, d, f, E, k, r, alpha, weights: dict, shared_expert=False,
                 device="cuda", gather=False, full_grads=False, rank_r_tokens=False):
        """full_grads: the backward also returns dW_gu [G,2f,d] and dW_dn
        [G,d,f] (fp32 gradients of the expert weights, for full fine-tuning;
        needs the permuted-row mode).  rank_r_tokens (permuted-row mode):
        the LoRA-A products xa_gu and u read the token rows of X / dY (small
        enough to stay in L2) instead of the permuted copies."""
        if full_grads and gather:
            raise ValueError("full weight gradients need the permuted-row mode (gather=False)")
        self.gather = bool(gather)
        self.rank_r_tokens = bool(rank_r_tokens) and not self.gather
        self.full_grads = bool(full_grads)
        self.dims = L.make_dims(T, d, f, E, k, r, alpha / r, shared_expert)
        self.T, self.d, self.f, self.E, self.k, self.r = T, d, f, E, k, r
        self.shared = bool(shared_expert)
        self.G = E + (1 if shared_expert else 0)
        self.K = k + (1 if shared_expert else 0)
        self.N = T * self.K          # permuted rows, in sorted order
        dev = torch.device(device)
        self.w = {n: weights[n].contiguous() for n in ("W_gu", "A_gu", "B_gu", "W_dn", "A_dn",
                                                          "B_dn")}
        i32 = dict(dtype=torch.int32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        P, G = self.N, self.G
        self.counts = torch.zeros(G, **i32)
        self.offsets = torch.zeros(G + 1, **i32)
        self.tile_off = torch.zeros(G + 1, **i32)
        self.sorted_src = torch.zeros(self.N, **i32)
        self.dest_pos = torch.zeros(self.N, **i32)
        self.route_ws = torch.empty(max(16, L.moe_route_workspace_size(T, self.K, G)),
                                    dtype=torch.uint8, device=dev)
        self.Xp = None if self.gather else torch.empty(P, d, **bf)
        self.Yp = torch.empty(P, d, **bf)
        # saved intermediates: h in fp32; act / xa_gu / xa_dn as hi+lo bf16 pairs
        self.h = torch.empty(P, 32 * ((f + 15) // 16), **f32)  # [gate 16 | up 16] chunks
        self.act = torch.empty(2, P, f, **bf)
        self.xa_gu = torch.empty(2, P, r, **bf)
        self.xa_dn = torch.empty(2, P, r, **bf)
        self.Y = torch.empty(T, d, **bf)
        self.dYp = None if self.gather else torch.empty(P, d, **bf)
        self.dXp = torch.empty(P, d, **bf)
        self.dw_rows = torch.empty(P, **f32)
        self.dX = torch.empty(T, d, **bf)
        self.dw = torch.empty(T, k, **f32)
        self.grads = {
            "dA_gu": torch.empty(G, r, d, **f32), "dB_gu": torch.empty(G, 2 * f, r, **f32),
            "dA_dn": torch.empty(G, r, f, **f32), "dB_dn": torch.empty(G, d, r, **f32),
        }
        if self.full_grads:
            self.grads["dW_gu"] = torch.empty(G, 2 * f, d, **f32)
            self.grads["dW_dn"] = torch.empty(G, d, f, **f32)
        self.bwd_ws = torch.empty(L.moe_mlp_bwd_workspace_size(self.dims), dtype=torch.uint8,
                                  device=dev)
        self._ids = None
        self._topk_w = None

    def launches_per_step(self):
        """Kernel launches of one forward + backward in this layer's mode."""
        return (L.moe_route_kernel_count(self.T, self.K, self.G) + LAUNCHES_FWD + LAUNCHES_BWD
                - (2 if self.gather else 0) + (2 if self.full_grads else 0))

    # ------------------------------------------------------------------ steps
    def route(self, ids, stream=None):
        L.moe_route(ids, self.E, self.shared, self.counts, self.offsets, self.tile_off,
                    self.sorted_src, self.dest_pos, self.route_ws, stream)

    def forward(self, X, ids, topk_w, stream=None):
        """Y [T,d] bf16 for token rows X [T,d], top-k ids [T,k], weights [T,k]."""
        self._ids, self._topk_w, self._X = ids, topk_w, X
        self.route(ids, stream)
        if not self.gather:
            L.moe_permute(X, self.K, self.dest_pos, self.Xp, stream)
        w = self.w
        X_tok = X if (self.Xp is None or self.rank_r_tokens) else None
        L.moe_lora_grouped_mlp_fwd(self.dims, self.Xp, X_tok,
                                   self.counts, self.offsets, self.tile_off,
                                   self.sorted_src, topk_w, w["W_gu"], w["A_gu"], w["B_gu"],
                                   w["W_dn"], w["A_dn"], w["B_dn"], self.Yp, self.h, self.act,
                                   self.xa_gu, self.xa_dn, stream)
        L.moe_unpermute_combine(self.Yp, self.dest_pos, self.k, self.shared, self.Y,
                                stream=stream)
        return self.Y

    def backward(self, dY, stream=None):
        """dX [T,d] bf16, dw [T,k] fp32 and the four fp32 LoRA gradients."""
        if self._ids is None:
            raise RuntimeError("backward before forward")
        if not self.gather:
            L.moe_permute(dY, self.K, self.dest_pos, self.dYp, stream)
        w, g = self.w, self.grads
        dY_tok = dY if (self.dYp is None or self.rank_r_tokens) else None
        L.moe_lora_grouped_mlp_bwd(self.dims, self.dYp, dY_tok,
                                   self.Xp, None if self.Xp is not None else self._X,
                                   self.counts, self.offsets,
                                   self.tile_off, self.sorted_src, self._topk_w, w["W_gu"],
                                   w["A_gu"], w["B_gu"], w["W_dn"], w["A_dn"], w["B_dn"], self.h,
                                   self.act, self.xa_gu, self.xa_dn, self.dXp, self.dw_rows,
                                   g["dA_gu"], g["dB_gu"], g["dA_dn"], g["dB_dn"], self.bwd_ws,
                                   stream, dW_gu=g.get("dW_gu"), dW_dn=g.get("dW_dn"))
        L.moe_unpermute_combine(self.dXp, self.dest_pos, self.k, self.shared, self.dX,
                                row_scalars=self.dw_rows, slot_out=self.dw, stream=stream)
        return {"dX": self.dX, "dw": self.dw, **g}

    def step(self, X, ids, topk_w, dY, stream=None):
        """One forward + backward pass of the layer (the hot path)."""
        self.forward(X, ids, topk_w, stream)
        return self.backward(dY, stream)

    def h_gate_up(self):
        """The saved pre-activations as a plain [N, 2f] (gate | up) fp32 tensor
        (un-interleaves the 16-feature chunks of the stored layout)."""
        n, f = self.N, self.f
        hc = self.h.view(n, -1, 2, 16)
        gate = hc[:, :, 0, :].reshape(n, -1)[:, :f]
        up = hc[:, :, 1, :].reshape(n, -1)[:, :f]
        return torch.cat([gate, up], dim=1)
