"""NumPy fp64 oracle for routing, split-LoRA SwiGLU experts and combine.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every array that comes
in is converted to float64 (bf16 and fp32 values are exact in fp64) and no
intermediate is rounded.  Sources, cited by page and section:

[R]  Unsloth x NVIDIA article on three training optimisations, section
     "Optimisation 3: MoE routing done in one grouped pass" -- the old
     per-expert ``torch.where`` loop and the new five steps: flatten the
     top-k assignments, stable-sort by expert id, one bincount, offsets from
     the counts, slice the token list by offsets.
[G]  Unsloth "Faster MoE" docs, section "What is torch._grouped_mm" --
     experts stored as one ``gate_up_proj`` parameter [E, 2*inter, hidden];
     ``gate, up = linear(x, gate_up_proj[e]).chunk(2, dim=-1)``.
[L]  Unsloth "Faster MoE" docs, section "Faster LoRA MoE training" -- split
     LoRA: compute (X A) B beside X W instead of merging B A into W; the
     result is mathematically identical (associativity), so outputs and
     gradients are unchanged; the router is frozen; lora_alpha = 2 r.
[S]  same docs, section "Implementation details / MoE LoRA changes the
     picture" -- the split-LoRA equations Y = X A (s x r), Z = Y B (s x n)
     next to X W, per routed token-expert pair.
[I]  same docs, introduction -- the MoE kernels serve full fine-tuning as
     well as LoRA (the section "Faster LoRA MoE training" likewise advises
     bf16 for LoRA or full fine-tuning): the full gradients of the expert
     weights are the plain chain rule through the same forward.

Readings where the pages are silent (each listed in the design notes):
* LoRA orientation is PEFT's: A [r, in], B [out, r], delta = s * B @ A with
  s = alpha / r, so a row x maps to x @ W.T + s * (x @ A.T) @ B.T ([L], [S]
  write the same product transposed).
* One adapter on the fused gate_up projection (A_gu [r,d], B_gu [2f,r]) and
  one on down (A_dn [r,f], B_dn [d,r]).
* SwiGLU is silu(gate) * up with silu(z) = z / (1 + exp(-z)); the first f
  outputs of gate_up are gate, the next f are up ([G] ``chunk(2, -1)``).
* Combine: Y[t] = sum_j w[t,j] * expert_{ids[t,j]}(X[t]) (+ the shared
  expert's output with weight 1).  The pages do not print this step; it is
  the plain top-k mixture.
* Router: softmax over all E logits, top-k by descending logit (ties: lower
  expert id first), weights renormalised to sum to one.
"""
from __future__ import annotations

import dataclasses

import numpy as np


# ---------------------------------------------------------------------------
# Router (upstream of the layer; frozen per [L])
# ---------------------------------------------------------------------------

def router_topk(logits, k: int):
    """Softmax over E, top-k by descending logit, renormalised weights.

    Ties between equal logits go to the lower expert id.  Returns ids [T,k]
    int32 (slot order = descending logit) and weights [T,k] float32.
    """
    z = np.asarray(logits, dtype=np.float64)
    T, E = z.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # lexsort sorts by the last key first: descending logit, then ascending id
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    eidx = np.arange(E)
    for t in range(T):
        order = np.lexsort((eidx, -z[t]))
        sel = order[:k]
        m = np.max(z[t][np.isfinite(z[t])]) if np.isfinite(z[t]).any() else 0.0
        p = np.exp(z[t] - m)
        p = p / p.sum()
        ps = p[sel]
        ids[t] = sel
        w[t] = (ps / ps.sum()).astype(np.float32)
    return ids, w


# ---------------------------------------------------------------------------
# Routing [R]
# ---------------------------------------------------------------------------

def route(ids, E: int):
    """The grouped routing pass of [R], steps 1-5.

    1. flatten the [T,k] assignments row-major: flat index i = t*k + j;
    2. stable-sort the flat list by expert id -> ``sorted_src`` (the flat
       index found at each sorted position);
    3. one bincount -> ``counts[E]``;
    4. offsets = exclusive prefix sum of the counts -> ``offsets[E+1]``;
    5. expert e's slice of the token list is sorted_src[offsets[e]:offsets[e+1]].
    ``dest_pos`` is the inverse permutation (sorted position of flat index i).
    """
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    sorted_src = np.argsort(flat, kind="stable").astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    dest_pos = np.empty_like(sorted_src)
    dest_pos[sorted_src] = np.arange(flat.size)
    return {"counts": counts, "offsets": offsets,
            "sorted_src": sorted_src, "dest_pos": dest_pos}


def route_where_loop(ids, E: int):
    """The old per-expert loop of [R]: for each expert, the (token, slot)
    pairs where the router picked it, scanning the [T,k] id matrix row-major.
    Returns a list of flat-index arrays, one per expert."""
    a = np.asarray(ids)
    T, k = a.shape
    out = []
    for e in range(E):
        tok, slot = np.where(a == e)        # row-major scan, like torch.where
        out.append((tok * k + slot).astype(np.int64))
    return out


def permute(X, sorted_src, K: int):
    """Step 5 of [R] applied to the token rows: the rows in expert-grouped
    order.  Sorted position p holds the assignment with flat index
    i = sorted_src[p] = t*K + j, so row p of the result is token t's row:
        Xp[p] = X[sorted_src[p] // K]
    (K slots per token: the top-k slots, plus the shared expert's slot when
    there is one).  A pure gather; no value changes."""
    X = np.asarray(X)
    src = np.asarray(sorted_src, dtype=np.int64)
    if src.size and (src.min() < 0 or src.max() >= X.shape[0] * K):
        raise ValueError("sorted_src entry out of range")
    return X[src // K]


def combine(rows, dest_pos, K: int, weights=None):
    """Weighted combine of permuted rows back into token order (the top-k
    mixture; the pages do not print this step).  Token t's slot j sits at
    permuted row dest_pos[t*K + j]; with c_j its coefficient,
        Y[t] = sum_j c_j * rows[dest_pos[t*K + j]]
    c_j = weights[t, j] for the weights' k columns and 1 for any further slot
    (the shared expert's), or 1 for every slot when weights is None.  Exact
    fp64 sum (no rounding order to match)."""
    R = np.asarray(rows, dtype=np.float64)
    dp = np.asarray(dest_pos, dtype=np.int64)
    if dp.size % K:
        raise ValueError("dest_pos length is not a multiple of K")
    T = dp.size // K
    c = np.ones((T, K))
    if weights is not None:
        w = np.asarray(weights, dtype=np.float64)
        c[:, :w.shape[1]] = w
    Y = np.zeros((T, R.shape[1]))
    for j in range(K):
        Y += c[:, j:j + 1] * R[dp.reshape(T, K)[:, j]]
    return Y


# ---------------------------------------------------------------------------
# Expert MLP with split LoRA [G], [L], [S]
# ---------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def dsilu(z):
    """d/dz [z * sigmoid(z)] = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    z = np.asarray(z, dtype=np.float64)
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


@dataclasses.dataclass
class OracleParams:
    """Expert weights in fp64.  Group index E (if ``shared``) is the shared expert."""
    W_gu: np.ndarray  # [G, 2f, d]
    A_gu: np.ndarray  # [G, r, d]
    B_gu: np.ndarray  # [G, 2f, r]
    W_dn: np.ndarray  # [G, d, f]
    A_dn: np.ndarray  # [G, r, f]
    B_dn: np.ndarray  # [G, d, r]
    s: float          # alpha / r
    E: int            # routed experts
    shared: bool = False

    @classmethod
    def from_arrays(cls, arrays: dict, s: float, E: int, shared: bool = False):
        cv = {n: np.asarray(arrays[n], dtype=np.float64)
              for n in ("W_gu", "A_gu", "B_gu", "W_dn", "A_dn", "B_dn")}
        return cls(s=float(s), E=int(E), shared=bool(shared), **cv)

    @property
    def f(self):
        return self.W_dn.shape[2]


def expert_forward(x, P: OracleParams, g: int):
    """Rows x [n,d] through expert group g.  Returns every intermediate:
    xa = x A^T, h = x W^T + s xa B^T, act = silu(gate) * up,
    xa_dn = act A_dn^T, o = act W_dn^T + s xa_dn B_dn^T."""
    x = np.asarray(x, dtype=np.float64)
    f = P.f
    xa = x @ P.A_gu[g].T
    h = x @ P.W_gu[g].T + P.s * (xa @ P.B_gu[g].T)
    gate, up = h[:, :f], h[:, f:]
    act = silu(gate) * up
    xa_dn = act @ P.A_dn[g].T
    o = act @ P.W_dn[g].T + P.s * (xa_dn @ P.B_dn[g].T)
    return {"xa": xa, "h": h, "act": act, "xa_dn": xa_dn, "o": o}


def _assignments(ids, w, P: OracleParams):
    """(group, flat index list, token list, weight list) per expert group,
    built from the routing pass; the shared expert takes every token with
    weight 1 in token order."""
    ids = np.asarray(ids)
    T, k = ids.shape
    wf = np.asarray(w, dtype=np.float64).reshape(-1)
    rt = route(ids, P.E)
    groups = []
    for e in range(P.E):
        flat = rt["sorted_src"][rt["offsets"][e]:rt["offsets"][e + 1]]
        groups.append((e, flat, flat // k, wf[flat]))
    if P.shared:
        tok = np.arange(T)
        groups.append((P.E, None, tok, np.ones(T)))
    return groups


def layer_forward(X, ids, w, P: OracleParams):
    """Y [T,d] = sum_j w[t,j] * expert_{ids[t,j]}(X[t])  (+ shared expert)."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.zeros_like(X)
    for g, _flat, tok, wt in _assignments(ids, w, P):
        if tok.size == 0:
            continue
        fw = expert_forward(X[tok], P, g)
        np.add.at(Y, tok, wt[:, None] * fw["o"])
    return Y


def layer_backward(X, ids, w, dY, P: OracleParams, full: bool = False):
    """Gradients of L = sum(Y * dY) for frozen W and router.

    Returns dX [T,d], dw [T,k] (gradient w.r.t. the routing weights),
    dA_gu, dB_gu, dA_dn, dB_dn (shapes of the adapters, every group), and with
    full=True the full fine-tuning gradients of the expert weights too ([I]):
      dW_dn = dO^T act  [G,d,f];  dW_gu = dh^T x  [G,2f,d].
    Chain rule through the definitions of ``expert_forward``:
      dO = w dY_t;  dw = <dY_t, o>
      dB_dn = s dO^T xa_dn;  u = dO B_dn;  dA_dn = s u^T act
      dact = dO W_dn + s u A_dn
      dgate = dact * up * silu'(gate);  dup = dact * silu(gate);  dh = [dgate | dup]
      dB_gu = s dh^T xa;  v = dh B_gu;  dA_gu = s v^T x
      dx = dh W_gu + s v A_gu
    """
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    f = P.f
    dX = np.zeros_like(X)
    dw = np.zeros(T * k)
    names = ("A_gu", "B_gu", "A_dn", "B_dn") + (("W_gu", "W_dn") if full else ())
    grads = {n: np.zeros_like(getattr(P, n)) for n in names}
    for g, flat, tok, wt in _assignments(ids, w, P):
        if tok.size == 0:
            continue
        x = X[tok]
        fw = expert_forward(x, P, g)
        dyt = dY[tok]
        if flat is not None:
            dw[flat] = np.sum(dyt * fw["o"], axis=1)
        dO = wt[:, None] * dyt
        grads["B_dn"][g] = P.s * dO.T @ fw["xa_dn"]
        u = dO @ P.B_dn[g]
        grads["A_dn"][g] = P.s * u.T @ fw["act"]
        dact = dO @ P.W_dn[g] + P.s * (u @ P.A_dn[g])
        gate, up = fw["h"][:, :f], fw["h"][:, f:]
        dh = np.concatenate([dact * up * dsilu(gate), dact * silu(gate)], axis=1)
        grads["B_gu"][g] = P.s * dh.T @ fw["xa"]
        v = dh @ P.B_gu[g]
        grads["A_gu"][g] = P.s * v.T @ x
        if full:
            grads["W_dn"][g] = dO.T @ fw["act"]
            grads["W_gu"][g] = dh.T @ x
        dx = dh @ P.W_gu[g] + P.s * (v @ P.A_gu[g])
        np.add.at(dX, tok, dx)
    return {"dX": dX, "dw": dw.reshape(T, k),
            **{"d" + n: grads[n] for n in names}}


# ---------------------------------------------------------------------------
# PEFT-style merged evaluation ([L]: what split LoRA avoids) -- a pin
# ---------------------------------------------------------------------------

def merged_weights(P: OracleParams):
    """W' = W + s * B @ A for every group (materialises the delta)."""
    Wgu = P.W_gu + P.s * np.einsum("gor,gri->goi", P.B_gu, P.A_gu)
    Wdn = P.W_dn + P.s * np.einsum("gor,gri->goi", P.B_dn, P.A_dn)
    return Wgu, Wdn


def layer_forward_merged(X, ids, w, P: OracleParams):
    """Same layer evaluated with merged weights; equal to ``layer_forward``
    up to fp64 rounding by associativity ([L])."""
    X = np.asarray(X, dtype=np.float64)
    Wgu, Wdn = merged_weights(P)
    f = P.f
    Y = np.zeros_like(X)
    for g, _flat, tok, wt in _assignments(ids, w, P):
        if tok.size == 0:
            continue
        h = X[tok] @ Wgu[g].T
        o = (silu(h[:, :f]) * h[:, f:]) @ Wdn[g].T
        np.add.at(Y, tok, wt[:, None] * o)
    return Y


# ---------------------------------------------------------------------------
# Sampled evaluation for full-size checks: one token or one expert at a time
# ---------------------------------------------------------------------------

def _token_groups(t, ids, w, P):
    ids = np.asarray(ids)
    out = [(int(ids[t, j]), float(np.asarray(w)[t, j]), j) for j in range(ids.shape[1])]
    if P.shared:
        out.append((P.E, 1.0, None))
    return out


def token_forward(t: int, X, ids, w, P: OracleParams):
    """Y[t] alone: sum over the token's slots of w * expert(X[t])."""
    x = np.asarray(X[t], dtype=np.float64)[None, :]
    y = np.zeros(x.shape[1])
    for g, wt, _j in _token_groups(t, ids, w, P):
        y += wt * expert_forward(x, P, g)["o"][0]
    return y


def token_backward_dx(t: int, X, ids, w, dY, P: OracleParams):
    """dX[t] and dw[t,:] alone (the same chain rule as ``layer_backward``,
    restricted to token t's rows)."""
    x = np.asarray(X[t], dtype=np.float64)[None, :]
    dy = np.asarray(dY[t], dtype=np.float64)[None, :]
    f = P.f
    dx = np.zeros(x.shape[1])
    k = np.asarray(ids).shape[1]
    dw = np.zeros(k)
    for g, wt, j in _token_groups(t, ids, w, P):
        fw = expert_forward(x, P, g)
        if j is not None:
            dw[j] = float(np.sum(dy * fw["o"]))
        dO = wt * dy
        u = dO @ P.B_dn[g]
        dact = dO @ P.W_dn[g] + P.s * (u @ P.A_dn[g])
        gate, up = fw["h"][:, :f], fw["h"][:, f:]
        dh = np.concatenate([dact * up * dsilu(gate), dact * silu(gate)], axis=1)
        v = dh @ P.B_gu[g]
        dx += (dh @ P.W_gu[g] + P.s * (v @ P.A_gu[g]))[0]
    return dx, dw


def expert_lora_grads(g: int, X, ids, w, dY, P: OracleParams, full: bool = False):
    """dA_gu[g], dB_gu[g], dA_dn[g], dB_dn[g] alone: sums over the rows that
    group g receives (its routed rows, or every token for the shared expert);
    with full=True also dW_gu[g] and dW_dn[g]."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    f = P.f
    if g == P.E and P.shared:
        tok = np.arange(T)
        wt = np.ones(T)
    else:
        tt, jj = np.where(ids == g)
        tok = tt
        wt = np.asarray(w, dtype=np.float64)[tt, jj]
    out = {"dA_gu": np.zeros_like(P.A_gu[g]), "dB_gu": np.zeros_like(P.B_gu[g]),
           "dA_dn": np.zeros_like(P.A_dn[g]), "dB_dn": np.zeros_like(P.B_dn[g])}
    if full:
        out["dW_gu"] = np.zeros_like(P.W_gu[g])
        out["dW_dn"] = np.zeros_like(P.W_dn[g])
    if tok.size == 0:
        return out
    x = X[tok]
    fw = expert_forward(x, P, g)
    dO = wt[:, None] * dY[tok]
    out["dB_dn"] = P.s * dO.T @ fw["xa_dn"]
    u = dO @ P.B_dn[g]
    out["dA_dn"] = P.s * u.T @ fw["act"]
    dact = dO @ P.W_dn[g] + P.s * (u @ P.A_dn[g])
    gate, up = fw["h"][:, :f], fw["h"][:, f:]
    dh = np.concatenate([dact * up * dsilu(gate), dact * silu(gate)], axis=1)
    out["dB_gu"] = P.s * dh.T @ fw["xa"]
    out["dA_gu"] = P.s * (dh @ P.B_gu[g]).T @ x
    if full:
        out["dW_dn"] = dO.T @ fw["act"]
        out["dW_gu"] = dh.T @ x
    return out
