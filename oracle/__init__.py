"""CPU oracle for the MoE-LoRA expert layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct NumPy (fp64) restatement of what the layer
computes, written from the pages' definitions.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path (the CUDA library and its Python binding) never
does, and this package imports nothing from the product path.

Pins (checked by ``tests/test_oracle_*.py`` on the CPU):

* ``route``            -- pinned: brute-force per-expert ``where`` loop, hand-worked
                          golden example, counting invariants.
* ``permute``, ``combine`` -- pinned: hand-worked golden example, the
                          round trip combine(permute(X)) = (sum of weights) X,
                          combine of per-row expert outputs = ``layer_forward``.
* ``router_topk``      -- pinned: brute-force sort on tiny inputs, hand-worked
                          golden example, softmax-over-selected identity.
* ``layer_forward``    -- pinned: merged-weight (PEFT) evaluation, hand-worked
                          1x1 SwiGLU golden example, B=0 and k=1 reductions,
                          linearity in the routing weights.
* ``layer_backward``   -- pinned: central finite differences of
                          L = sum(Y * dY) in fp64 for every gradient.
"""
from .moe_oracle import (  # noqa: F401
    router_topk,
    route,
    route_where_loop,
    permute,
    combine,
    silu,
    dsilu,
    OracleParams,
    expert_forward,
    layer_forward,
    layer_backward,
    merged_weights,
    layer_forward_merged,
    token_forward,
    token_backward_dx,
    expert_lora_grads,
)
