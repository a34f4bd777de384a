"""Shared helpers for the parity tests (no layer arithmetic here)."""
import os

import numpy as np
import torch

# bf16 outputs and gradients: relative Frobenius error and elementwise bound
REL_FRO = 5e-3
ELEM_ABS = 2e-2


def assert_close_bf16(got, ref, name, rel_fro=REL_FRO, elem=ELEM_ABS):
    """rel-Frobenius <= 5e-3 and |got - ref| <= 2e-2 * (1 + |ref|) elementwise."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    nref = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    rf = err / nref if nref > 0 else err
    bound = elem * (1.0 + np.abs(ref))
    over = np.abs(got - ref) > bound
    worst = float(np.max(np.abs(got - ref) / bound)) if got.size else 0.0
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write("%-28s relF %.3e  worst/bound %.3f  n=%d\n" % (name, rf, worst, got.size))
    assert rf <= rel_fro, "%s: rel-Frobenius %.3e > %.1e" % (name, rf, rel_fro)
    assert not over.any(), "%s: %d elements over the elementwise bound (worst %.2fx)" % (
        name, int(over.sum()), worst)
    return rf


def to64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def oracle_params(weights: dict, cfg, groups=None):
    """fp64 oracle parameters from bf16 device weights; with ``groups`` only
    those groups are filled (the others stay zero, never touched)."""
    import oracle
    arrs = {}
    for n, t in weights.items():
        if groups is None:
            arrs[n] = to64(t)
        else:
            a = np.zeros(tuple(t.shape), dtype=np.float64)
            for g in groups:
                a[g] = to64(t[g])
            arrs[n] = a
    return oracle.OracleParams.from_arrays(arrs, s=cfg.scale, E=cfg.E, shared=cfg.shared)
