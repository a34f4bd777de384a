"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some hosts own all device memory through their own pool and give a library
only raw pointers and a stream, so the library cannot ask them for scratch.
moe_route_noalloc keeps its routing histogram in an array inside the library.
Its results must be the workspace-taking moe_route's, bit for bit (routing is
integer work), on consecutive calls that share that array.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from expert_routing_grouped_moe_gb300 import _lib as L, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_routing_grouped_moe_gb300 import build
    build.build()
    L.load()


def _outputs(T, k, E, shared):
    K, G = k + int(shared), E + int(shared)
    mk = lambda n: torch.full((n,), -9, dtype=torch.int32, device=DEV)  # noqa: E731
    return {"counts": mk(G), "offsets": mk(G + 1), "tile_off": mk(G + 1),
            "sorted_src": mk(T * K), "dest_pos": mk(T * K)}


def _route_with_ws(ids, E, shared):
    T, k = ids.shape
    o = _outputs(T, k, E, shared)
    ws = torch.empty(L.moe_route_workspace_size(T, k + int(shared), E + int(shared)),
                     dtype=torch.uint8, device=DEV)
    L.moe_route(ids, E, shared, o["counts"], o["offsets"], o["tile_off"], o["sorted_src"],
                o["dest_pos"], ws)
    return o


def _route_no_alloc(ids, E, shared):
    """Straight through the C ABI (ctypes), no workspace argument."""
    T, k = ids.shape
    o = _outputs(T, k, E, shared)
    lib = L.load()
    rc = lib.moe_route_noalloc(
        ctypes.c_void_p(ids.data_ptr()), T, k, E, int(shared),
        ctypes.c_void_p(o["counts"].data_ptr()), ctypes.c_void_p(o["offsets"].data_ptr()),
        ctypes.c_void_p(o["tile_off"].data_ptr()), ctypes.c_void_p(o["sorted_src"].data_ptr()),
        ctypes.c_void_p(o["dest_pos"].data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == L.MOE_OK, lib.moe_last_error()
    return o


@pytest.mark.parametrize("first,second", [
    ((4096, 128, 8, "uniform", False), (300, 5, 3, "zipf", True)),
    ((1 << 20, 128, 8, "zipf", False), (1 << 14, 64, 4, "uniform", True)),
])
def test_no_alloc_route_matches_route_twice_in_a_row(first, second):
    cases = []
    for (T, E, k, dist, shared), seed in ((first, 1), (second, 2)):
        ids = synth.topk_ids(T, E, k, dist, seed=seed, device=DEV)
        cases.append((ids, E, shared))
    got = [_route_no_alloc(*c) for c in cases]      # two calls sharing the array
    ref = [_route_with_ws(*c) for c in cases]
    torch.cuda.synchronize()
    assert L.moe_status() == L.MOE_OK
    for g, r in zip(got, ref):
        for key in r:
            assert torch.equal(g[key], r[key]), key


def test_no_alloc_route_rejects_too_large():
    T, k, E = 1 << 20, 8, 1024   # its histogram would need 4 MiB
    ids = torch.zeros(1, 1, dtype=torch.int32, device=DEV)
    lib = L.load()
    dummy = ctypes.c_void_p(ids.data_ptr())
    rc = lib.moe_route_noalloc(dummy, T, k, E, 0, dummy, dummy, dummy, dummy, dummy, None)
    assert rc == L.MOE_ERR_WORKSPACE
    assert b"2 MiB" in lib.moe_last_error()
