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
    # the first call's histogram fills the 2 MiB array exactly (256 experts,
    # 8,388,608 routed rows); the second reuses a small corner of it
    ((1 << 20, 256, 8, "uniform", False), (1000, 16, 2, "zipf", False)),
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


def test_no_alloc_route_at_the_limit_is_exactly_2_mib():
    assert L.moe_route_workspace_size(1 << 20, 8, 256) == 2 << 20
    assert L.moe_route_workspace_size(1 << 20, 8, 257) > 2 << 20


def test_no_alloc_route_bad_id_through_the_shared_array():
    """An id outside [0, E) is reported through the status word and its slot
    gets dest_pos -1, exactly as moe_route does; the next call is clean."""
    T, k, E = 64, 2, 8
    ids = synth.topk_ids(T, E, k, "uniform", seed=5, device=DEV)
    bad = ids.clone()
    bad[17, 1] = E + 3
    assert L.moe_status() == L.MOE_OK
    got = _route_no_alloc(bad, E, False)
    assert L.moe_status() == L.MOE_ERR_BAD_IDS
    ref = _route_with_ws(bad, E, False)
    assert L.moe_status() == L.MOE_ERR_BAD_IDS
    assert int(got["dest_pos"][17 * k + 1]) == -1
    for key in ref:
        assert torch.equal(got[key], ref[key]), key
    assert int(got["counts"].sum()) == T * k - 1
    clean = _route_no_alloc(ids, E, False)
    assert L.moe_status() == L.MOE_OK
    ref2 = _route_with_ws(ids, E, False)
    for key in ref2:
        assert torch.equal(clean[key], ref2[key]), key


def test_no_alloc_route_rejects_too_large():
    T, k, E = 1 << 20, 8, 1024   # its histogram would need 8 MiB
    ids = torch.zeros(1, 1, dtype=torch.int32, device=DEV)
    lib = L.load()
    dummy = ctypes.c_void_p(ids.data_ptr())
    rc = lib.moe_route_noalloc(dummy, T, k, E, 0, dummy, dummy, dummy, dummy, dummy, None)
    assert rc == L.MOE_ERR_WORKSPACE
    assert b"2 MiB" in lib.moe_last_error()
