"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks return their error codes before anything is launched.  No
compute call runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from expert_routing_grouped_moe_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API [^(]*?\b(moe_\w+)\(", txt, flags=re.M)))


def test_header_declares_the_five_layer_calls():
    syms = declared_symbols()
    for s in ("moe_route", "moe_permute", "moe_lora_grouped_mlp_fwd",
              "moe_lora_grouped_mlp_bwd", "moe_unpermute_combine"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
    from expert_routing_grouped_moe_gb300 import _lib
    assert set(_lib.EXPORTED) == set(declared_symbols())


def test_sizes(lib):
    assert lib.moe_abi_version() == 1
    assert lib.moe_route_workspace_size(4096, 8, 128) >= 128 * 4
    assert lib.moe_route_workspace_size(0, 8, 128) == 0


def test_route_kernel_count(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    assert lib.moe_route_kernel_count(4096, 8, 128) == 2        # 32 chunks: scan fused
    assert lib.moe_route_kernel_count(1 << 20, 8, 128) == 3     # 2048 chunks
    assert lib.moe_route_kernel_count(0, 8, 128) == _lib.MOE_ERR_INVALID_ARG


def test_read_stream_probe_argument_checks(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    lin, til = _lib.MOE_PROBE_LINEAR, _lib.MOE_PROBE_TILES
    bad = _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_probe_read_stream(None, 1024, lin, None) == bad
    assert lib.moe_probe_read_stream(ctypes.c_void_p(4096 + 8), 1024, lin, None) == bad
    assert lib.moe_probe_read_stream(ctypes.c_void_p(4096), 0, lin, None) == bad
    assert lib.moe_probe_read_stream(ctypes.c_void_p(4096), 100, lin, None) == bad
    assert lib.moe_probe_read_stream(ctypes.c_void_p(4096), 1024, 2, None) == bad
    # tiles: whole 128-row blocks of a [rows, 2048] bf16 matrix (512 KiB each)
    assert lib.moe_probe_read_stream(ctypes.c_void_p(4096), 1 << 18, til, None) == bad


def _dims(**kw):
    from expert_routing_grouped_moe_gb300 import _lib
    base = dict(T=256, d=128, f=64, E=8, k=2, r=8, lora_scale=2.0, shared_expert=0)
    base.update(kw)
    return _lib.MoeDims(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9), -1), (dict(d=100), -1), (dict(r=12), -1), (dict(T=0), -1),
    (dict(shared_expert=2), -1), (dict(E=2000, k=2), -2), (dict(r=128), -2),
])
def test_bwd_workspace_rejects_bad_dims(lib, kw, code):
    from expert_routing_grouped_moe_gb300 import _lib
    d = _dims(**kw)
    assert lib.moe_mlp_bwd_workspace_size(ctypes.byref(d)) == 0


def test_fwd_argument_errors_before_launch(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: checks fail first
    d = _dims(k=9)
    rc = lib.moe_lora_grouped_mlp_fwd(ctypes.byref(d), None, *([fake] * 17), None)
    assert rc == _lib.MOE_ERR_INVALID_ARG
    assert b"k=9" in lib.moe_last_error()
    d = _dims()
    # at least one of Xp (permuted rows) and X (token rows)
    rc = lib.moe_lora_grouped_mlp_fwd(ctypes.byref(d), None, None, *([fake] * 16), None)
    assert rc == _lib.MOE_ERR_INVALID_ARG
    assert b"pass Xp" in lib.moe_last_error()
    args = [None] + [fake] * 17
    args[14] = P((1 << 20) + 4)  # Yp misaligned
    rc = lib.moe_lora_grouped_mlp_fwd(ctypes.byref(d), *args, None)
    assert rc == _lib.MOE_ERR_INVALID_ARG
    assert b"aligned" in lib.moe_last_error()
    args = [None] + [fake] * 17
    args[7] = None  # W_gu
    rc = lib.moe_lora_grouped_mlp_fwd(ctypes.byref(d), *args, None)
    assert rc == _lib.MOE_ERR_INVALID_ARG
    assert b"W_gu" in lib.moe_last_error()


def test_bwd_full_gradients_need_permuted_rows(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: checks fail first
    d = _dims()
    # dYp = NULL (gathered dY) with dW_gu requested: dYp, dY, Xp, X, then
    # counts .. dB_dn (21 pointers), dW_gu, dW_dn, ws
    args = [None, fake, fake, None] + [fake] * 21 + [fake, None] + [fake]
    rc = lib.moe_lora_grouped_mlp_bwd(ctypes.byref(d), *args, 1 << 40, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED
    assert b"permuted rows" in lib.moe_last_error()


def test_wait_selftest_argument_range(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    assert lib.moe_selftest_wait_timeout(0, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(2000001, None) == _lib.MOE_ERR_INVALID_ARG


def test_route_argument_errors_before_launch(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    assert lib.moe_route(None, 4, 2, 8, 0, *([fake] * 6), 1 << 20, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(fake, 4, 9, 8, 0, *([fake] * 6), 1 << 20, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(fake, 4, 2, 2048, 0, *([fake] * 6), 1 << 20, None) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_route(fake, 4, 2, 8, 0, *([fake] * 6), 4, None) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_route(fake, 4, 2, 8, 3, *([fake] * 6), 1 << 20, None) == _lib.MOE_ERR_INVALID_ARG


def test_rows_and_router_argument_errors(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    assert lib.moe_permute(fake, 4, 12, 2, fake, fake, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(fake, 4, 16, 2, None, fake, None) == _lib.MOE_ERR_INVALID_ARG
    # row_scalars without slot_out
    assert lib.moe_unpermute_combine(fake, fake, 4, 16, 2, 0, None, fake, None, fake,
                                     None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_unpermute_combine(fake, fake, 4, 16, 2, 2, None, None, None, fake,
                                     None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_router_topk(fake, 4, 8, 9, fake, fake, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_router_topk(fake, 4, 2048, 2, fake, fake, None) == _lib.MOE_ERR_UNSUPPORTED


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle and has no CPU compute path."""
    pkg = os.path.join(ROOT, "expert_routing_grouped_moe_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn


def test_route_and_route_noalloc_accept_the_same_shapes(lib):
    """Both routing entry points share one shape limit: a shape that
    moe_route refuses for its row count is refused by moe_route_noalloc too,
    before any device work (the checks fail before a pointer is used)."""
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    # E = 1, k = 1: the tile-rounded row count passes 2^31 while the routing
    # histogram (one group) stays far below the no-alloc array's 2 MiB
    T = (1 << 31) - 200
    assert lib.moe_route_workspace_size(T, 1, 1) <= (2 << 20)
    assert lib.moe_route(fake, T, 1, 1, 0, *([fake] * 6), 1 << 40, None) == \
        _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_noalloc(fake, T, 1, 1, 0, *([fake] * 5), None) == \
        _lib.MOE_ERR_UNSUPPORTED
    # just below the limit both accept the shape as far as the host checks go
    # (moe_route then fails only on its too-small workspace)
    T_ok = (1 << 31) - 256
    assert lib.moe_route(fake, T_ok, 1, 1, 0, *([fake] * 6), 4, None) == \
        _lib.MOE_ERR_WORKSPACE


def test_route_logits_checks_before_launch(lib):
    from expert_routing_grouped_moe_gb300 import _lib
    P = ctypes.c_void_p
    fake = P(1 << 20)
    # NULL logits, k > E, too small a workspace: refused before anything runs
    assert lib.moe_route_logits(None, 4, 8, 2, 0, *([fake] * 8), 1 << 20, None) == \
        _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route_logits(fake, 4, 8, 9, 0, *([fake] * 8), 1 << 20, None) == \
        _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route_logits(fake, 4, 8, 2, 0, *([fake] * 8), 4, None) == \
        _lib.MOE_ERR_WORKSPACE
