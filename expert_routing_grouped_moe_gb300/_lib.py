"""ctypes binding of the C ABI in ``include/moe_gb300.h``.

Argument marshalling only: every function takes torch CUDA tensors (device
memory) and an optional ``torch.cuda.Stream`` and forwards raw pointers to
the library of the same name.  No arithmetic of the layer happens here.  If
the compiled library is missing the calls raise; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_gb300.so")
TILE_M = 128

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_BAD_IDS = -5
MOE_ERR_TIMEOUT = -6
MOE_PROBE_LINEAR = 0
MOE_PROBE_TILES = 1

EXPORTED = (
    "moe_router_topk", "moe_route_workspace_size", "moe_route",
    "moe_permute", "moe_unpermute_combine", "moe_lora_grouped_mlp_fwd",
    "moe_mlp_bwd_workspace_size", "moe_lora_grouped_mlp_bwd", "moe_status",
    "moe_last_error", "moe_abi_version", "moe_kernel_name", "moe_probe_arm", "moe_probe_count",
    "moe_route_noalloc", "moe_selftest_wait_timeout", "moe_probe_read_stream",
    "moe_route_kernel_count", "moe_ep_row_weights", "moe_ep_segment_ids", "moe_route_logits",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__("%s failed (%d): %s" % (where, code, msg))
        self.code = code


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("r", ctypes.c_int32),
                ("lora_scale", ctypes.c_float), ("shared_expert", ctypes.c_int32)]

    @property
    def G(self):
        return self.E + self.shared_expert

    @property
    def K(self):
        return self.k + self.shared_expert


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t


def load(path: str = LIB_PATH):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("MoE CUDA library not built (%s); run "
                               "expert_routing_grouped_moe_gb300.build.build()" % path)
        lib = ctypes.CDLL(path)
        sig = {
            "moe_router_topk": (ctypes.c_int, [_P, _I, _I, _I, _P, _P, _P]),
            "moe_route_workspace_size": (_SZ, [_I, _I, _I]),
            "moe_route": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
            "moe_permute": (ctypes.c_int, [_P, _I, _I, _I, _P, _P, _P]),
            "moe_unpermute_combine": (ctypes.c_int, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                                     _P]),
            "moe_lora_grouped_mlp_fwd": (ctypes.c_int, [ctypes.POINTER(MoeDims)] + [_P] * 19),
            "moe_mlp_bwd_workspace_size": (_SZ, [ctypes.POINTER(MoeDims)]),
            "moe_lora_grouped_mlp_bwd": (ctypes.c_int, [ctypes.POINTER(MoeDims)] + [_P] * 28
                                         + [_SZ, _P]),
            "moe_status": (ctypes.c_int, [_P]),
            "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, _P]),
            "moe_last_error": (ctypes.c_char_p, []),
            "moe_abi_version": (ctypes.c_int, []),
            "moe_kernel_name": (ctypes.c_char_p, [_I]),
            "moe_probe_arm": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(_P),
                                             ctypes.POINTER(_P), _I]),
            "moe_probe_count": (_I, [ctypes.c_char_p]),
            "moe_route_noalloc": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
            "moe_probe_read_stream": (ctypes.c_int, [_P, _SZ, _I, _P]),
            "moe_route_kernel_count": (_I, [_I, _I, _I]),
            "moe_ep_row_weights": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _P]),
            "moe_route_logits": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                                _P, _SZ, _P]),
            "moe_ep_segment_ids": (ctypes.c_int, [_P, _I, _I, ctypes.c_int64, _P, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int, where: str):
    if rc != MOE_OK:
        msg = load().moe_last_error().decode(errors="replace")
        raise MoeError(rc, where, msg)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _bf(t, name):
    return _ptr(t, torch.bfloat16, name)


def _i32(t, name):
    return _ptr(t, torch.int32, name)


def _f32(t, name):
    return _ptr(t, torch.float32, name)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_dims(T, d, f, E, k, r, lora_scale, shared_expert=False) -> MoeDims:
    return MoeDims(int(T), int(d), int(f), int(E), int(k), int(r), float(lora_scale),
                   1 if shared_expert else 0)


# ---------------------------------------------------------------- C ABI calls

def moe_router_topk(logits, k, ids, weights, stream=None):
    T, E = logits.shape
    _check(load().moe_router_topk(_f32(logits, "logits"), T, E, int(k), _i32(ids, "ids"),
                                  _f32(weights, "weights"), _stream(stream)), "moe_router_topk")


def moe_probe_read_stream(buf, pattern=0, stream=None):
    """Stream the bytes of a device tensor into shared memory (measurement);
    pattern MOE_PROBE_LINEAR or MOE_PROBE_TILES."""
    _check(load().moe_probe_read_stream(_ptr(buf, name="buf"), buf.numel() * buf.element_size(),
                                        int(pattern), _stream(stream)), "moe_probe_read_stream")


def moe_route_kernel_count(T, K, G) -> int:
    """Kernels moe_route launches for this shape (2 or 3)."""
    n = int(load().moe_route_kernel_count(int(T), int(K), int(G)))
    _check(n if n < 0 else MOE_OK, "moe_route_kernel_count")
    return n


def moe_route_workspace_size(T, K, G) -> int:
    return int(load().moe_route_workspace_size(int(T), int(K), int(G)))


def moe_route(ids, E, shared_expert, counts, offsets, tile_off, sorted_src, dest_pos, ws,
              stream=None):
    T, k = ids.shape
    _check(load().moe_route(_i32(ids, "ids"), T, k, int(E), 1 if shared_expert else 0,
                            _i32(counts, "counts"), _i32(offsets, "offsets"),
                            _i32(tile_off, "tile_off"), _i32(sorted_src, "sorted_src"),
                            _i32(dest_pos, "dest_pos"), _ptr(ws, name="ws"),
                            ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def moe_route_logits(logits, k, shared_expert, ids, weights, counts, offsets, tile_off,
                     sorted_src, dest_pos, ws, stream=None):
    """moe_router_topk then moe_route in one call (ids, weights written)."""
    T, E = logits.shape
    _check(load().moe_route_logits(
        _f32(logits, "logits"), T, E, int(k), 1 if shared_expert else 0, _i32(ids, "ids"),
        _f32(weights, "weights"), _i32(counts, "counts"), _i32(offsets, "offsets"),
        _i32(tile_off, "tile_off"), _i32(sorted_src, "sorted_src"), _i32(dest_pos, "dest_pos"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "moe_route_logits")


def moe_route_noalloc(ids, E, shared_expert, counts, offsets, tile_off, sorted_src, dest_pos,
                      stream=None):
    """moe_route with its scratch inside the library (no workspace argument)."""
    T, k = ids.shape
    _check(load().moe_route_noalloc(_i32(ids, "ids"), T, k, int(E), 1 if shared_expert else 0,
                                    _i32(counts, "counts"), _i32(offsets, "offsets"),
                                    _i32(tile_off, "tile_off"), _i32(sorted_src, "sorted_src"),
                                    _i32(dest_pos, "dest_pos"), _stream(stream)),
           "moe_route_noalloc")


def moe_permute(src, K, dest_pos, dst, stream=None):
    T, d = src.shape
    _check(load().moe_permute(_bf(src, "src"), T, d, int(K), _i32(dest_pos, "dest_pos"),
                              _bf(dst, "dst"), _stream(stream)), "moe_permute")


def moe_unpermute_combine(rows, dest_pos, k, shared_expert, out, weights=None, row_scalars=None,
                          slot_out=None, stream=None):
    T, d = out.shape
    _check(load().moe_unpermute_combine(
        _bf(rows, "rows"), _i32(dest_pos, "dest_pos"), T, d, int(k), 1 if shared_expert else 0,
        _f32(weights, "weights"), _f32(row_scalars, "row_scalars"), _f32(slot_out, "slot_out"),
        _bf(out, "out"), _stream(stream)), "moe_unpermute_combine")


def moe_lora_grouped_mlp_fwd(dims: MoeDims, Xp, X, counts, offsets, tile_off, sorted_src, topk_w,
                             W_gu, A_gu, B_gu, W_dn, A_dn, B_dn, Yp, h, act, xa_gu, xa_dn,
                             stream=None):
    """Pass the permuted rows Xp, or Xp=None and the token rows X (gathered)."""
    _check(load().moe_lora_grouped_mlp_fwd(
        ctypes.byref(dims), _bf(Xp, "Xp"), _bf(X, "X"), _i32(counts, "counts"),
        _i32(offsets, "offsets"),
        _i32(tile_off, "tile_off"), _i32(sorted_src, "sorted_src"), _f32(topk_w, "topk_w"),
        _bf(W_gu, "W_gu"), _bf(A_gu, "A_gu"), _bf(B_gu, "B_gu"), _bf(W_dn, "W_dn"),
        _bf(A_dn, "A_dn"), _bf(B_dn, "B_dn"), _bf(Yp, "Yp"), _f32(h, "h"), _bf(act, "act"),
        _bf(xa_gu, "xa_gu"), _bf(xa_dn, "xa_dn"), _stream(stream)), "moe_lora_grouped_mlp_fwd")


def moe_mlp_bwd_workspace_size(dims: MoeDims) -> int:
    return int(load().moe_mlp_bwd_workspace_size(ctypes.byref(dims)))


def moe_lora_grouped_mlp_bwd(dims: MoeDims, dYp, dY, Xp, X, counts, offsets, tile_off,
                             sorted_src, topk_w, W_gu, A_gu, B_gu, W_dn, A_dn, B_dn, h, act,
                             xa_gu, xa_dn, dXp, dw_rows, dA_gu, dB_gu, dA_dn, dB_dn, ws,
                             stream=None, dW_gu=None, dW_dn=None):
    """Pass permuted rows (dYp, Xp) or None and the token rows (dY, X).
    dW_gu [G,2f,d] / dW_dn [G,d,f] fp32: optional full weight gradients."""
    _check(load().moe_lora_grouped_mlp_bwd(
        ctypes.byref(dims), _bf(dYp, "dYp"), _bf(dY, "dY"), _bf(Xp, "Xp"), _bf(X, "X"),
        _i32(counts, "counts"),
        _i32(offsets, "offsets"), _i32(tile_off, "tile_off"), _i32(sorted_src, "sorted_src"),
        _f32(topk_w, "topk_w"), _bf(W_gu, "W_gu"), _bf(A_gu, "A_gu"), _bf(B_gu, "B_gu"),
        _bf(W_dn, "W_dn"), _bf(A_dn, "A_dn"), _bf(B_dn, "B_dn"), _f32(h, "h"), _bf(act, "act"),
        _bf(xa_gu, "xa_gu"), _bf(xa_dn, "xa_dn"), _bf(dXp, "dXp"), _f32(dw_rows, "dw_rows"),
        _f32(dA_gu, "dA_gu"), _f32(dB_gu, "dB_gu"), _f32(dA_dn, "dA_dn"), _f32(dB_dn, "dB_dn"),
        _f32(dW_gu, "dW_gu"), _f32(dW_dn, "dW_dn"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(), _stream(stream)),
        "moe_lora_grouped_mlp_bwd")


def moe_ep_row_weights(topk_w, dest_pos, shared_expert, row_w, stream=None):
    """row_w[dest_pos[t*K + j]] = topk_w[t, j] (1 for the shared slot)."""
    T, k = topk_w.shape
    _check(load().moe_ep_row_weights(_f32(topk_w, "topk_w"), _i32(dest_pos, "dest_pos"), T, k,
                                     1 if shared_expert else 0, _f32(row_w, "row_w"),
                                     _stream(stream)), "moe_ep_row_weights")


def moe_ep_segment_ids(counts, ids, stream=None):
    """ids[i] = local expert of received row i, for counts [P, E_loc]."""
    P, E_loc = counts.shape
    _check(load().moe_ep_segment_ids(_i32(counts, "counts"), P, E_loc, ids.numel(),
                                     _i32(ids, "ids") if ids.numel() else None, _stream(stream)),
           "moe_ep_segment_ids")


def moe_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load().moe_status(_stream(stream)))


def moe_selftest_wait_timeout(timeout_us: int, stream=None):
    """Enqueue the bounded-wait self-test: a GPU thread that waits on an
    mbarrier nothing arrives on for timeout_us, then records MOE_ERR_TIMEOUT
    (read it with moe_status)."""
    _check(load().moe_selftest_wait_timeout(int(timeout_us), _stream(stream)),
           "moe_selftest_wait_timeout")


# ------------------------------------------------------------------ tracing

def kernel_names():
    lib, out, i = load(), [], 0
    while True:
        n = lib.moe_kernel_name(i)
        if n is None:
            return out
        out.append(n.decode())
        i += 1


class KernelProbe:
    """Device time of the next ``n`` launches of one kernel, from CUDA events
    the library records on the launch stream (see moe_probe_arm)."""

    def __init__(self, kernel: str, n: int):
        self.kernel = kernel
        self.start = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        self.stop = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        s = torch.cuda.current_stream()
        for e in self.start + self.stop:   # materialise the event handles
            e.record(s)
        torch.cuda.synchronize()
        arr = _P * n
        self._a = arr(*[e.cuda_event for e in self.start])
        self._b = arr(*[e.cuda_event for e in self.stop])
        _check(load().moe_probe_arm(kernel.encode(), self._a, self._b, n), "moe_probe_arm")

    def disarm(self):
        load().moe_probe_arm(self.kernel.encode(), None, None, 0)

    def times_ms(self):
        """Durations (ms) of the recorded launches (synchronises)."""
        n = int(load().moe_probe_count(self.kernel.encode()))
        torch.cuda.synchronize()
        return [self.start[i].elapsed_time(self.stop[i]) for i in range(n)]
