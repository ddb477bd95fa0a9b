"""Python binding of the ft_moe C ABI (``include/ft_moe.h``): argument marshalling only.

Every step of the layer runs in the CUDA library ``libft_moe.so``; this module converts
Python ints and tensors (``data_ptr()``) to the C types and raises on error codes.  There is
no fallback: importing the binding without the built library, or calling it without a CUDA
device, raises.

Low-level functions carry the C names (``ft_moe_create``, ``ft_moe_forward``, ...); the
``MoELayerStack`` class wraps one handle.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libft_moe.so")

FT_OK, FT_ERR_INVALID, FT_ERR_STATE, FT_ERR_CUDA, FT_ERR_OOM, FT_ERR_CAPACITY, FT_ERR_TIMEOUT = range(7)
ERROR_NAMES = {0: "FT_OK", 1: "FT_ERR_INVALID", 2: "FT_ERR_STATE", 3: "FT_ERR_CUDA",
               4: "FT_ERR_OOM", 5: "FT_ERR_CAPACITY", 6: "FT_ERR_TIMEOUT"}

# every symbol include/ft_moe.h declares
EXPORTS = [
    "ft_last_error", "ft_moe_create", "ft_moe_destroy", "ft_moe_load_router",
    "ft_moe_set_router_bias", "ft_moe_load_pool", "ft_moe_load_shared", "ft_moe_forward",
    "ft_moe_decode_host", "ft_moe_prefill_stream", "ft_moe_prefill_bytes",
    "ft_moe_prefill_timing", "ft_cache_resize",
    "ft_cache_stats", "ft_cache_stats_reset", "ft_moe_status", "ft_moe_get_routing",
    "ft_moe_get_logits", "ft_moe_get_perm", "ft_moe_get_cache_state", "ft_moe_get_fills",
    "ft_moe_get_dims", "ft_moe_profile", "ft_moe_profile_read", "ft_moe_debug_set",
    "ft_route_topk_noalloc",
]

FT_WEIGHTS_BF16, FT_WEIGHTS_MXFP4 = 0, 1

PROF_CLASSES = ["router", "topk", "control", "fill", "gateup", "down", "other",
                "experts_hit", "experts_miss"]
FT_DEBUG_HOLD_FILLS, FT_DEBUG_WAIT_NS = 1, 2


class FtError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class ft_moe_opts(ctypes.Structure):
    _fields_ = [("n_shared", ctypes.c_int), ("prewarm", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("debug_checks", ctypes.c_int),
                ("prefill_topup", ctypes.c_int), ("admission", ctypes.c_int),
                ("weight_format", ctypes.c_int)]


class ft_cache_stats_t(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("fill_bytes", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("near_ties", ctypes.c_uint64),
                ("resizes", ctypes.c_uint64), ("tick", ctypes.c_uint64),
                ("bypasses", ctypes.c_uint64),
                ("n_slots", ctypes.c_int32), ("occupied", ctypes.c_int32),
                ("status", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libft_moe.so (raises if it is missing: build it with
    ``python -m expert_cached_routed_router_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with "
                          "`python -m expert_cached_routed_router_b300.build`")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "ft_last_error": (ctypes.c_char_p, []),
        "ft_moe_create": (I, [I, I, I, I, I, I, ctypes.POINTER(ft_moe_opts), ctypes.POINTER(P)]),
        "ft_moe_destroy": (None, [P]),
        "ft_moe_load_router": (I, [P, I, P, P]),
        "ft_moe_set_router_bias": (I, [P, I, P, P]),
        "ft_moe_load_pool": (I, [P, P, Z]),
        "ft_moe_load_shared": (I, [P, I, P]),
        "ft_moe_forward": (I, [P, I, P, I, P, P]),
        "ft_moe_decode_host": (I, [P, I, I, P, I, P, P]),
        "ft_moe_prefill_stream": (I, [P, I, I, P, I, P, P]),
        "ft_moe_prefill_bytes": (I, [P, ctypes.POINTER(ctypes.c_uint64),
                                     ctypes.POINTER(ctypes.c_uint64)]),
        "ft_moe_prefill_timing": (I, [P, ctypes.POINTER(ctypes.c_float),
                                      ctypes.POINTER(ctypes.c_float),
                                      ctypes.POINTER(ctypes.c_float)]),
        "ft_cache_resize": (I, [P, I]),
        "ft_cache_stats": (I, [P, ctypes.POINTER(ft_cache_stats_t)]),
        "ft_cache_stats_reset": (I, [P]),
        "ft_moe_status": (I, [P, ctypes.POINTER(I)]),
        "ft_moe_get_routing": (I, [P, P, P, P]),
        "ft_moe_get_logits": (I, [P, P]),
        "ft_moe_get_perm": (I, [P, P, P, P]),
        "ft_moe_get_cache_state": (I, [P, P, P, P, ctypes.POINTER(ctypes.c_uint64)]),
        "ft_moe_get_fills": (I, [P, ctypes.POINTER(ctypes.c_int32), P, I]),
        "ft_moe_get_dims": (I, [P, P]),
        "ft_moe_profile": (I, [P, I]),
        "ft_moe_profile_read": (I, [P, P, P, P]),
        "ft_moe_debug_set": (I, [P, I, ctypes.c_int64]),
        "ft_route_topk_noalloc": (I, [P, P, P, I, I, I, I, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int):
    if rc != FT_OK:
        raise FtError(rc, _lib.ft_last_error().decode())


def _ptr(t) -> int | None:
    """Address of a tensor / numpy array / int (None for None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# -------- functions with the C names (marshalling only) ----------------------------------

def ft_moe_create(L, E, k, d, d_ff, n_slots, n_shared=0, prewarm=1, max_tokens=4096,
                  debug_checks=0, prefill_topup=0, admission=0, weight_format=0) -> int:
    lib = load_library()
    opts = ft_moe_opts(n_shared, prewarm, max_tokens, debug_checks, prefill_topup, admission,
                       weight_format)
    h = ctypes.c_void_p()
    _check(lib.ft_moe_create(L, E, k, d, d_ff, n_slots, ctypes.byref(opts), ctypes.byref(h)))
    return h.value


def ft_moe_destroy(h):
    load_library().ft_moe_destroy(h)


def ft_moe_load_router(h, layer, wr, bias=None):
    _check(load_library().ft_moe_load_router(h, layer, _ptr(wr), _ptr(bias)))


def ft_moe_set_router_bias(h, layer, bias, stream=None):
    _check(load_library().ft_moe_set_router_bias(h, layer, _ptr(bias), _stream(stream)))


def ft_moe_load_pool(h, pool, nbytes):
    _check(load_library().ft_moe_load_pool(h, _ptr(pool), nbytes))


def ft_moe_load_shared(h, layer, entry):
    _check(load_library().ft_moe_load_shared(h, layer, _ptr(entry)))


def ft_moe_forward(h, layer, x, T, out, stream=None):
    _check(load_library().ft_moe_forward(h, layer, _ptr(x), T, _ptr(out), _stream(stream)))


def ft_moe_decode_host(h, layer0, n_layers, x_host, T, out_host, stream=None):
    _check(load_library().ft_moe_decode_host(h, layer0, n_layers, _ptr(x_host), T,
                                             _ptr(out_host), _stream(stream)))


def ft_moe_prefill_stream(h, layer0, n_layers, x, T, out, stream=None):
    _check(load_library().ft_moe_prefill_stream(h, layer0, n_layers, _ptr(x), T, _ptr(out),
                                                _stream(stream)))


def ft_moe_prefill_bytes(h):
    a, b = ctypes.c_uint64(), ctypes.c_uint64()
    _check(load_library().ft_moe_prefill_bytes(h, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def ft_moe_prefill_timing(h):
    c, k, w = ctypes.c_float(), ctypes.c_float(), ctypes.c_float()
    _check(load_library().ft_moe_prefill_timing(h, ctypes.byref(c), ctypes.byref(k),
                                                ctypes.byref(w)))
    return c.value, k.value, w.value


def ft_cache_resize(h, n_slots):
    _check(load_library().ft_cache_resize(h, n_slots))


def ft_cache_stats(h) -> dict:
    s = ft_cache_stats_t()
    _check(load_library().ft_cache_stats(h, ctypes.byref(s)))
    return s.as_dict()


def ft_cache_stats_reset(h):
    _check(load_library().ft_cache_stats_reset(h))


def ft_moe_status(h) -> int:
    v = ctypes.c_int()
    _check(load_library().ft_moe_status(h, ctypes.byref(v)))
    return v.value


def ft_moe_get_dims(h):
    import numpy as np
    dims = np.zeros(8, np.int32)
    _check(load_library().ft_moe_get_dims(h, dims.ctypes.data))
    return dict(zip(["L", "E", "k", "d", "d_ff", "n_slots", "max_tokens", "n_shared"],
                    (int(v) for v in dims)))


def ft_moe_get_routing(h, T, k):
    import numpy as np
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    tie = np.zeros(T, np.uint8)
    _check(load_library().ft_moe_get_routing(h, idx.ctypes.data, w.ctypes.data, tie.ctypes.data))
    return idx, w, tie


def ft_moe_get_logits(h, T, E):
    import numpy as np
    lg = np.zeros((T, E), np.float32)
    _check(load_library().ft_moe_get_logits(h, lg.ctypes.data))
    return lg


def ft_moe_get_perm(h, T, k, E):
    import numpy as np
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    _check(load_library().ft_moe_get_perm(h, counts.ctypes.data, offsets.ctypes.data,
                                          perm.ctypes.data))
    return counts, offsets, perm


def ft_moe_get_cache_state(h):
    import numpy as np
    dims = ft_moe_get_dims(h)
    table = np.zeros((dims["L"], dims["E"]), np.int32)
    owner = np.zeros(dims["n_slots"], np.int32)
    stamps = np.zeros(dims["n_slots"], np.uint64)
    tick = ctypes.c_uint64()
    _check(load_library().ft_moe_get_cache_state(h, table.ctypes.data, owner.ctypes.data,
                                                 stamps.ctypes.data, ctypes.byref(tick)))
    return table, owner, stamps, tick.value


def ft_moe_get_fills(h, cap=1024):
    import numpy as np
    n = ctypes.c_int32()
    fills = np.zeros((cap, 3), np.int32)
    _check(load_library().ft_moe_get_fills(h, ctypes.byref(n), fills.ctypes.data, cap))
    return fills[:min(n.value, cap)].copy()


def ft_moe_profile(h, enable):
    """enable: 0 off, 1 eager calls (True), 2 graph mode (events become graph nodes)."""
    _check(load_library().ft_moe_profile(h, int(enable)))


def ft_moe_profile_read(h) -> dict:
    """{class: (total ms, launches, expert entries processed)} since the last read."""
    import numpy as np
    ms = np.zeros(len(PROF_CLASSES), np.float64)
    n = np.zeros(len(PROF_CLASSES), np.int64)
    items = np.zeros(len(PROF_CLASSES), np.int64)
    _check(load_library().ft_moe_profile_read(h, ms.ctypes.data, n.ctypes.data,
                                              items.ctypes.data))
    return {c: (float(ms[i]), int(n[i]), int(items[i])) for i, c in enumerate(PROF_CLASSES)}


def ft_moe_debug_set(h, what, value):
    """Test hooks: FT_DEBUG_HOLD_FILLS (fills never reported done), FT_DEBUG_WAIT_NS."""
    _check(load_library().ft_moe_debug_set(h, what, int(value)))


def ft_route_topk_noalloc(x, wr, bias, T, E, d, k, idx, w, tie, stream=None):
    """Routing for callers that cannot allocate device memory: the caller passes every input
    and output as device memory; the library keeps its scratch in a fixed device array."""
    _check(load_library().ft_route_topk_noalloc(_ptr(x), _ptr(wr), _ptr(bias), T, E, d, k,
                                                _ptr(idx), _ptr(w), _ptr(tie),
                                                _stream(stream)))


class MoELayerStack:
    """One ft_moe handle: L routed-MoE layers sharing one LRU expert-slot cache."""

    def __init__(self, L, E, k, d, d_ff, n_slots, n_shared=0, prewarm=1, max_tokens=4096,
                 debug_checks=0, prefill_topup=0, admission=0, weight_format=0):
        self.L, self.E, self.k, self.d, self.d_ff = L, E, k, d, d_ff
        self.n_shared = n_shared
        self.entry_elems = 3 * d * d_ff
        self.weight_format = weight_format
        self.h = ft_moe_create(L, E, k, d, d_ff, n_slots, n_shared, prewarm, max_tokens,
                               debug_checks, prefill_topup, admission, weight_format)

    def close(self):
        if self.h:
            ft_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_router(self, layer, wr, bias=None):
        ft_moe_load_router(self.h, layer, wr, bias)

    def set_router_bias(self, layer, bias, stream=None):
        ft_moe_set_router_bias(self.h, layer, bias, stream)

    def load_pool(self, pool, nbytes):
        ft_moe_load_pool(self.h, pool, nbytes)

    def load_shared(self, layer, entry):
        ft_moe_load_shared(self.h, layer, entry)

    def forward(self, layer, x, out, stream=None):
        ft_moe_forward(self.h, layer, x, x.shape[0], out, stream)

    def decode_host(self, layer0, n_layers, x_host, out_host, stream=None):
        ft_moe_decode_host(self.h, layer0, n_layers, x_host, x_host.shape[0], out_host, stream)

    def prefill(self, layer0, n_layers, x, out, stream=None):
        ft_moe_prefill_stream(self.h, layer0, n_layers, x, x.shape[0], out, stream)

    def prefill_timing(self):
        return ft_moe_prefill_timing(self.h)

    def prefill_bytes(self):
        """(host -> device, slot -> buffer) bytes moved by the most recent prefill."""
        return ft_moe_prefill_bytes(self.h)

    def resize(self, n_slots):
        ft_cache_resize(self.h, n_slots)

    def stats(self):
        return ft_cache_stats(self.h)

    def stats_reset(self):
        ft_cache_stats_reset(self.h)

    def status(self):
        return ft_moe_status(self.h)

    def routing(self, T):
        return ft_moe_get_routing(self.h, T, self.k)

    def logits(self, T):
        return ft_moe_get_logits(self.h, T, self.E)

    def perm(self, T):
        return ft_moe_get_perm(self.h, T, self.k, self.E)

    def cache_state(self):
        return ft_moe_get_cache_state(self.h)

    def fills(self):
        return ft_moe_get_fills(self.h, cap=max(self.E, 1))

    def profile(self, enable):
        ft_moe_profile(self.h, enable)

    def profile_read(self):
        return ft_moe_profile_read(self.h)

    def debug_set(self, what, value):
        ft_moe_debug_set(self.h, what, value)
