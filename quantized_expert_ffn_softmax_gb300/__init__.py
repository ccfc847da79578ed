"""GB300 routed Mixture-of-Experts FFN layer with 4-bit block-quantized experts.

Thin ctypes binding of libmoe_gb300.so: the functions below carry the names
of the C ABI (include/moe.h) and only marshal arguments.  Every step of the
layer runs in the library's CUDA kernels; there is no Python or CPU fallback:
if the library is missing or fails to load, every call raises.

Pointer arguments accept torch tensors (device or host), numpy arrays (host)
or raw integer addresses.  ``stream`` accepts a torch.cuda.Stream, a raw
cudaStream_t integer, or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_CUDA = -2
MOE_ERR_OOM = -3
MOE_ERR_CAPACITY = -4
MOE_ERR_BOUNDS = -5
MOE_ERR_TIMEOUT = -6
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID", -2: "MOE_ERR_CUDA", -3: "MOE_ERR_OOM",
                -4: "MOE_ERR_CAPACITY", -5: "MOE_ERR_BOUNDS", -6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s (%d): %s" % (STATUS_NAMES.get(status, "?"), status, message))
        self.status = status


class moe_layer_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("shared_ffn", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("routing_flags", ctypes.c_int32)]


# routing variant bits of moe_layer_config.routing_flags (moe.h)
ROUTING_NO_RENORM = 1
ROUTING_BIAS_SELECT_ONLY = 2
ROUTING_SHARED_GATE = 4


WEIGHT_FIELDS = ("router_w", "router_bias", "slot_of_expert", "gate_q", "gate_s", "up_q", "up_s",
                 "down_q", "down_s", "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q",
                 "sh_down_s", "sh_gate_w", "expert_profile")


class moe_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


_lib = None


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_gb300.so is not built (run __graft_entry__.build()); "
                               "there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.moe_version.restype = i32
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_layer_create.argtypes = [ctypes.POINTER(moe_layer_config),
                                       ctypes.POINTER(moe_layer_weights), i32,
                                       ctypes.POINTER(vp)]
        L.moe_layer_create.restype = i32
        L.moe_layer_destroy.argtypes = [vp]
        L.moe_layer_destroy.restype = None
        L.moe_route.argtypes = [vp, vp, i32, vp, vp, vp]
        L.moe_route.restype = i32
        L.moe_forward.argtypes = [vp, vp, i32, vp, vp]
        L.moe_forward.restype = i32
        L.moe_stack_forward.argtypes = [ctypes.POINTER(vp), i32, vp, i32, vp, vp]
        L.moe_stack_forward.restype = i32
        L.moe_stack_forward_traced.argtypes = [ctypes.POINTER(vp), i32, vp, i32, vp, vp, vp, vp,
                                               vp, vp]
        L.moe_stack_forward_traced.restype = i32
        L.moe_forward_noalloc.argtypes = [ctypes.POINTER(moe_layer_config),
                                          ctypes.POINTER(moe_layer_weights), vp, i32, vp, vp, vp]
        L.moe_forward_noalloc.restype = i32
        L.moe_last_buckets.argtypes = [vp, i32, vp, vp, vp]
        L.moe_last_buckets.restype = i32
        L.moe_profile_enable.argtypes = [i32]
        L.moe_profile_enable.restype = i32
        L.moe_profile_read.argtypes = [ctypes.c_char_p, i32, vp, vp, i32]
        L.moe_profile_read.restype = i32
        L.moe_status_sync.argtypes = [vp, vp]
        L.moe_status_sync.restype = i32
        L.moe_cache_stats.argtypes = [vp, vp, vp, vp, i32, vp]
        L.moe_cache_stats.restype = i32
        _lib = L
    return _lib


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    raise TypeError("cannot take the address of %r" % type(a))


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, moe_last_error())


def moe_version() -> int:
    return lib().moe_version()


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def moe_layer_create(config: dict, weights: dict, weights_on_device: bool) -> int:
    """Creates a layer; returns its opaque handle (an integer address)."""
    cfg = moe_layer_config(config["hidden"], config["n_experts"], config["top_k"],
                           config["ffn"], config.get("shared_ffn", 0),
                           config.get("n_slots", config["n_experts"]), config["max_tokens"],
                           config.get("routing_flags", 0))
    w = moe_layer_weights(*[_ptr(weights.get(n)) for n in WEIGHT_FIELDS])
    out = ctypes.c_void_p()
    _check(lib().moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), int(bool(weights_on_device)),
                                  ctypes.byref(out)))
    return out.value


def _cfg_struct(config: dict) -> moe_layer_config:
    return moe_layer_config(config["hidden"], config["n_experts"], config["top_k"],
                            config["ffn"], config.get("shared_ffn", 0),
                            config.get("n_slots", config["n_experts"]),
                            config.get("max_tokens", 4), config.get("routing_flags", 0))


def moe_forward_noalloc(config: dict, weights: dict, x, n_tokens: int, y, status_out=None,
                        stream=None) -> None:
    """Allocation-free decode (1..4 tokens) from caller-owned device weights;
    scratch comes from the library's static device array."""
    cfg = _cfg_struct(config)
    w = moe_layer_weights(*[_ptr(weights.get(n)) for n in WEIGHT_FIELDS])
    _check(lib().moe_forward_noalloc(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), n_tokens,
                                     _ptr(y), _ptr(status_out), _stream(stream)))


def moe_layer_destroy(layer: int) -> None:
    lib().moe_layer_destroy(layer)


def moe_route(layer: int, x, n_tokens: int, topk_ids, topk_w, stream=None) -> None:
    _check(lib().moe_route(layer, _ptr(x), n_tokens, _ptr(topk_ids), _ptr(topk_w),
                           _stream(stream)))


def moe_forward(layer: int, x, n_tokens: int, y, stream=None) -> None:
    _check(lib().moe_forward(layer, _ptr(x), n_tokens, _ptr(y), _stream(stream)))


def _layer_array(layers):
    if isinstance(layers, ctypes.Array):
        return layers
    return (ctypes.c_void_p * len(layers))(*layers)


def layer_array(layers: Sequence[int]):
    """The layer handles of a stack as the C array moe_stack_forward takes;
    a caller that runs the same stack repeatedly can build it once."""
    return (ctypes.c_void_p * len(layers))(*layers)


def moe_stack_forward(layers: Sequence[int], n_layers: int, x, n_tokens: int, y,
                      stream=None) -> None:
    _check(lib().moe_stack_forward(_layer_array(layers), n_layers, _ptr(x), n_tokens, _ptr(y),
                                   _stream(stream)))


def moe_stack_forward_traced(layers: Sequence[int], n_layers: int, x, n_tokens: int, y, h_trace,
                             in_trace, y_trace, ids_trace, stream=None) -> None:
    _check(lib().moe_stack_forward_traced(_layer_array(layers), n_layers, _ptr(x), n_tokens,
                                          _ptr(y), _ptr(h_trace), _ptr(in_trace), _ptr(y_trace),
                                          _ptr(ids_trace), _stream(stream)))


def moe_last_buckets(layer: int, n_tokens: int, offsets, perm_token, stream=None) -> None:
    _check(lib().moe_last_buckets(layer, n_tokens, _ptr(offsets), _ptr(perm_token),
                                  _stream(stream)))


def moe_cache_stats(layer: int, reset: bool = False, stream=None):
    """(hits, misses) of a layer's expert cache; reset zeroes them after reading."""
    h = ctypes.c_uint64()
    m = ctypes.c_uint64()
    _check(lib().moe_cache_stats(layer, ctypes.byref(h), ctypes.byref(m), None, int(bool(reset)),
                                 _stream(stream)))
    return h.value, m.value


def moe_cache_slots(layer: int, n_experts: int, stream=None):
    """Current slot of every expert of a layer (-1: host tier only)."""
    import numpy as np

    tab = np.empty(n_experts, np.int32)
    _check(lib().moe_cache_stats(layer, None, None, tab.ctypes.data, 0, _stream(stream)))
    return tab


def moe_status_sync(layer: int, stream=None) -> int:
    """Synchronises and returns (and clears) the layer's device error word."""
    return lib().moe_status_sync(layer, _stream(stream))


def moe_profile_enable(enable: bool) -> None:
    _check(lib().moe_profile_enable(int(bool(enable))))


def moe_profile_read(max_entries: int = 64) -> dict:
    """{kernel name: (launch count, total ms)} since the last read."""
    import numpy as np

    name_len = 64
    names = ctypes.create_string_buffer(name_len * max_entries)
    counts = np.zeros(max_entries, np.int32)
    ms = np.zeros(max_entries, np.float32)
    n = lib().moe_profile_read(names, name_len, counts.ctypes.data, ms.ctypes.data, max_entries)
    raw = names.raw
    out = {}
    for i in range(n):
        nm = raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (int(counts[i]), float(ms[i]))
    return out


class MoELayer:
    """Owns one layer handle; convenience calls allocate outputs with torch."""

    def __init__(self, config: dict, weights: dict, weights_on_device: bool):
        self.config = dict(config)
        self.handle = moe_layer_create(config, weights, weights_on_device)

    def close(self):
        if getattr(self, "handle", None):
            moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, stream=None):
        import torch

        y = torch.empty_like(x)
        moe_forward(self.handle, x, x.shape[0], y, stream)
        return y

    def route(self, x, stream=None):
        import torch

        T, k = x.shape[0], self.config["top_k"]
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
        moe_route(self.handle, x, T, ids, w, stream)
        return ids, w


def stack_forward(layers: Sequence[MoELayer], x, stream=None, trace: bool = False):
    """Runs the pre-norm residual stack; with trace=True also returns each
    layer's h_{l+1}, normalised input u_l, output bf16(y_l) and top-k ids."""
    import torch

    y = torch.empty_like(x)
    hs = [l.handle for l in layers]
    if not trace:
        moe_stack_forward(hs, len(hs), x, x.shape[0], y, stream)
        return y
    L, T, H = len(hs), x.shape[0], x.shape[1]
    k = layers[0].config["top_k"]
    h_trace = torch.empty((L, T, H), dtype=x.dtype, device=x.device)
    in_trace = torch.empty((L, T, H), dtype=x.dtype, device=x.device)
    y_trace = torch.empty((L, T, H), dtype=x.dtype, device=x.device)
    ids = torch.empty((L, T, k), dtype=torch.int32, device=x.device)
    moe_stack_forward_traced(hs, L, x, T, y, h_trace, in_trace, y_trace, ids, stream)
    return y, h_trace, in_trace, y_trace, ids
