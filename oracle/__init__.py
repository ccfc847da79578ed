"""ORACLE -- test infrastructure only.

A plain, slow, fp64 CPU statement of the routed MoE FFN layer (oracle.c),
with ctypes marshalling.  Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of bench.py may import it.  It shares no code with the CUDA
library and imports nothing from it; its inputs come from the seeded
``workload`` generator.  See oracle.c for the readings it takes and the
page passages it follows.

Parity status of each function (what pins it, in tests/test_oracle_pins.py):
  dequant_row        round-trip bound against the generator's fp32 weights,
                     exact reconstruction of already-representable blocks
  router_logits      closed forms (one-hot inputs pick a router column)
  topk_softmax       brute-force rank selection; two-logit sigmoid closed
                     form; full-softmax-renormalised identity
  bucket             counting invariants, stability, brute-force grouping
  expert_ffn         hand-computed one-block example; dense numpy matmul
                     special case (top-1, weight 1, no shared expert)
  moe_forward        dense identity (k = E), slot-permutation invariance,
                     token independence, SwiGLU zero cases
  residual / stack   zero-expert identity; bf16 rounding vs torch
  rmsnorm            numpy RMS of the row; constant rows; power-of-two scale
                     invariance
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_oracle.so")
_lib = None


def build() -> str:
    """Compile oracle.c (plain C, fp64, no contraction) into _oracle.so."""
    src = os.path.join(_HERE, "oracle.c")
    with open(_SO + ".lock", "w") as lf:
        fcntl.flock(lf, fcntl.LOCK_EX)
        try:
            if not (os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src)):
                tmp = _SO + ".tmp%d" % os.getpid()
                subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                                "-fno-fast-math", src, "-lm", "-o", tmp], check=True)
                os.replace(tmp, _SO)
        finally:
            fcntl.flock(lf, fcntl.LOCK_UN)
    return _SO


class OracleLayer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("ffn", ctypes.c_int), ("shared_ffn", ctypes.c_int), ("n_slots", ctypes.c_int)] + [
        (n, ctypes.c_void_p) for n in (
            "router_w", "router_b", "slot_of_expert", "gate_q", "gate_s", "up_q", "up_s",
            "down_q", "down_s", "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q",
            "sh_down_s")] + [("routing_flags", ctypes.c_int), ("sh_gate_w", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i32, i64, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_double.restype = d
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = d
        L.oracle_double_to_bf16.argtypes = [d]
        L.oracle_double_to_bf16.restype = ctypes.c_uint16
        L.oracle_round_bf16.argtypes = [vp, vp, i64]
        L.oracle_silu.argtypes = [d]
        L.oracle_silu.restype = d
        L.oracle_dequant_row.argtypes = [vp, vp, i32, vp]
        L.oracle_router_logits.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.oracle_topk_softmax.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.oracle_topk_softmax_full.argtypes = [i32, i32, i32, vp, vp, vp]
        L.oracle_route_weights.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_shared_gate.argtypes = [i32, vp, vp]
        L.oracle_shared_gate.restype = d
        L.oracle_bucket.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_expert_ffn.argtypes = [i32, i32] + [vp] * 8
        L.oracle_combine_token.argtypes = [i32, i32, i32, i32] + [vp] * 15
        L.oracle_moe_forward.argtypes = [ctypes.POINTER(OracleLayer), i32, vp, vp, vp, vp, vp, vp]
        L.oracle_moe_forward.restype = i32
        L.oracle_residual.argtypes = [vp, vp, vp, i64]
        L.oracle_rmsnorm.argtypes = [vp, i32, i32, d, vp]
        L.oracle_stack_forward.argtypes = [ctypes.POINTER(OracleLayer), i32, i32, vp, vp, vp, vp]
        L.oracle_stack_forward.restype = i32
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


# ------------------------------------------------------------------ scalars

def half_to_double(bits) -> float:
    return lib().oracle_half_to_double(int(bits))


def round_bf16(y) -> np.ndarray:
    y = _c(y, np.float64)
    out = np.empty(y.shape, np.uint16)
    lib().oracle_round_bf16(_p(y), _p(out), y.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(g: float) -> float:
    return lib().oracle_silu(float(g))


# ------------------------------------------------------------------ steps

def dequant_row(q, s) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint16)
    K = q.size * 2
    out = np.empty(K, np.float64)
    lib().oracle_dequant_row(_p(q), _p(s), K, _p(out))
    return out


def dequant_matrix(q, s) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint16)
    return np.stack([dequant_row(q[r], s[r]) for r in range(q.shape[0])])


def router_logits(W, b, x_bf16) -> np.ndarray:
    W = _c(W, np.float32)
    x = _c(x_bf16, np.uint16)
    E, H = W.shape
    T = x.shape[0]
    b = None if b is None else _c(b, np.float32)
    z = np.empty((T, E), np.float64)
    lib().oracle_router_logits(T, H, E, _p(W), _p(b), _p(x), _p(z))
    return z


def topk_softmax(z, k):
    z = _c(z, np.float64)
    T, E = z.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    margin = np.empty((T,), np.float64)
    lib().oracle_topk_softmax(T, E, k, _p(z), _p(ids), _p(w), _p(margin))
    return ids, w, margin


def topk_softmax_full(z, k):
    z = _c(z, np.float64)
    T, E = z.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_topk_softmax_full(T, E, k, _p(z), _p(ids), _p(w))
    return ids, w


def route_weights(zsel, b, ids, flags: int) -> np.ndarray:
    """Routing weights [T][k] of the selection ids under the variant flags
    (1: no renormalisation, 2: bias for selection only); zsel = W_r x + b."""
    zsel = _c(zsel, np.float64)
    T, E = zsel.shape
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    bb = None if b is None else _c(b, np.float32)
    w = np.empty((T, k), np.float64)
    lib().oracle_route_weights(T, E, k, int(flags), _p(zsel), _p(bb), _p(ids), _p(w))
    return w


def shared_gate(g, x_bf16) -> float:
    """sigmoid(g . x) for one token (g fp32 [H], x bf16 bits [H])."""
    g = _c(g, np.float32)
    x = _c(x_bf16, np.uint16).reshape(-1)
    return float(lib().oracle_shared_gate(x.size, _p(g), _p(x)))


def bucket(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pt = np.empty(T * k, np.int32)
    pj = np.empty(T * k, np.int32)
    lib().oracle_bucket(T, k, E, _p(ids), _p(counts), _p(offsets), _p(pt), _p(pj))
    return counts, offsets, pt, pj


def expert_ffn(ex: dict, x) -> np.ndarray:
    """y[H] for fp64 x[H] through one expert (dict of *_q / *_s arrays)."""
    x = _c(x, np.float64)
    H = x.size
    F = ex["gate_q"].shape[0]
    arrs = [_c(ex[n], t) for n, t in (("gate_q", np.uint8), ("gate_s", np.uint16),
                                       ("up_q", np.uint8), ("up_s", np.uint16),
                                       ("down_q", np.uint8), ("down_s", np.uint16))]
    y = np.empty(H, np.float64)
    lib().oracle_expert_ffn(H, F, *[_p(a) for a in arrs], _p(x), _p(y))
    return y


def combine_token(experts: list, w, shared, x_bf16) -> np.ndarray:
    """One token: sum_j w[j] FFN(experts[j]) + FFN(shared); x is bf16 bits [H]."""
    x = _c(x_bf16, np.uint16).reshape(-1)
    H = x.size
    k = len(experts)
    F = experts[0]["gate_q"].shape[0] if k else 32
    keep = []

    def arr(name, t):
        a = [_c(e[name], t) for e in experts]
        keep.append(a)
        return (ctypes.c_void_p * max(1, k))(*[_p(v) for v in a])

    ptrs = [arr("gate_q", np.uint8), arr("gate_s", np.uint16), arr("up_q", np.uint8),
            arr("up_s", np.uint16), arr("down_q", np.uint8), arr("down_s", np.uint16)]
    if shared is not None:
        sh = [_c(shared[n], t) for n, t in (("gate_q", np.uint8), ("gate_s", np.uint16),
                                             ("up_q", np.uint8), ("up_s", np.uint16),
                                             ("down_q", np.uint8), ("down_s", np.uint16))]
        Fs = sh[0].shape[0]
        shp = [_p(a) for a in sh]
    else:
        Fs, shp, sh = 0, [None] * 6, None
    w = _c(w, np.float64)
    y = np.empty(H, np.float64)
    lib().oracle_combine_token(H, F, Fs, k, _p(w), *[ctypes.cast(p, ctypes.c_void_p) for p in ptrs],
                               *shp, _p(x), _p(y))
    return y


def _layer_struct(Ld: dict, top_k: int):
    keep = {}

    def g(name, t):
        if name not in Ld or Ld[name] is None:
            return None
        a = _c(Ld[name], t)
        keep[name] = a
        return _p(a)

    E, H = Ld["router_w"].shape
    F = Ld["gate_q"].shape[1]
    Fs = Ld["sh_gate_q"].shape[0] if Ld.get("sh_gate_q") is not None else 0
    st = OracleLayer(H, E, top_k, F, Fs, Ld["gate_q"].shape[0],
                     g("router_w", np.float32), g("router_b", np.float32),
                     g("slot_of_expert", np.int32),
                     g("gate_q", np.uint8), g("gate_s", np.uint16), g("up_q", np.uint8),
                     g("up_s", np.uint16), g("down_q", np.uint8), g("down_s", np.uint16),
                     g("sh_gate_q", np.uint8), g("sh_gate_s", np.uint16), g("sh_up_q", np.uint8),
                     g("sh_up_s", np.uint16), g("sh_down_q", np.uint8), g("sh_down_s", np.uint16),
                     int(Ld.get("routing_flags", 0)), g("sh_gate_w", np.float32))
    return st, keep


def moe_forward(Ld: dict, top_k: int, x_bf16, forced_ids=None):
    """Whole layer (weights in slot order): returns y fp64 [T][H], ids [T][k],
    routing weights fp64 [T][k] and top-k margins [T]."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    st, keep = _layer_struct(Ld, top_k)
    y = np.empty((T, H), np.float64)
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float64)
    m = np.empty((T,), np.float64)
    f = None if forced_ids is None else _c(forced_ids, np.int32)
    rc = lib().oracle_moe_forward(ctypes.byref(st), T, _p(x), _p(f), _p(y), _p(ids), _p(w), _p(m))
    if rc != 0:
        raise ValueError("oracle_moe_forward failed: %d" % rc)
    return y, ids, w, m


def residual(h_bf16, y) -> np.ndarray:
    h = _c(h_bf16, np.uint16)
    y = _c(y, np.float64)
    out = np.empty(h.shape, np.uint16)
    lib().oracle_residual(_p(h), _p(y), _p(out), h.size)
    return out


def rmsnorm(h_bf16, eps: float = 1e-6) -> np.ndarray:
    """Unit-gain RMS normalisation of each row, rounded once to bf16."""
    h = _c(h_bf16, np.uint16)
    T, H = h.shape
    out = np.empty(h.shape, np.uint16)
    lib().oracle_rmsnorm(_p(h), T, H, float(eps), _p(out))
    return out


def stack_forward(layers: list, top_k: int, x_bf16):
    """Pre-norm residual stack over in-memory layers: h_L, h trace, id trace."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    structs, keeps = zip(*[_layer_struct(Ld, top_k) for Ld in layers])
    arr = (OracleLayer * len(layers))(*structs)
    out = np.empty((T, H), np.uint16)
    trace = np.empty((len(layers), T, H), np.uint16)
    ids = np.empty((len(layers), T, top_k), np.int32)
    rc = lib().oracle_stack_forward(arr, len(layers), T, _p(x), _p(out), _p(trace), _p(ids))
    if rc != 0:
        raise ValueError("oracle_stack_forward failed: %d" % rc)
    return out, trace, ids
