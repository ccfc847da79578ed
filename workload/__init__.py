"""Seeded synthetic workloads for the routed MoE FFN layer.

This module only draws inputs: expert weights (sigma*N(0,1), encoded as
symmetric 4-bit codes in blocks of 32 along K with one binary16 scale per
block), fp32 router weights, a Zipf(s) logit bias, expert-slot tables and
bf16 activations.  It holds none of the layer's arithmetic.  Both the CPU
oracle and the CUDA library consume its bytes; the host build (gen.c) and the
device build (gen_device.cu) are bit-identical by construction.

The workload shapes are those of the pages' MoE models: a 35B-A3B-shaped
stack (256 experts per layer, 8 active; "cyber-on-strata" page, two-tier
memory section) and a 125B-A6B-shaped stack (512 experts per layer x 48
layers = 24,576 experts, ~10 active; Strata/Project Maya page, MoE
architecture section), run as single-token decode, a 1+3-token MTP verify
batch ("nano-cuda-moe-qwen38" page, CPU/GPU async and speculative decoding
section) and an 8K-token prefill chunk (same page, prefill paragraph).
"""
from __future__ import annotations

import ctypes
import dataclasses
import fcntl
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "_gen_host.so")
_DEV_SO = os.path.join(_HERE, "_gen_device.so")

T_ROUTER, T_GATE, T_UP, T_DOWN, T_SH_GATE, T_SH_UP, T_SH_DOWN = 1, 2, 3, 4, 5, 6, 7
T_X, T_BIAS_PERM, T_SLOT_PERM, T_DRAFT = 8, 9, 10, 11
T_SH_GATE_W = 12  # gate vector of a gated shared expert


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One synthetic workload: layer shape, token count, stack depth, recipe."""

    name: str
    n_tokens: int  # T
    n_layers: int  # L
    hidden: int  # H
    n_experts: int  # E
    top_k: int  # k
    ffn: int  # F   (routed expert intermediate size)
    shared_ffn: int  # Fs  (0: no shared expert)
    permuted_slots: bool  # expert->slot table is a seeded permutation
    zipf_s: float  # 0: no router bias
    wset: int  # weight-set id; configs with equal wset share weights
    xset: int  # activation-set id
    draft_sigma: float = 0.0  # >0: tokens 1.. are token 0 + sigma*N(0,1)
    seed: int = 0
    weight_sigma: float = 0.02
    router_sigma: float = 0.02
    routing_flags: int = 0  # routing variant bits (1 no renorm, 2 bias selects only, 4 gated shared)

    @property
    def n_slots(self) -> int:
        return self.n_experts

    def expert_bytes(self, ffn: Optional[int] = None) -> int:
        """Packed bytes of one expert (gate+up+down codes and scales)."""
        f = self.ffn if ffn is None else ffn
        w = 3 * self.hidden * f
        return w // 2 + (w // 32) * 2

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# Calibrated draft noise for the MTP verify batch: the literal sigma = 0.1
# leaves the drafts' top-8 sets almost identical to token 0's (about 96 %
# overlap); sigma = 1.55 gives a mean overlap of 0.50 over 64 input sets.  It was
# chosen with workload/calibrate_draft_sigma.py, which routes with the oracle.
MTP_SIGMA_CALIBRATED = 1.55

CONFIGS = {
    "tiny": MoEConfig("tiny", 4, 1, 256, 16, 2, 128, 128, False, 0.0, 1, 1),
    "decode35b": MoEConfig("decode35b", 1, 40, 2048, 256, 8, 512, 512, False, 1.1, 2, 2),
    "mtp35b": MoEConfig("mtp35b", 4, 40, 2048, 256, 8, 512, 512, False, 1.1, 2, 3,
                        draft_sigma=MTP_SIGMA_CALIBRATED),
    "mtp35b_literal": MoEConfig("mtp35b_literal", 4, 40, 2048, 256, 8, 512, 512, False, 1.1,
                                2, 3, draft_sigma=0.1),
    "decode125b": MoEConfig("decode125b", 1, 48, 2048, 512, 10, 768, 1536, True, 1.1, 4, 4),
    "prefill125b": MoEConfig("prefill125b", 8192, 1, 2048, 512, 10, 768, 1536, True, 1.1, 4, 5),
    # the decode35b shape (first 8 layers, same weights and inputs) with every
    # routing variant on: no renormalisation, bias for selection only, gated
    # shared expert
    "decode35b_variants": MoEConfig("decode35b_variants", 1, 8, 2048, 256, 8, 512, 512, False,
                                    1.1, 2, 2, routing_flags=7),
}


# --------------------------------------------------------------------------- build

def _locked_build(target: str, cmd: list[str]) -> None:
    lock = target + ".lock"
    with open(lock, "w") as lf:
        fcntl.flock(lf, fcntl.LOCK_EX)
        try:
            srcs = [os.path.join(_HERE, f) for f in ("gen.c", "gen_device.cu", "gen_common.h")]
            newest = max(os.path.getmtime(s) for s in srcs)
            if os.path.exists(target) and os.path.getmtime(target) >= newest:
                return
            tmp = target + ".tmp%d" % os.getpid()
            subprocess.run(cmd + ["-o", tmp], check=True, cwd=_HERE)
            os.replace(tmp, target)
        finally:
            fcntl.flock(lf, fcntl.LOCK_UN)


def build_host() -> str:
    _locked_build(_HOST_SO, ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                             "-fno-fast-math", "-pthread", "gen.c"])
    return _HOST_SO


def build_device() -> str:
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    _locked_build(_DEV_SO, [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                            "-Xcompiler", "-fPIC", "-shared", "gen_device.cu"])
    return _DEV_SO


_host = None
_dev = None


def _hostlib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        u64, u32, i32, f32, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_void_p)
        lib.gen_quant_matrix.argtypes = [u64, u32, u32, u32, u32, i32, i32, f32, vp, vp, i32]
        lib.gen_dense_matrix.argtypes = [u64, u32, u32, u32, u32, i32, i32, f32, vp, vp, i32]
        lib.gen_permutation.argtypes = [u64, u32, u32, u32, i32, vp]
        lib.gen_zipf_bias.argtypes = [u64, u32, u32, i32, f32, vp]
        lib.gen_ln_f.argtypes = [f32]
        lib.gen_ln_f.restype = f32
        lib.gen_cossin_f.argtypes = [f32, vp, vp]
        lib.gen_normal_f.argtypes = [u64, u64]
        lib.gen_normal_f.restype = f32
        lib.gen_key_u64.argtypes = [u64, u32, u32, u32, u32]
        lib.gen_key_u64.restype = u64
        lib.gen_u64_at.argtypes = [u64, u64]
        lib.gen_u64_at.restype = u64
        for n in ("gen_f32_to_f16_array", "gen_f16_to_f32_array", "gen_f32_to_bf16_array"):
            getattr(lib, n).argtypes = [vp, vp, ctypes.c_int64]
        lib.gen_quant_block.argtypes = [vp, vp]
        lib.gen_quant_block.restype = ctypes.c_uint16
        _host = lib
    return _host


def _devlib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_device())
        u64, u32, i32, f32, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                                  ctypes.c_float, ctypes.c_void_p)
        lib.gen_dev_quant_experts.argtypes = [u64, u32, u32, u32, i32, vp, i32, i32, f32, vp, vp,
                                              vp]
        lib.gen_dev_dense.argtypes = [u64, u32, u32, u32, u32, ctypes.c_int64, f32, vp, vp, vp]
        _dev = lib
    return _dev


def _nthreads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------- host tensors

def quant_matrix(cfg: MoEConfig, layer: int, tensor: int, expert: int, rows: int, K: int):
    """Codes [rows][K/2] (uint8) and binary16 scale bits [rows][K/32] (uint16)."""
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 32), np.uint16)
    rc = _hostlib().gen_quant_matrix(cfg.seed, cfg.wset, layer, tensor, expert, rows, K,
                                     cfg.weight_sigma, _ptr(q), _ptr(s), _nthreads())
    assert rc == 0
    return q, s


def router(cfg: MoEConfig, layer: int):
    """Router weight fp32 [E][H] and bias fp32 [E] (zeros when zipf_s == 0)."""
    w = np.empty((cfg.n_experts, cfg.hidden), np.float32)
    rc = _hostlib().gen_dense_matrix(cfg.seed, cfg.wset, layer, T_ROUTER, 0, cfg.n_experts,
                                     cfg.hidden, cfg.router_sigma, _ptr(w), None, _nthreads())
    assert rc == 0
    b = np.zeros((cfg.n_experts,), np.float32)
    if cfg.zipf_s > 0:
        assert _hostlib().gen_zipf_bias(cfg.seed, cfg.wset, layer, cfg.n_experts, cfg.zipf_s,
                                        _ptr(b)) == 0
    return w, b


def shared_gate_vector(cfg: MoEConfig, layer: int) -> np.ndarray:
    """fp32 [H] gate vector of a gated shared expert, router_sigma * N(0,1)."""
    g = np.empty((1, cfg.hidden), np.float32)
    rc = _hostlib().gen_dense_matrix(cfg.seed, cfg.wset, layer, T_SH_GATE_W, 0, 1, cfg.hidden,
                                     cfg.router_sigma, _ptr(g), None, _nthreads())
    assert rc == 0
    return g.reshape(-1)


def slot_table(cfg: MoEConfig, layer: int) -> np.ndarray:
    """int32 [E]: slot of each logical expert (identity or seeded permutation)."""
    t = np.arange(cfg.n_experts, dtype=np.int32)
    if cfg.permuted_slots:
        assert _hostlib().gen_permutation(cfg.seed, cfg.wset, layer, T_SLOT_PERM,
                                          cfg.n_experts, _ptr(t)) == 0
    return t


def expert(cfg: MoEConfig, layer: int, e: int) -> dict:
    """Packed weights of logical expert e of a layer (canonical layout)."""
    H, F = cfg.hidden, cfg.ffn
    gq, gs = quant_matrix(cfg, layer, T_GATE, e, F, H)
    uq, us = quant_matrix(cfg, layer, T_UP, e, F, H)
    dq, ds = quant_matrix(cfg, layer, T_DOWN, e, H, F)
    return dict(gate_q=gq, gate_s=gs, up_q=uq, up_s=us, down_q=dq, down_s=ds)


def shared_expert(cfg: MoEConfig, layer: int) -> Optional[dict]:
    if cfg.shared_ffn == 0:
        return None
    H, Fs = cfg.hidden, cfg.shared_ffn
    gq, gs = quant_matrix(cfg, layer, T_SH_GATE, 0, Fs, H)
    uq, us = quant_matrix(cfg, layer, T_SH_UP, 0, Fs, H)
    dq, ds = quant_matrix(cfg, layer, T_SH_DOWN, 0, H, Fs)
    return dict(gate_q=gq, gate_s=gs, up_q=uq, up_s=us, down_q=dq, down_s=ds)


def layer(cfg: MoEConfig, layer_idx: int) -> dict:
    """Every tensor of one layer on the host, experts stored in slot order."""
    E, H, F = cfg.n_experts, cfg.hidden, cfg.ffn
    w, b = router(cfg, layer_idx)
    slots = slot_table(cfg, layer_idx)
    out = dict(router_w=w, router_b=b, slot_of_expert=slots)
    for name, rows, K in (("gate", F, H), ("up", F, H), ("down", H, F)):
        out[name + "_q"] = np.empty((E, rows, K // 2), np.uint8)
        out[name + "_s"] = np.empty((E, rows, K // 32), np.uint16)
    for e in range(E):
        ex = expert(cfg, layer_idx, e)
        s = slots[e]
        for k, v in ex.items():
            out[k][s] = v
    sh = shared_expert(cfg, layer_idx)
    if sh is not None:
        for k, v in sh.items():
            out["sh_" + k] = v
    if cfg.routing_flags & 4:
        out["sh_gate_w"] = shared_gate_vector(cfg, layer_idx)
    out["routing_flags"] = cfg.routing_flags
    return out


def activations(cfg: MoEConfig, index: int = 0, n_tokens: Optional[int] = None) -> np.ndarray:
    """bf16 bits [T][H] of input set `index`.  With draft_sigma > 0, token 0
    is N(0,1) and tokens 1.. are bf16(token0 + sigma*N(0,1))."""
    T = cfg.n_tokens if n_tokens is None else n_tokens
    H = cfg.hidden
    lib = _hostlib()
    if cfg.draft_sigma <= 0:
        x = np.empty((T, H), np.uint16)
        assert lib.gen_dense_matrix(cfg.seed, cfg.xset, index, T_X, 0, T, H, 1.0, None, _ptr(x),
                                    _nthreads()) == 0
        return x
    x0f = np.empty((1, H), np.float32)
    x0 = np.empty((1, H), np.uint16)
    assert lib.gen_dense_matrix(cfg.seed, cfg.xset, index, T_X, 0, 1, H, 1.0, _ptr(x0f),
                                _ptr(x0), 1) == 0
    x0_exact = bf16_bits_to_f32(x0)
    out = np.empty((T, H), np.uint16)
    out[0] = x0[0]
    if T > 1:
        noise = np.empty((T - 1, H), np.float32)
        assert lib.gen_dense_matrix(cfg.seed, cfg.xset, index, T_DRAFT, 0, T - 1, H,
                                    cfg.draft_sigma, _ptr(noise), None, _nthreads()) == 0
        xd = (x0_exact + noise).astype(np.float32)  # one fp32 add, round to nearest
        out[1:] = f32_to_bf16_bits(xd)
    return out


# --------------------------------------------------------------------------- conversions

def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _hostlib().gen_f32_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out


def f16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.uint16)
    out = np.empty(a.shape, np.float32)
    _hostlib().gen_f16_to_f32_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _hostlib().gen_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- device tensors

def device_layer(cfg: MoEConfig, layer_idx: int, device="cuda", stream=None) -> dict:
    """Every tensor of one layer generated directly in device memory (torch
    tensors, slot order).  Bytes equal `layer(cfg, layer_idx)`."""
    import torch

    lib = _devlib()
    E, H, F, Fs = cfg.n_experts, cfg.hidden, cfg.ffn, cfg.shared_ffn
    st = stream if stream is not None else torch.cuda.current_stream(device).cuda_stream
    w, b = router(cfg, layer_idx)  # small: drawn on the host
    slots = slot_table(cfg, layer_idx)
    out = dict(router_w=torch.from_numpy(w).to(device), router_b=torch.from_numpy(b).to(device),
               slot_of_expert=torch.from_numpy(slots).to(device))
    slots_d = out["slot_of_expert"]
    for name, tid, rows, K in (("gate", T_GATE, F, H), ("up", T_UP, F, H),
                               ("down", T_DOWN, H, F)):
        q = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=device)
        s = torch.empty((E, rows, K // 32), dtype=torch.int16, device=device)
        rc = lib.gen_dev_quant_experts(cfg.seed, cfg.wset, layer_idx, tid, E,
                                       slots_d.data_ptr(), rows, K, cfg.weight_sigma,
                                       q.data_ptr(), s.data_ptr(), st)
        assert rc == 0, rc
        out[name + "_q"], out[name + "_s"] = q, s
    if Fs:
        for name, tid, rows, K in (("sh_gate", T_SH_GATE, Fs, H), ("sh_up", T_SH_UP, Fs, H),
                                   ("sh_down", T_SH_DOWN, H, Fs)):
            q = torch.empty((rows, K // 2), dtype=torch.uint8, device=device)
            s = torch.empty((rows, K // 32), dtype=torch.int16, device=device)
            rc = lib.gen_dev_quant_experts(cfg.seed, cfg.wset, layer_idx, tid, 1, None, rows, K,
                                           cfg.weight_sigma, q.data_ptr(), s.data_ptr(), st)
            assert rc == 0, rc
            out[name + "_q"], out[name + "_s"] = q, s
    if cfg.routing_flags & 4:
        out["sh_gate_w"] = torch.from_numpy(shared_gate_vector(cfg, layer_idx)).to(device)
    return out
