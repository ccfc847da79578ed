"""Helpers of the GPU parity tests: build library layers from the seeded
workloads, run the oracle on the same bytes, and apply the parity rule:

* top-k ids equal the oracle's bit for bit, except where the oracle's logits
  are within 1e-4 (the k-th/(k+1)-th margin, or adjacent entries for order);
  there the oracle adopts the GPU's ids for the output check;
* outputs: max|y_gpu - y_ref| <= 1e-2 * max|y_ref| + 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W

TIE_MARGIN = 1e-4
NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def y_tol(y_ref) -> float:
    return 1e-2 * float(np.abs(y_ref).max()) + 1e-3


def h_tol_elem(y_ref, h_ref, tol_y: float) -> np.ndarray:
    """Per-element bound on a stack output h = bf16(h_in + bf16(y)) when the
    GPU's y is within tol_y of y_ref (same bf16 h_in on both sides): the
    difference in y, plus half a bf16 unit in the last place (2^-8 relative)
    for each of the four roundings -- bf16(y) and the bf16 sum on either side
    --, which is at most 2^-7 * (|y| + |h|) up to terms in tol_y."""
    return tol_y * (1.0 + 2.0 ** -7) + 2.0 ** -7 * (np.abs(y_ref) + np.abs(h_ref))


def check_stack_outputs(h_in, y_gpu, h_gpu, y_ref, where=""):
    """One stack layer, teacher-forced: every token's y (bf16 bits from the
    GPU's trace) against the oracle's y_ref (fp64, computed from the GPU's
    normalised input) at the stated tolerance, and every element of the
    residual h_{l+1} = bf16(h_l + bf16(y)) against the oracle's residual of
    the GPU's own h_l.  Returns the worst y error over its tolerance."""
    worst = 0.0
    for t in range(y_ref.shape[0]):
        tol = y_tol(y_ref[t])
        err = float(np.max(np.abs(bf16_f64(y_gpu[t]) - y_ref[t])))
        assert err <= tol, ("y", where, t, err, tol)
        worst = max(worst, err / tol)
        h_ref = bf16_f64(oracle.residual(h_in[t][None, :], y_ref[t][None, :]))[0]
        dh = np.abs(bf16_f64(h_gpu[t]) - h_ref)
        bound = h_tol_elem(y_ref[t], h_ref, tol)
        assert np.all(dh <= bound), ("h", where, t, float(np.max(dh - bound)))
    return worst


def parallel_map(fn, items, workers: int = 0):
    """fn over items on a thread pool (the oracle and the generator are C
    calls that release the GIL); results in item order."""
    import concurrent.futures as cf
    import os

    n = workers or max(1, min(16, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(fn, items))


def config_dict(cfg: W.MoEConfig, max_tokens: int) -> dict:
    return dict(hidden=cfg.hidden, n_experts=cfg.n_experts, top_k=cfg.top_k, ffn=cfg.ffn,
                shared_ffn=cfg.shared_ffn, max_tokens=max_tokens, routing_flags=cfg.routing_flags)


def host_weights(Ld: dict) -> dict:
    w = {n: Ld[n] for n in ("router_w", "slot_of_expert") + NAMES}
    w["router_bias"] = Ld["router_b"]
    if "sh_gate_q" in Ld:
        for n in NAMES:
            w["sh_" + n] = Ld["sh_" + n]
    if "sh_gate_w" in Ld:
        w["sh_gate_w"] = Ld["sh_gate_w"]
    return w


def make_layer_host(cfg, layer_idx, max_tokens=16):
    Ld = W.layer(cfg, layer_idx)
    return moe.MoELayer(config_dict(cfg, max_tokens), host_weights(Ld), False), Ld


def make_layer_device(cfg, layer_idx, max_tokens=16):
    Dd = W.device_layer(cfg, layer_idx)
    w = {n: Dd[n] for n in ("router_w", "slot_of_expert") + NAMES}
    w["router_bias"] = Dd["router_b"]
    if cfg.shared_ffn:
        for n in NAMES:
            w["sh_" + n] = Dd["sh_" + n]
    if "sh_gate_w" in Dd:
        w["sh_gate_w"] = Dd["sh_gate_w"]
    torch.cuda.synchronize()
    layer = moe.MoELayer(config_dict(cfg, max_tokens), w, True)
    del Dd, w
    return layer


def to_dev(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def bf16_f64(bits) -> np.ndarray:
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def check_topk(gpu_ids: np.ndarray, z: np.ndarray, k: int) -> np.ndarray:
    """Asserts the parity rule for one token's ids against oracle logits z
    [E]; returns True when the GPU's ids differ from the oracle's (so the
    output check must adopt them)."""
    ids_o, _, _ = oracle.topk_softmax(z[None, :], k)
    ids_o = ids_o[0]
    g = np.asarray(gpu_ids, dtype=np.int64)
    assert len(set(g.tolist())) == k, "duplicate ids %s" % g
    assert np.all((g >= 0) & (g < z.size)), "id out of range %s" % g
    if np.array_equal(g, ids_o):
        return False
    zs = np.sort(z)[::-1]
    for j in range(k):
        assert abs(z[g[j]] - zs[j]) < TIE_MARGIN, (
            "top-k mismatch beyond the tie margin at position %d: gpu %s oracle %s" % (j, g, ids_o))
    return True


def oracle_token(cfg, layer_idx: int, x_row: np.ndarray, gpu_ids=None, router=None,
                 shared=None, expert_cache=None):
    """Oracle of one token through one layer, experts fetched from the host
    generator.  Returns (y fp64 [H], oracle ids, adopted flag)."""
    Wr, b = router if router is not None else W.router(cfg, layer_idx)
    z = oracle.router_logits(Wr, b, x_row[None, :])[0]
    ids, w, _ = oracle.topk_softmax(z[None, :], cfg.top_k)
    ids, w = ids[0], w[0]
    adopted = False
    if gpu_ids is not None:
        adopted = check_topk(gpu_ids, z, cfg.top_k)
        if adopted:
            ids = np.asarray(gpu_ids, np.int32)
            zz = z[ids]
            e = np.exp(zz - zz.max())
            w = e / e.sum()
    exs = []
    for e_id in ids:
        key = (layer_idx, int(e_id))
        if expert_cache is not None and key in expert_cache:
            exs.append(expert_cache[key])
        else:
            ex = W.expert(cfg, layer_idx, int(e_id))
            if expert_cache is not None:
                expert_cache[key] = ex
            exs.append(ex)
    sh = shared if shared is not None else W.shared_expert(cfg, layer_idx)
    y = oracle.combine_token(exs, w, sh, x_row)
    return y, ids, adopted
