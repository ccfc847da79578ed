"""GPU parity of the prefill path (5 or more tokens: tcgen05 router GEMM,
top-k, bucketing, grouped gate/up and down GEMMs) against the oracle,
through the C ABI."""
import gc

import numpy as np
import pytest
import torch

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import (bf16_f64, check_topk, config_dict, h_tol, host_weights, make_layer_device,
                    make_layer_host, oracle_token, to_dev, to_host_bits, y_tol)

pytestmark = pytest.mark.gpu


def _check_layer_all_tokens(cfg, Ld, layer, x):
    """Full oracle on every token: ids, weights, bucketing and outputs."""
    T = x.shape[0]
    xd = to_dev(x)
    y = layer.forward(xd)
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    offs = np.zeros(cfg.n_experts + 1, np.int32)
    perm = np.zeros(T * cfg.top_k, np.int32)
    moe.moe_last_buckets(layer.handle, T, offs, perm)
    ids, w = layer.route(xd)
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    ids = ids.cpu().numpy()
    w = w.cpu().numpy()
    z = oracle.router_logits(Ld["router_w"], Ld["router_b"], x)
    adopt = [check_topk(ids[t], z[t], cfg.top_k) for t in range(T)]
    forced = ids if any(adopt) else None
    y_ref, _, w_ref, _ = oracle.moe_forward(Ld, cfg.top_k, x, forced_ids=forced)
    assert np.max(np.abs(w - w_ref)) < 1e-5
    # bucketing: bit-exact against the oracle's stable counting sort of the
    # GPU's own selection
    counts, offs_ref, pt_ref, _ = oracle.bucket(ids, cfg.n_experts)
    assert np.array_equal(offs, offs_ref)
    assert np.array_equal(perm, pt_ref)
    yg = bf16_f64(to_host_bits(y))
    err = np.max(np.abs(yg - y_ref))
    assert err <= y_tol(y_ref), (err, y_tol(y_ref))
    return y


@pytest.mark.parametrize("T", [5, 8, 17, 100, 300])
@pytest.mark.parametrize("permuted", [False, True])
def test_tiny_prefill(cuda_device, T, permuted):
    cfg = W.CONFIGS["tiny"].replace(permuted_slots=permuted)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=512)
    x = W.activations(cfg, 11, n_tokens=T)
    _check_layer_all_tokens(cfg, Ld, layer, x)
    layer.close()


def test_mid_shape_multi_tile_prefill(cuda_device):
    # several K steps, several 128-row M tiles, buckets larger than one
    # 128-token tile, experts that receive no token, and E not a multiple of 128
    cfg = W.MoEConfig("mid", 700, 1, 512, 40, 4, 256, 384, True, 1.1, 21, 21)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=1024)
    x = W.activations(cfg, 0)
    _check_layer_all_tokens(cfg, Ld, layer, x)
    layer.close()


def test_prefill_without_shared_expert_top1(cuda_device):
    cfg = W.MoEConfig("mid1", 260, 1, 256, 24, 1, 128, 0, False, 1.1, 22, 22)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=512)
    x = W.activations(cfg, 0)
    _check_layer_all_tokens(cfg, Ld, layer, x)
    layer.close()


def test_prefill_host_pointers_and_repeatability(cuda_device):
    cfg = W.CONFIGS["tiny"]
    layer, Ld = make_layer_host(cfg, 0, max_tokens=64)
    x = W.activations(cfg, 3, n_tokens=64)
    y_host = np.zeros_like(x)
    moe.moe_forward(layer.handle, x, 64, y_host)
    y_dev = to_host_bits(layer.forward(to_dev(x)))
    # fp32 reductions in L2 may add in any order: equal within one bf16 ulp
    a, b = bf16_f64(y_host), bf16_f64(y_dev)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-30)
    layer.close()


def test_prefill_stack_teacher_forced(cuda_device):
    cfg = W.CONFIGS["tiny"].replace(n_tokens=40)
    L = 3
    made = [make_layer_host(cfg, l, max_tokens=64) for l in range(L)]
    layers = [m[0] for m in made]
    x = W.activations(cfg, 4, n_tokens=40)
    y, h_trace, in_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
    assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
    h_trace, in_trace = to_host_bits(h_trace), to_host_bits(in_trace)
    ids_trace = ids_trace.cpu().numpy()
    h_prev = x
    for l in range(L):
        Ld = made[l][1]
        u = in_trace[l]
        u_ref = bf16_f64(oracle.rmsnorm(h_prev))
        assert np.all(np.abs(bf16_f64(u) - u_ref) <= 2.0 ** -7 * np.abs(u_ref) + 1e-30)
        z = oracle.router_logits(Ld["router_w"], Ld["router_b"], u)
        adopt = [check_topk(ids_trace[l, t], z[t], cfg.top_k) for t in range(40)]
        y_ref = oracle.moe_forward(Ld, cfg.top_k, u, forced_ids=ids_trace[l] if any(adopt) else None)[0]
        h_ref = bf16_f64(oracle.residual(h_prev, y_ref))
        assert np.max(np.abs(bf16_f64(h_trace[l]) - h_ref)) <= h_tol(y_ref, h_ref), l
        h_prev = h_trace[l]
    for l in layers:
        l.close()


def test_prefill125b_chunk_sampled_parity(cuda_device):
    """The full 8192-token chunk through one 125B-shaped layer: every
    token's top-k against the oracle's logits, the bucketing bit-exact, and
    a sample of tokens' outputs against the oracle computed token by token."""
    cfg = W.CONFIGS["prefill125b"]
    layer = make_layer_device(cfg, 0, max_tokens=cfg.n_tokens)
    try:
        x = W.activations(cfg, 0)
        xd = to_dev(x)
        y = to_host_bits(layer.forward(xd))
        assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
        # repeated runs agree up to the order of the fp32 combine reductions
        # (one bf16 rounding of each element, plus reordering noise): a
        # pipeline race that hands a buffer back early shows up here as
        # whole rows that differ
        y0 = bf16_f64(y)
        for _ in range(2):
            yr = bf16_f64(to_host_bits(layer.forward(xd)))
            assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
            bound = 2.0 ** -7 * np.abs(y0) + 1e-5 * np.abs(y0).max()
            assert np.all(np.abs(yr - y0) <= bound), float(np.max(np.abs(yr - y0)))
        ids, w = layer.route(xd)
        ids, w = ids.cpu().numpy(), w.cpu().numpy()
        offs = np.zeros(cfg.n_experts + 1, np.int32)
        perm = np.zeros(cfg.n_tokens * cfg.top_k, np.int32)
        moe.moe_last_buckets(layer.handle, cfg.n_tokens, offs, perm)
    finally:
        layer.close()
        gc.collect()
        torch.cuda.empty_cache()
    counts, offs_ref, pt_ref, _ = oracle.bucket(ids, cfg.n_experts)
    assert np.array_equal(offs, offs_ref) and np.array_equal(perm, pt_ref)
    # skew of the Zipf-biased router: bucket sizes from 0 to thousands
    assert counts.max() > 1000 and (counts == 0).sum() > 50
    Wr, b = W.router(cfg, 0)
    rng = np.random.default_rng(0)
    sample = np.concatenate([[0, 1, cfg.n_tokens - 1], rng.choice(cfg.n_tokens, 29, replace=False)])
    # top-k of a larger sample against the oracle's logits
    tk = np.sort(rng.choice(cfg.n_tokens, 512, replace=False))
    zs = oracle.router_logits(Wr, b, x[tk])
    for i, t in enumerate(tk):
        check_topk(ids[t], zs[i], cfg.top_k)
        assert abs(w[t].sum() - 1.0) < 1e-5
    sh = W.shared_expert(cfg, 0)
    cache = {}
    for t in sample:
        y_ref, _, _ = oracle_token(cfg, 0, x[t], gpu_ids=ids[t], router=(Wr, b), shared=sh,
                                   expert_cache=cache)
        err = np.max(np.abs(bf16_f64(y[t]) - y_ref))
        assert err <= y_tol(y_ref), (t, err, y_tol(y_ref))
    assert zs.shape[0] == 512
