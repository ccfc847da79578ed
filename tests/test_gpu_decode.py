"""GPU parity of the decode / MTP-verify path (1..4 tokens) against the oracle,
through the C ABI, on the seeded workloads: the tiny layer, the 40-layer
35B-A3B-shaped stack (1 token and the 1+3-token verify batch) and the
48-layer 125B-A6B-shaped stack with permuted slot tables."""
import gc
import os

import numpy as np
import pytest
import torch

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import (bf16_f64, check_stack_outputs, check_topk, make_layer_device,
                    make_layer_host, oracle_token, parallel_map, to_dev, to_host_bits, y_tol)

pytestmark = pytest.mark.gpu


def _tiny(permuted=True, **kw):
    return W.CONFIGS["tiny"].replace(permuted_slots=permuted, **kw)


# ----------------------------------------------------------------- generator

def test_generator_device_bytes_equal_host_bytes(cuda_device):
    cfg = _tiny()
    host = W.layer(cfg, 0)
    dev = W.device_layer(cfg, 0)
    torch.cuda.synchronize()
    for k, v in dev.items():
        d = v.cpu().numpy()
        h = host[k]
        if d.dtype == np.int16:
            d = d.view(np.uint16)
        assert np.array_equal(d.reshape(h.shape), h), k
    # a few experts of a full-size layer
    big = W.CONFIGS["decode125b"]
    dq = W.device_layer(big, 3)
    slots = W.slot_table(big, 3)
    for e in (0, 77, 511):
        ex = W.expert(big, 3, e)
        s = slots[e]
        for n in ("gate_q", "up_s", "down_q", "down_s"):
            d = dq[n][s].cpu().numpy()
            if d.dtype == np.int16:
                d = d.view(np.uint16)
            assert np.array_equal(d, ex[n]), (e, n)
    del dq
    torch.cuda.empty_cache()


# ----------------------------------------------------------------- tiny layer

@pytest.mark.parametrize("permuted", [False, True])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_tiny_forward_and_route(cuda_device, permuted, T):
    cfg = _tiny(permuted)
    layer, Ld = make_layer_host(cfg, 0)
    for idx in range(3):
        x = W.activations(cfg, idx, n_tokens=T)
        xd = to_dev(x)
        y = layer.forward(xd)
        ids, w = layer.route(xd)
        assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
        ids = ids.cpu().numpy()
        w = w.cpu().numpy()
        z = oracle.router_logits(Ld["router_w"], Ld["router_b"], x)
        adopt = [check_topk(ids[t], z[t], cfg.top_k) for t in range(T)]
        forced = ids if any(adopt) else None
        y_ref, ids_ref, w_ref, _ = oracle.moe_forward(Ld, cfg.top_k, x, forced_ids=forced)
        assert np.max(np.abs(w - w_ref)) < 1e-5
        assert np.allclose(w.sum(1), 1.0, atol=1e-5)
        yg = bf16_f64(to_host_bits(y))
        assert np.max(np.abs(yg - y_ref)) <= y_tol(y_ref)
    layer.close()


def test_tiny_host_pointers_match_device_pointers(cuda_device):
    cfg = _tiny()
    layer, Ld = make_layer_host(cfg, 0)
    x = W.activations(cfg, 5)
    y_dev = to_host_bits(layer.forward(to_dev(x)))
    y_host = np.zeros_like(x)
    moe.moe_forward(layer.handle, x, x.shape[0], y_host)
    # the two runs' fp32 reductions may add in another order: one bf16
    # rounding apart at most
    a, b = bf16_f64(y_host), bf16_f64(y_dev)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-30)
    ids = np.zeros((x.shape[0], cfg.top_k), np.int32)
    w = np.zeros((x.shape[0], cfg.top_k), np.float32)
    moe.moe_route(layer.handle, x, x.shape[0], ids, w)
    ids_d, w_d = layer.route(to_dev(x))
    assert np.array_equal(ids, ids_d.cpu().numpy()) and np.array_equal(w, w_d.cpu().numpy())
    layer.close()


def test_tiny_pinned_host_buffers_read_and_written_in_place(cuda_device):
    """Decode-sized calls read a pinned host x and write a pinned host y
    through their device addresses (no staging copies); the results equal the
    device-pointer calls up to the order of the fp32 reductions (one bf16
    rounding per layer), for a layer, a stack, and a stack with x == y."""
    cfg = _tiny()
    L = 3
    made = [make_layer_host(cfg, l) for l in range(L)]
    layers = [m[0] for m in made]
    hs = [l.handle for l in layers]
    x = W.activations(cfg, 6)
    T = x.shape[0]

    def close(a_bits, b_bits, layers=1):
        # one bf16 rounding per layer (the fp32 reductions add in a
        # run-dependent order, and a stack feeds each layer's rounding into
        # the next layer's input), plus one rounding of the largest element
        # for entries the residual sum brings near zero
        a, b = bf16_f64(a_bits), bf16_f64(b_bits)
        bound = layers * 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b))
        if layers > 1:
            bound = bound + 2.0 ** -7 * np.abs(b).max()
        ok = np.all(np.abs(a - b) <= bound + 1e-30)
        if not ok:
            i = np.unravel_index(np.argmax(np.abs(a - b) - bound), a.shape)
            print("worst", i, a[i], b[i], bound[i], "max|b|", np.abs(b).max())
        return ok

    xp = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
    yp = torch.zeros_like(xp).pin_memory()
    y_dev = to_host_bits(layers[0].forward(to_dev(x)))
    moe.moe_forward(hs[0], xp, T, yp)  # returns after y is written
    assert close(yp.numpy().view(np.uint16), y_dev)
    yd = to_dev(np.zeros_like(x))
    moe.moe_stack_forward(hs, L, to_dev(x), T, yd)
    ys_dev = to_host_bits(yd)
    yp.zero_()
    moe.moe_stack_forward(hs, L, xp, T, yp)
    assert close(yp.numpy().view(np.uint16), ys_dev, L)
    moe.moe_stack_forward(hs, L, xp, T, xp)  # in place: x == y
    assert close(xp.numpy().view(np.uint16), ys_dev, L)
    for l in layers:
        l.close()


def test_tiny_no_shared_expert_and_top1(cuda_device):
    cfg = _tiny(shared_ffn=0, top_k=1)
    layer, Ld = make_layer_host(cfg, 0)
    x = W.activations(cfg, 1)
    y = bf16_f64(to_host_bits(layer.forward(to_dev(x))))
    y_ref = oracle.moe_forward(Ld, 1, x)[0]
    assert np.max(np.abs(y - y_ref)) <= y_tol(y_ref)
    layer.close()


def check_norm(u_gpu, h_in):
    """The GPU's normalised layer input equals the oracle's RMS norm of the
    same h within one bf16 unit in the last place per element."""
    u_ref = bf16_f64(oracle.rmsnorm(h_in))
    ug = bf16_f64(u_gpu)
    assert np.all(np.abs(ug - u_ref) <= 2.0 ** -7 * np.abs(u_ref) + 1e-30)


def test_tiny_stack_teacher_forced(cuda_device):
    cfg = _tiny()
    L = 5
    made = [make_layer_host(cfg, l) for l in range(L)]
    layers = [m[0] for m in made]
    x = W.activations(cfg, 2)
    y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
    assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
    h_trace, in_trace, y_trace = to_host_bits(h_trace), to_host_bits(in_trace), to_host_bits(y_trace)
    ids_trace = ids_trace.cpu().numpy()
    assert np.array_equal(to_host_bits(y), h_trace[-1])
    h_prev = x
    for l in range(L):
        Ld = made[l][1]
        u = in_trace[l]
        check_norm(u, h_prev)
        z = oracle.router_logits(Ld["router_w"], Ld["router_b"], u)
        adopt = [check_topk(ids_trace[l, t], z[t], cfg.top_k) for t in range(cfg.n_tokens)]
        y_ref = oracle.moe_forward(Ld, cfg.top_k, u,
                                   forced_ids=ids_trace[l] if any(adopt) else None)[0]
        check_stack_outputs(h_prev, y_trace[l], h_trace[l], y_ref, where=l)
        h_prev = h_trace[l]
    # in place: x == y is allowed for stacks
    xd = to_dev(x)
    moe.moe_stack_forward([l.handle for l in layers], L, xd, cfg.n_tokens, xd)
    assert np.array_equal(to_host_bits(xd), h_trace[-1])
    for l in layers:
        l.close()


def test_errors_and_timeout_status(cuda_device):
    cfg = _tiny()
    layer, Ld = make_layer_host(cfg, 0, max_tokens=4)
    x = to_dev(W.activations(cfg, 0))
    y = torch.empty_like(x)
    for bad_T in (0, 5, -1):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_forward(layer.handle, x, bad_T, y)
        assert ei.value.status == moe.MOE_ERR_CAPACITY
    with pytest.raises(moe.MoeError):
        moe.moe_forward(layer.handle, x, 4, x)  # aliasing
    # a bad slot table is rejected at create
    w = dict(Ld)
    bad = Ld["slot_of_expert"].copy()
    bad[3] = bad[4]
    from parity import host_weights, config_dict
    hw = host_weights(Ld)
    hw["slot_of_expert"] = bad
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_create(config_dict(cfg, 4), hw, False)
    assert ei.value.status == moe.MOE_ERR_INVALID
    # bounded device wait: a barrier that can never fill must time out,
    # record MOE_ERR_TIMEOUT and leave the context usable
    os.environ["MOE_DEBUG_UNREACHABLE_BARRIER"] = "1"
    os.environ["MOE_WAIT_TIMEOUT_US"] = "20000"
    try:
        moe.moe_forward(layer.handle, x, 4, y)
        st = moe.moe_status_sync(layer.handle)
    finally:
        del os.environ["MOE_DEBUG_UNREACHABLE_BARRIER"]
        del os.environ["MOE_WAIT_TIMEOUT_US"]
    assert st == moe.MOE_ERR_TIMEOUT
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK  # cleared
    y2 = layer.forward(x)
    y_ref = oracle.moe_forward(Ld, cfg.top_k, W.activations(cfg, 0))[0]
    assert np.max(np.abs(bf16_f64(to_host_bits(y2)) - y_ref)) <= y_tol(y_ref)
    layer.close()


# ----------------------------------------------------------------- full-size stacks

def _stack_check(cfg, input_index=0):
    """Runs the full stack (device-generated weights) once with traces and
    checks EVERY layer with teacher forcing (the oracle takes the GPU's bf16
    input of that layer): the RMS norm, every token's top-k, every token's
    layer output y_l at the stated tolerance
    max|y_gpu - y_ref| <= 1e-2 max|y_ref| + 1e-3, and every element of the
    residual h_{l+1}.  Layers are checked concurrently on host threads."""
    layers = [make_layer_device(cfg, l, max_tokens=8) for l in range(cfg.n_layers)]
    try:
        x = W.activations(cfg, input_index)
        y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
        assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
        h_trace, in_trace = to_host_bits(h_trace), to_host_bits(in_trace)
        y_trace = to_host_bits(y_trace)
        ids_trace = ids_trace.cpu().numpy()
        assert np.array_equal(to_host_bits(y), h_trace[-1])
    finally:
        for l in layers:
            l.close()
        del layers
        gc.collect()
        torch.cuda.empty_cache()
    assert np.all(np.isfinite(bf16_f64(h_trace[-1])))
    T = cfg.n_tokens
    h_in = [x] + [h_trace[l] for l in range(cfg.n_layers - 1)]

    def check_layer(l):
        u = in_trace[l]
        check_norm(u, h_in[l])
        Wr, b = W.router(cfg, l)
        sh = W.shared_expert(cfg, l)
        cache = {}
        y_ref = np.empty((T, cfg.hidden), np.float64)
        adopted = 0
        for t in range(T):
            y_ref[t], _, a = oracle_token(cfg, l, u[t], gpu_ids=ids_trace[l, t], router=(Wr, b),
                                          shared=sh, expert_cache=cache)
            adopted += a
        worst = check_stack_outputs(h_in[l], y_trace[l], h_trace[l], y_ref, where=l)
        return adopted, worst

    res = parallel_map(check_layer, range(cfg.n_layers))
    n_adopted = sum(r[0] for r in res)
    worst = max(r[1] for r in res)
    return ids_trace, n_adopted, worst


def test_decode35b_stack_parity(cuda_device):
    cfg = W.CONFIGS["decode35b"]
    _, _, worst = _stack_check(cfg)
    print("decode35b: worst y error / tolerance over 40 layers = %.3f" % worst)


def test_mtp35b_verify_batch_parity(cuda_device):
    cfg = W.CONFIGS["mtp35b"]
    ids, _, worst = _stack_check(cfg)
    print("mtp35b: worst y error / tolerance over 40 layers x 4 tokens = %.3f" % worst)
    # the calibrated drafts overlap token 0's selection by about one half
    ov = [len(set(ids[0, 0]) & set(ids[0, t])) / cfg.top_k for t in range(1, 4)]
    assert 0.2 <= np.mean(ov) <= 0.85


def test_decode125b_stack_parity(cuda_device):
    cfg = W.CONFIGS["decode125b"]
    _, _, worst = _stack_check(cfg)
    print("decode125b: worst y error / tolerance over 48 layers = %.3f" % worst)
