"""The allocation-free decode entry point (moe_forward_noalloc), checked
through the C ABI against moe_forward on the same weights and inputs.

It exists for callers that cannot allocate device memory when they run a
layer (graph capture into a pool they do not own, plug-ins under a host
framework's allocator, fixed post-start-up memory budgets): its scratch is a
static 128 KiB device array inside the library.  This file is collected
last."""
import numpy as np
import pytest
import torch

import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import bf16_f64, config_dict, to_dev, to_host_bits, y_tol

pytestmark = pytest.mark.gpu

NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def _device_weights(cfg, layer_idx):
    D = W.device_layer(cfg, layer_idx)
    w = {n: D[n] for n in ("router_w", "slot_of_expert") + NAMES}
    w["router_bias"] = D["router_b"]
    if cfg.shared_ffn:
        for n in NAMES:
            w["sh_" + n] = D["sh_" + n]
    torch.cuda.synchronize()
    return w


@pytest.mark.parametrize("name", ["decode35b", "tiny"])
def test_noalloc_matches_moe_forward_on_consecutive_calls(cuda_device, name):
    cfg = W.CONFIGS[name].replace(permuted_slots=True)
    w = _device_weights(cfg, 0)
    config = config_dict(cfg, 8)
    layer = moe.MoELayer(config, w, True)
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    try:
        # 1..4 tokens (3 runs in the 4-token instantiation with a padded slot)
        for T in (1, 2, 3, 4):
            for call in range(2):  # two calls in a row share the static scratch
                x = to_dev(W.activations(cfg, 40 + 2 * T + call, n_tokens=T))
                y_ref = bf16_f64(to_host_bits(layer.forward(x)))
                y = torch.empty_like(x)
                moe.moe_forward_noalloc(config, w, x, T, y, status)
                torch.cuda.synchronize()
                assert int(status.item()) == moe.MOE_OK
                err = np.max(np.abs(bf16_f64(to_host_bits(y)) - y_ref))
                assert err <= y_tol(y_ref), (T, call, err)
        assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    finally:
        layer.close()
        del w
        torch.cuda.empty_cache()


def test_noalloc_gated_shared_expert_without_renormalisation(cuda_device):
    # reads the caller's shared-gate vector; compared with moe_forward on the
    # same weights
    flags = moe.ROUTING_SHARED_GATE | moe.ROUTING_NO_RENORM
    cfg = W.CONFIGS["tiny"].replace(permuted_slots=True, zipf_s=1.1, routing_flags=flags)
    w = _device_weights(cfg, 0)
    w["sh_gate_w"] = torch.from_numpy(W.shared_gate_vector(cfg, 0)).cuda()
    config = config_dict(cfg, 8)
    layer = moe.MoELayer(config, w, True)
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    try:
        for T in (1, 3):
            x = to_dev(W.activations(cfg, 60 + T, n_tokens=T))
            y_ref = bf16_f64(to_host_bits(layer.forward(x)))
            y = torch.empty_like(x)
            moe.moe_forward_noalloc(config, w, x, T, y, status)
            torch.cuda.synchronize()
            assert int(status.item()) == moe.MOE_OK
            err = np.max(np.abs(bf16_f64(to_host_bits(y)) - y_ref))
            assert err <= y_tol(y_ref), (T, err)
    finally:
        layer.close()


def test_noalloc_rejects_what_it_cannot_serve(cuda_device):
    cfg = W.CONFIGS["tiny"]
    w = _device_weights(cfg, 0)
    config = config_dict(cfg, 8)
    x = to_dev(W.activations(cfg, 0))
    y = torch.empty_like(x)
    with pytest.raises(moe.MoeError) as ei:  # more than 4 tokens
        moe.moe_forward_noalloc(config, w, torch.cat([x, x]), 8, torch.cat([y, y]))
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    # scratch would not fit: hidden 4096 needs two 4-token fp32 output
    # accumulators of 64 KiB each, beyond the 128 KiB array with the rest;
    # refused before any launch (a valid layer shape otherwise)
    big = dict(config, hidden=4096, n_experts=128, n_slots=128, top_k=8, ffn=512, shared_ffn=512)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_noalloc(big, w, x, 1, y)
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    w2 = dict(w)
    w2["router_bias"] = None
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_noalloc(config, w2, x, 4, y)
    assert ei.value.status == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:  # host memory is not accepted
        moe.moe_forward_noalloc(config, w, x.cpu(), 4, y)
    assert ei.value.status == moe.MOE_ERR_INVALID
    # a weight tensor that starts 2 bytes into its allocation cannot feed the
    # kernel's 16-byte copies: refused on the host, nothing is launched
    for name in ("down_q", "up_s", "router_w"):
        w3 = dict(w)
        flat = w[name].reshape(-1).view(torch.uint8)
        shifted = torch.empty(flat.numel() + 16, dtype=torch.uint8, device="cuda")
        w3[name] = shifted[2:2 + flat.numel()]
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_forward_noalloc(config, w3, x, 4, y)
        assert ei.value.status == moe.MOE_ERR_INVALID, name
    torch.cuda.synchronize()
