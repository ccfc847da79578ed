"""The allocation-free decode entry point (moe_forward_noalloc), checked
through the C ABI against moe_forward on the same weights and inputs.

It exists for callers that cannot allocate device memory when they run a
layer (graph capture into a pool they do not own, plug-ins under a host
framework's allocator, fixed post-start-up memory budgets): its scratch is a
static device array inside the library.  This file is collected last."""
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
        for T in (1, 4):
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


def test_noalloc_rejects_what_it_cannot_serve(cuda_device):
    cfg = W.CONFIGS["tiny"]
    w = _device_weights(cfg, 0)
    config = config_dict(cfg, 8)
    x = to_dev(W.activations(cfg, 0))
    y = torch.empty_like(x)
    with pytest.raises(moe.MoeError) as ei:  # more than 4 tokens
        moe.moe_forward_noalloc(config, w, torch.cat([x, x]), 8, torch.cat([y, y]))
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    # scratch would not fit: 4 tokens x (64 routed units x F 4096 + Fs 4096)
    # fp32 intermediates exceed the 4 MiB array; rejected before any launch
    big = dict(config, n_experts=1024, n_slots=1024, top_k=16, ffn=4096, shared_ffn=4096)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_noalloc(big, w, x, 4, y)
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    w2 = dict(w)
    w2["router_bias"] = None
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_noalloc(config, w2, x, 4, y)
    assert ei.value.status == moe.MOE_ERR_INVALID
    with pytest.raises(moe.MoeError) as ei:  # host memory is not accepted
        moe.moe_forward_noalloc(config, w, x.cpu(), 4, y)
    assert ei.value.status == moe.MOE_ERR_INVALID
