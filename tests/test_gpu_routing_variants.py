"""GPU parity of the routing variants (no renormalisation, bias for selection
only, sigmoid-gated shared expert, and all three together) against the
oracle through the C ABI: decode (1..4 tokens), prefill (tile-sized and
ragged batches), routing only, a short residual stack of each path, and the
allocation-free entry point."""
import numpy as np
import pytest
import torch

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import (bf16_f64, check_stack_outputs, check_topk, config_dict, host_weights,
                    make_layer_host, to_dev, to_host_bits, y_tol)

pytestmark = pytest.mark.gpu

NO_RENORM, SELECT_ONLY, SHARED_GATE = (moe.ROUTING_NO_RENORM, moe.ROUTING_BIAS_SELECT_ONLY,
                                       moe.ROUTING_SHARED_GATE)
ALL = NO_RENORM | SELECT_ONLY | SHARED_GATE


def _cfg(flags, **kw):
    # the Zipf bias makes the selection-only weights differ from the default
    return W.CONFIGS["tiny"].replace(zipf_s=1.1, permuted_slots=True, routing_flags=flags, **kw)


def _check(cfg, Ld, layer, x):
    T = x.shape[0]
    xd = to_dev(x)
    y = layer.forward(xd)
    ids, w = layer.route(xd)
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    z = oracle.router_logits(Ld["router_w"], Ld["router_b"], x)
    adopt = [check_topk(ids[t], z[t], cfg.top_k) for t in range(T)]
    y_ref, _, w_ref, _ = oracle.moe_forward(Ld, cfg.top_k, x, forced_ids=ids if any(adopt) else None)
    assert np.max(np.abs(w - w_ref)) < 1e-5
    if cfg.routing_flags & NO_RENORM:
        assert np.all(w.sum(1) < 1.0)
    yg = bf16_f64(to_host_bits(y))
    err = np.max(np.abs(yg - y_ref))
    assert err <= y_tol(y_ref), (err, y_tol(y_ref))


@pytest.mark.parametrize("flags", [NO_RENORM, SELECT_ONLY, SHARED_GATE, NO_RENORM | SELECT_ONLY, ALL])
@pytest.mark.parametrize("T", [1, 3, 4, 40, 300])
def test_variant_forward_and_route(cuda_device, flags, T):
    cfg = _cfg(flags)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=512)
    for idx in range(2):
        _check(cfg, Ld, layer, W.activations(cfg, 7 + idx, n_tokens=T))
    layer.close()


def test_variant_mid_shape_prefill(cuda_device):
    # several 128-row tiles and K steps, E not a multiple of 128, all variants
    cfg = W.MoEConfig("mid", 700, 1, 512, 40, 4, 256, 384, True, 1.1, 21, 21, routing_flags=ALL)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=1024)
    _check(cfg, Ld, layer, W.activations(cfg, 0))
    layer.close()


@pytest.mark.parametrize("T", [2, 40])
def test_variant_stack_teacher_forced(cuda_device, T):
    cfg = _cfg(ALL)
    L = 3
    made = [make_layer_host(cfg, l, max_tokens=64) for l in range(L)]
    layers = [m[0] for m in made]
    x = W.activations(cfg, 4, n_tokens=T)
    y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
    assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
    h_trace, in_trace = to_host_bits(h_trace), to_host_bits(in_trace)
    y_trace = to_host_bits(y_trace)
    ids_trace = ids_trace.cpu().numpy()
    h_prev = x
    for l in range(L):
        Ld = made[l][1]
        u = in_trace[l]
        z = oracle.router_logits(Ld["router_w"], Ld["router_b"], u)
        adopt = [check_topk(ids_trace[l, t], z[t], cfg.top_k) for t in range(T)]
        y_ref = oracle.moe_forward(Ld, cfg.top_k, u, forced_ids=ids_trace[l] if any(adopt) else None)[0]
        check_stack_outputs(h_prev, y_trace[l], h_trace[l], y_ref, where=l)
        h_prev = h_trace[l]
    for lay in layers:
        lay.close()


def test_variant_noalloc_matches_layer(cuda_device):
    cfg = _cfg(ALL)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=8)
    w = {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if isinstance(v, np.ndarray) else v)
         for k, v in host_weights(Ld).items()}
    config = config_dict(cfg, 4)
    for T in (1, 4):
        xh = W.activations(cfg, 9, n_tokens=T)
        x = to_dev(xh)
        y = torch.empty_like(x)
        moe.moe_forward_noalloc(config, w, x, T, y)
        torch.cuda.synchronize()
        a, b = bf16_f64(to_host_bits(y)), bf16_f64(to_host_bits(layer.forward(x)))
        if T == 1:
            # same kernel path; the fp32 reductions may add in another order
            assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-30)
        else:
            # more than one token: the library layer runs its gate/up items on
            # the tensor cores (block-major tensor maps it owns), the
            # allocation-free call keeps the fp16 path (caller-owned weights,
            # no maps): each within the y tolerance of the oracle
            ids, _ = layer.route(x)
            ids = ids.cpu().numpy()
            z = oracle.router_logits(Ld["router_w"], Ld["router_b"], xh)
            adopt = [check_topk(ids[t], z[t], cfg.top_k) for t in range(T)]
            y_ref = oracle.moe_forward(Ld, cfg.top_k, xh, forced_ids=ids if any(adopt) else None)[0]
            for yv in (a, b):
                assert np.max(np.abs(yv - y_ref)) <= y_tol(y_ref)
    layer.close()
