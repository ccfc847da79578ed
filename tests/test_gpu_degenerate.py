"""Degenerate shapes and inputs through both paths, against the oracle:
dense routing (k = E), a single expert (E = 1), and an all-zero input (every
logit ties, so the selection is the lowest ids and the output is exactly
zero)."""
import numpy as np
import pytest

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import bf16_f64, check_topk, make_layer_host, to_dev, to_host_bits, y_tol

pytestmark = pytest.mark.gpu


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
    yg = bf16_f64(to_host_bits(y))
    assert np.max(np.abs(yg - y_ref)) <= y_tol(y_ref)
    return ids, yg


@pytest.mark.parametrize("T", [1, 4, 40])
def test_dense_routing_k_equals_E(cuda_device, T):
    cfg = W.CONFIGS["tiny"].replace(top_k=16, zipf_s=1.1, permuted_slots=True)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=64)
    ids, _ = _check(cfg, Ld, layer, W.activations(cfg, 2, n_tokens=T))
    assert all(sorted(r) == list(range(16)) for r in ids.tolist())
    layer.close()


@pytest.mark.parametrize("T", [1, 3, 40])
def test_single_expert(cuda_device, T):
    cfg = W.CONFIGS["tiny"].replace(n_experts=1, top_k=1)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=64)
    ids, _ = _check(cfg, Ld, layer, W.activations(cfg, 3, n_tokens=T))
    assert np.all(ids == 0)
    layer.close()


@pytest.mark.parametrize("T", [2, 40])
def test_zero_input_ties_to_the_lowest_ids_and_gives_zero(cuda_device, T):
    cfg = W.CONFIGS["tiny"]  # no router bias: every logit of a zero input is 0
    layer, Ld = make_layer_host(cfg, 0, max_tokens=64)
    x = np.zeros((T, cfg.hidden), np.uint16)
    ids, yg = _check(cfg, Ld, layer, x)
    assert all(list(r) == list(range(cfg.top_k)) for r in ids.tolist())
    assert np.all(yg == 0.0)
    # a stack of such layers keeps the zero state (the norm of zero is zero)
    made = [make_layer_host(cfg, l, max_tokens=64) for l in range(2)]
    h = moe.stack_forward([m[0] for m in made], to_dev(x))
    assert moe.moe_status_sync(made[0][0].handle) == moe.MOE_OK
    assert np.all(bf16_f64(to_host_bits(h)) == 0.0)
    for m in made:
        m[0].close()
    layer.close()
