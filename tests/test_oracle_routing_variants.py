"""Pins of the oracle's routing variants (no renormalisation, bias for
selection only, sigmoid-gated shared expert) to closed forms, library
routines and special cases that reduce to the default routing."""
import math

import numpy as np
import pytest
import scipy.special

import oracle
import workload as W

NO_RENORM, SELECT_ONLY, SHARED_GATE = 1, 2, 4


def rng(seed=0):
    return np.random.default_rng(seed)


def test_default_flags_reproduce_the_selection_softmax():
    z = rng(1).standard_normal((30, 64)) * 2
    ids, w, _ = oracle.topk_softmax(z, 6)
    w0 = oracle.route_weights(z, None, ids, 0)
    assert np.allclose(w0, w, rtol=1e-13, atol=0)


def test_no_renorm_closed_form_three_experts():
    z = np.array([[0.0, 1.0, 2.0]])
    ids, _, _ = oracle.topk_softmax(z, 2)
    assert list(ids[0]) == [2, 1]
    w = oracle.route_weights(z, None, ids, NO_RENORM)
    den = 1.0 + math.e + math.e ** 2
    assert w[0, 0] == pytest.approx(math.e ** 2 / den, rel=1e-14)
    assert w[0, 1] == pytest.approx(math.e / den, rel=1e-14)


def test_no_renorm_is_the_full_softmax_at_the_selection():
    z = rng(2).standard_normal((20, 128)) * 3
    ids, w_sel, _ = oracle.topk_softmax(z, 8)
    w = oracle.route_weights(z, None, ids, NO_RENORM)
    for t in range(20):
        p = scipy.special.softmax(z[t])
        assert np.allclose(w[t], p[ids[t]], rtol=1e-12)
        # the renormalised weights are these divided by the selected mass
        assert np.allclose(w_sel[t], w[t] / w[t].sum(), rtol=1e-12)
    assert np.all(w.sum(1) < 1.0)
    # k = E: nothing is left out, so both readings agree
    ids_all, w_all, _ = oracle.topk_softmax(z[:3, :8], 8)
    assert np.allclose(oracle.route_weights(z[:3, :8], None, ids_all, NO_RENORM), w_all, rtol=1e-13)


def test_bias_for_selection_only_closed_form():
    z0 = np.array([[0.0, 1.0, 2.0]])
    b = np.array([5.0, 0.0, 0.0], np.float32)
    zsel = z0 + b.astype(np.float64)
    ids, _, _ = oracle.topk_softmax(zsel, 2)
    assert list(ids[0]) == [0, 2]  # the bias lifts expert 0 into the selection
    w = oracle.route_weights(zsel, b, ids, SELECT_ONLY)
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.e ** 2), rel=1e-14)
    assert w[0, 1] == pytest.approx(math.e ** 2 / (1.0 + math.e ** 2), rel=1e-14)
    w3 = oracle.route_weights(zsel, b, ids, SELECT_ONLY | NO_RENORM)
    den = 1.0 + math.e + math.e ** 2
    assert w3[0, 0] == pytest.approx(1.0 / den, rel=1e-14)
    assert w3[0, 1] == pytest.approx(math.e ** 2 / den, rel=1e-14)


def test_bias_for_selection_only_with_zero_bias_is_the_default():
    z = rng(3).standard_normal((10, 32))
    ids, w, _ = oracle.topk_softmax(z, 4)
    zero = np.zeros(32, np.float32)
    assert np.allclose(oracle.route_weights(z, zero, ids, SELECT_ONLY), w, rtol=1e-13)
    assert np.allclose(oracle.route_weights(z, zero, ids, SELECT_ONLY | NO_RENORM),
                       oracle.route_weights(z, None, ids, NO_RENORM), rtol=1e-13)


def test_shared_gate_closed_forms():
    H = 32
    one = W.f32_to_bf16_bits(np.ones(H, np.float32))
    assert oracle.shared_gate(np.zeros(H, np.float32), one) == 0.5
    g = np.zeros(H, np.float32)
    g[0] = math.log(3.0)
    assert oracle.shared_gate(g, one) == pytest.approx(0.75, abs=1e-7)
    g[0] = -math.log(3.0)
    assert oracle.shared_gate(g, one) == pytest.approx(0.25, abs=1e-7)
    # the dot product runs over the whole row
    x = W.f32_to_bf16_bits(np.arange(H, dtype=np.float32) / 8)
    gg = np.full(H, 0.01, np.float32)
    ref = 1.0 / (1.0 + math.exp(-sum(0.01 * i / 8 for i in range(H))))
    assert oracle.shared_gate(gg, x) == pytest.approx(ref, rel=1e-6)


def _tiny(flags, **kw):
    return W.CONFIGS["tiny"].replace(zipf_s=1.1, routing_flags=flags, **kw)


def test_gated_layer_scales_only_the_shared_term():
    cfg = _tiny(SHARED_GATE)
    Ld = W.layer(cfg, 0)
    x = W.activations(cfg, 2)
    yg, ids_g, w_g, _ = oracle.moe_forward(Ld, cfg.top_k, x)
    L0 = dict(Ld, routing_flags=0)
    y0, ids_0, w_0, _ = oracle.moe_forward(L0, cfg.top_k, x)
    assert np.array_equal(ids_g, ids_0) and np.array_equal(w_g, w_0)
    sh = W.shared_expert(cfg, 0)
    for t in range(x.shape[0]):
        ysh = oracle.combine_token([], [], sh, x[t])
        gate = oracle.shared_gate(Ld["sh_gate_w"], x[t])
        assert 0.0 < gate < 1.0
        ref = y0[t] - ysh + gate * ysh
        assert np.allclose(yg[t], ref, rtol=0, atol=1e-12 * np.abs(y0[t]).max())


def test_variants_keep_the_selection_and_change_only_the_weights():
    cfg = _tiny(0)
    Ld = W.layer(cfg, 0)
    x = W.activations(cfg, 4)
    z = oracle.router_logits(Ld["router_w"], Ld["router_b"], x)
    _, ids0, _, m0 = oracle.moe_forward(Ld, cfg.top_k, x)
    for flags in (NO_RENORM, SELECT_ONLY, NO_RENORM | SELECT_ONLY):
        _, ids, w, m = oracle.moe_forward(dict(Ld, routing_flags=flags), cfg.top_k, x)
        assert np.array_equal(ids, ids0) and np.array_equal(m, m0)
        assert np.allclose(w, oracle.route_weights(z, Ld["router_b"], ids, flags), rtol=1e-12)
    # with the Zipf bias the selection-only weights differ from the default
    _, _, w_sel, _ = oracle.moe_forward(dict(Ld, routing_flags=SELECT_ONLY), cfg.top_k, x)
    _, _, w_def, _ = oracle.moe_forward(Ld, cfg.top_k, x)
    assert np.max(np.abs(w_sel - w_def)) > 1e-3


def test_gated_layer_rejects_missing_gate_vector():
    cfg = _tiny(SHARED_GATE)
    Ld = dict(W.layer(cfg, 0))
    del Ld["sh_gate_w"]
    with pytest.raises(ValueError):
        oracle.moe_forward(Ld, cfg.top_k, W.activations(cfg, 0))
