"""GPU parity of partial residency (n_slots < n_experts): only n_slots experts
per layer keep an HBM slot, the rest live in the library's pinned host tier.
Results must equal those of a fully resident layer -- the oracle knows
nothing about residency -- while the cache evolves: decode calls fetch
missed experts into least-recently-used slots, prefill-sized calls stage
the experts they select.  Checked through the C ABI against the oracle, and
the slot table's invariants and the hit/miss counters after every call."""
import gc

import numpy as np
import pytest
import torch

import oracle
import quantized_expert_ffn_softmax_gb300 as moe
import workload as W
from parity import (bf16_f64, check_stack_outputs, check_topk, config_dict, host_weights,
                    make_layer_device, oracle_token, parallel_map, to_dev, to_host_bits, y_tol)

pytestmark = pytest.mark.gpu


def _profile(cfg, layer_idx):
    """A usage profile: the Zipf prior of the router bias (exp of the bias)."""
    _, b = W.router(cfg, layer_idx)
    return np.exp(b.astype(np.float64)).astype(np.float32)


def _partial_host_layer(cfg, layer_idx, n_slots, max_tokens=512, profile=True):
    Ld = W.layer(cfg, layer_idx)
    w = host_weights(Ld)
    if profile:
        w["expert_profile"] = _profile(cfg, layer_idx)
    conf = dict(config_dict(cfg, max_tokens), n_slots=n_slots)
    return moe.MoELayer(conf, w, False), Ld


def _check_slot_table(layer, E, S):
    tab = moe.moe_cache_slots(layer.handle, E)
    res = tab[tab >= 0]
    assert res.size == S, (res.size, S)
    assert np.array_equal(np.sort(res), np.arange(S))
    assert np.all(tab >= -1)
    return tab


def _check_call(cfg, Ld, layer, x):
    T = x.shape[0]
    xd = to_dev(x)
    y = layer.forward(xd)
    ids, w = layer.route(xd)
    assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
    ids = ids.cpu().numpy()
    z = oracle.router_logits(Ld["router_w"], Ld["router_b"], x)
    adopt = [check_topk(ids[t], z[t], cfg.top_k) for t in range(T)]
    y_ref = oracle.moe_forward(Ld, cfg.top_k, x, forced_ids=ids if any(adopt) else None)[0]
    yg = bf16_f64(to_host_bits(y))
    err = np.max(np.abs(yg - y_ref))
    assert err <= y_tol(y_ref), (err, y_tol(y_ref))
    return ids


@pytest.mark.parametrize("profile", [True, False])
def test_tiny_decode_partial_matches_oracle_and_keeps_the_table_valid(cuda_device, profile):
    cfg = W.CONFIGS["tiny"].replace(permuted_slots=True, zipf_s=1.1)
    S = 8  # half of the 16 experts (the least allowed: 4 tokens x top-2)
    layer, Ld = _partial_host_layer(cfg, 0, S, profile=profile)
    E = cfg.n_experts
    tab0 = _check_slot_table(layer, E, S)
    if profile:  # the first residents are the experts with the largest prior
        prof = _profile(cfg, 0)
        top = np.argsort(-prof, kind="stable")[:S]
        assert set(np.nonzero(tab0 >= 0)[0].tolist()) == set(top.tolist())
    else:
        assert set(np.nonzero(tab0 >= 0)[0].tolist()) == set(range(S))
    lookups = 0
    for i in range(24):
        T = 1 + i % 4
        before = moe.moe_cache_slots(layer.handle, E)
        ids = _check_call(cfg, Ld, layer, W.activations(cfg, 200 + i, n_tokens=T))
        after = _check_slot_table(layer, E, S)
        uniq = sorted(set(ids.ravel().tolist()))
        lookups += len(uniq)
        # every expert of the call is resident after it; the ones that were
        # not resident before took slots whose experts this call did not use
        assert np.all(after[uniq] >= 0)
        moved = [e for e in range(E) if before[e] >= 0 and after[e] < 0]
        assert not (set(moved) & set(uniq))
    hits, misses = moe.moe_cache_stats(layer.handle)
    assert hits + misses == lookups and hits > 0
    if not profile:  # experts 0..7 first: the Zipf-favoured others must come in
        assert misses > 0
    print("tiny, 8 of 16 experts resident, profile=%s: %d hits, %d misses" % (profile, hits, misses))
    moe.moe_cache_stats(layer.handle, reset=True)
    assert moe.moe_cache_stats(layer.handle) == (0, 0)
    layer.close()


@pytest.mark.parametrize("T", [5, 40, 300])
def test_tiny_prefill_partial_matches_oracle(cuda_device, T):
    cfg = W.CONFIGS["tiny"].replace(permuted_slots=True, zipf_s=1.1)
    layer, Ld = _partial_host_layer(cfg, 0, 8)
    for idx in range(2):
        _check_call(cfg, Ld, layer, W.activations(cfg, 300 + idx, n_tokens=T))
    # the prefill path reads the cache without changing it
    _check_slot_table(layer, cfg.n_experts, 8)
    layer.close()


@pytest.mark.parametrize("T", [2, 40])
def test_tiny_stack_partial_teacher_forced(cuda_device, T):
    cfg = W.CONFIGS["tiny"].replace(permuted_slots=True, zipf_s=1.1)
    L = 4
    made = [_partial_host_layer(cfg, l, 8, max_tokens=64) for l in range(L)]
    layers = [m[0] for m in made]
    x = W.activations(cfg, 5, n_tokens=T)
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


def test_fully_resident_layer_reports_no_cache_counts(cuda_device):
    cfg = W.CONFIGS["tiny"]
    Ld = W.layer(cfg, 0)
    layer = moe.MoELayer(config_dict(cfg, 8), host_weights(Ld), False)
    layer.forward(to_dev(W.activations(cfg, 0)))
    assert moe.moe_cache_stats(layer.handle) == (0, 0)
    tab = moe.moe_cache_slots(layer.handle, cfg.n_experts)
    assert np.array_equal(np.sort(tab), np.arange(cfg.n_experts))
    layer.close()


def _device_partial_layer(cfg, l, n_slots, max_tokens, profile=True):
    Dd = W.device_layer(cfg, l)
    w = {n: Dd[n] for n in ("router_w", "slot_of_expert", "gate_q", "gate_s", "up_q", "up_s",
                            "down_q", "down_s")}
    w["router_bias"] = Dd["router_b"]
    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        w["sh_" + n] = Dd["sh_" + n]
    if profile:
        w["expert_profile"] = torch.from_numpy(_profile(cfg, l)).cuda()
    torch.cuda.synchronize()
    conf = dict(config_dict(cfg, max_tokens), n_slots=n_slots)
    layer = moe.MoELayer(conf, w, True)
    del Dd, w
    return layer


@pytest.mark.parametrize("profile", [True, False])
def test_decode35b_quarter_resident_stack_parity(cuda_device, profile):
    """Eight layers of the 35B-shaped stack with 64 of 256 experts per layer
    in HBM (placed by the usage profile, or experts 0..63 without one, which
    misses): after a few steps of other inputs, one traced step checks every
    layer's y at the stated tolerance (teacher forced) and the residual."""
    cfg = W.CONFIGS["decode35b"].replace(n_layers=8)
    layers = [_device_partial_layer(cfg, l, 64, 8, profile) for l in range(cfg.n_layers)]
    try:
        for i in range(4):  # the cache moves
            moe.stack_forward(layers, to_dev(W.activations(cfg, 50 + i)))
        x = W.activations(cfg, 3)
        y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
        assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
        stats = [moe.moe_cache_stats(l.handle) for l in layers]
        for l in layers:
            _check_slot_table(l, cfg.n_experts, 64)
        h_trace, in_trace = to_host_bits(h_trace), to_host_bits(in_trace)
        y_trace, ids_trace = to_host_bits(y_trace), ids_trace.cpu().numpy()
    finally:
        for l in layers:
            l.close()
        del layers
        gc.collect()
        torch.cuda.empty_cache()
    assert all(h + m == 5 * cfg.top_k for h, m in stats)
    if not profile:
        assert sum(m for _, m in stats) > 0
    h_in = [x] + [h_trace[l] for l in range(cfg.n_layers - 1)]

    def check_layer(l):
        u = in_trace[l]
        Wr, b = W.router(cfg, l)
        sh = W.shared_expert(cfg, l)
        y_ref, _, _ = oracle_token(cfg, l, u[0], gpu_ids=ids_trace[l, 0], router=(Wr, b), shared=sh)
        return check_stack_outputs(h_in[l], y_trace[l], h_trace[l], y_ref[None, :], where=l)

    parallel_map(check_layer, range(cfg.n_layers))
    print("decode35b, 64 of 256 experts resident, profile=%s: hits/misses per layer %s"
          % (profile, stats))


def test_prefill125b_half_resident_equals_fully_resident(cuda_device):
    """The 8192-token chunk through one 125B-shaped layer with 256 of 512
    experts in HBM (the rest staged from the host tier) gives the same
    selection and, up to the order of the fp32 combine, the same output as
    the fully resident layer."""
    cfg = W.CONFIGS["prefill125b"]
    x = to_dev(W.activations(cfg, 1))
    full = make_layer_device(cfg, 0, max_tokens=cfg.n_tokens)
    try:
        y_full = bf16_f64(to_host_bits(full.forward(x)))
        ids_full = full.route(x)[0].cpu().numpy()
        assert moe.moe_status_sync(full.handle) == moe.MOE_OK
    finally:
        full.close()
        gc.collect()
        torch.cuda.empty_cache()
    part = _device_partial_layer(cfg, 0, 256, cfg.n_tokens)
    try:
        y_part = bf16_f64(to_host_bits(part.forward(x)))
        ids_part = part.route(x)[0].cpu().numpy()
        assert moe.moe_status_sync(part.handle) == moe.MOE_OK
    finally:
        part.close()
        gc.collect()
        torch.cuda.empty_cache()
    assert np.array_equal(ids_full, ids_part)
    bound = 2.0 ** -7 * np.abs(y_full) + 1e-5 * np.abs(y_full).max()
    assert np.all(np.abs(y_part - y_full) <= bound), float(np.max(np.abs(y_part - y_full)))
