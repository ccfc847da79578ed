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
from parity import (bf16_f64, check_stack_outputs, check_topk, config_dict, host_weights,
                    make_layer_device, make_layer_host, oracle_token, parallel_map, to_dev,
                    to_host_bits, y_tol)

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


def test_prefill_hidden_not_a_multiple_of_256(cuda_device):
    # the down GEMM takes H in 256-row tiles: with H = 384 the last tile's
    # second half lies past the matrix (zero weights, nothing written)
    cfg = W.MoEConfig("oddh", 300, 1, 384, 24, 3, 256, 256, True, 1.1, 23, 23)
    layer, Ld = make_layer_host(cfg, 0, max_tokens=512)
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
    # every token's partial rows are summed in one fixed order: bit-exact repeat
    assert np.array_equal(y_host, y_dev)
    layer.close()


def test_prefill_stack_teacher_forced(cuda_device):
    cfg = W.CONFIGS["tiny"].replace(n_tokens=40)
    L = 3
    made = [make_layer_host(cfg, l, max_tokens=64) for l in range(L)]
    layers = [m[0] for m in made]
    x = W.activations(cfg, 4, n_tokens=40)
    y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
    assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
    h_trace, in_trace = to_host_bits(h_trace), to_host_bits(in_trace)
    y_trace = to_host_bits(y_trace)
    ids_trace = ids_trace.cpu().numpy()
    assert np.array_equal(to_host_bits(y), h_trace[-1])
    h_prev = x
    for l in range(L):
        Ld = made[l][1]
        u = in_trace[l]
        u_ref = bf16_f64(oracle.rmsnorm(h_prev))
        assert np.all(np.abs(bf16_f64(u) - u_ref) <= 2.0 ** -7 * np.abs(u_ref) + 1e-30)
        z = oracle.router_logits(Ld["router_w"], Ld["router_b"], u)
        adopt = [check_topk(ids_trace[l, t], z[t], cfg.top_k) for t in range(40)]
        y_ref = oracle.moe_forward(Ld, cfg.top_k, u, forced_ids=ids_trace[l] if any(adopt) else None)[0]
        check_stack_outputs(h_prev, y_trace[l], h_trace[l], y_ref, where=l)
        h_prev = h_trace[l]
    for l in layers:
        l.close()


def _chunk_tokens_to_check(ids, offs, perm, T, rng):
    """Tokens whose outputs the 8192-token test checks against the oracle:
    the first and last 32 rows of the largest bucket (its first token tile
    and its ragged last tile), the token of every single-token bucket (up to
    64), the first 16 and last 32 tokens of the chunk, and random tokens up
    to 288 in all."""
    counts = np.diff(offs)
    e_big = int(np.argmax(counts))
    big = perm[offs[e_big]:offs[e_big + 1]]
    picks = [big[:32], big[-32:]]
    singles = np.nonzero(counts == 1)[0][:64]
    picks.append(perm[offs[singles]])
    picks.append(np.arange(16))
    picks.append(np.arange(T - 32, T))
    chosen = np.unique(np.concatenate(picks).astype(np.int64))
    rest = np.setdiff1d(np.arange(T), chosen)
    extra = rng.choice(rest, max(0, 288 - chosen.size), replace=False)
    return np.sort(np.concatenate([chosen, extra])), e_big, singles


def test_prefill125b_chunk_parity(cuda_device):
    """The full 8192-token chunk through one 125B-shaped layer: ALL 8192
    tokens' top-k ids against the oracle's fp64 logits (parity rule with the
    1e-4 tie margin) and their routing weights summing to 1; the bucketing
    (offsets and row order) bit-exact against the oracle's counting sort of
    the GPU's ids; repeated runs agreeing bit for bit;
    and 288 tokens' outputs against the oracle at the stated tolerance --
    rows of the largest bucket's first and ragged last tile, every
    single-token bucket's token (up to 64), both ends of the chunk and random
    tokens."""
    cfg = W.CONFIGS["prefill125b"]
    T = cfg.n_tokens
    layer = make_layer_device(cfg, 0, max_tokens=T)
    try:
        x = W.activations(cfg, 0)
        xd = to_dev(x)
        y = to_host_bits(layer.forward(xd))
        assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
        # every partial row is written once and each token's rows are summed
        # in one fixed order, so repeated runs agree bit for bit: a pipeline
        # race that hands a buffer back early shows up here
        for _ in range(2):
            yr = to_host_bits(layer.forward(xd))
            assert moe.moe_status_sync(layer.handle) == moe.MOE_OK
            assert np.array_equal(yr, y), int(np.sum(yr != y))
        ids, w = layer.route(xd)
        ids, w = ids.cpu().numpy(), w.cpu().numpy()
        offs = np.zeros(cfg.n_experts + 1, np.int32)
        perm = np.zeros(T * cfg.top_k, np.int32)
        moe.moe_last_buckets(layer.handle, T, offs, perm)
    finally:
        layer.close()
        gc.collect()
        torch.cuda.empty_cache()
    counts, offs_ref, pt_ref, _ = oracle.bucket(ids, cfg.n_experts)
    assert np.array_equal(offs, offs_ref) and np.array_equal(perm, pt_ref)
    # skew of the Zipf-biased router: bucket sizes from 0 to thousands
    assert counts.max() > 1000 and (counts == 0).sum() > 50
    Wr, b = W.router(cfg, 0)
    # every token's top-k against the oracle's logits (in 64 slices on threads)
    slices = np.array_split(np.arange(T), 64)

    def topk_slice(ts):
        zs = oracle.router_logits(Wr, b, x[ts])
        return sum(check_topk(ids[t], zs[i], cfg.top_k) for i, t in enumerate(ts))

    n_ties = sum(parallel_map(topk_slice, slices))
    assert np.all(np.abs(w.sum(1) - 1.0) < 1e-5)
    print("prefill125b: top-k of all %d tokens checked, %d near-tie adoptions" % (T, n_ties))
    rng = np.random.default_rng(0)
    toks, e_big, singles = _chunk_tokens_to_check(ids, offs, perm, T, rng)
    assert toks.size >= 256 and singles.size > 0
    sh = W.shared_expert(cfg, 0)
    need = sorted(set(ids[toks].ravel().tolist()))
    cache = dict(zip(((0, e) for e in need), parallel_map(lambda e: W.expert(cfg, 0, e), need)))

    def check_token(t):
        y_ref, _, _ = oracle_token(cfg, 0, x[t], gpu_ids=ids[t], router=(Wr, b), shared=sh,
                                   expert_cache=cache)
        err = float(np.max(np.abs(bf16_f64(y[t]) - y_ref)))
        assert err <= y_tol(y_ref), (int(t), err, y_tol(y_ref))
        return err / y_tol(y_ref)

    worst = max(parallel_map(check_token, toks))
    print("prefill125b: %d tokens' y checked (largest bucket %d: %d rows), worst error / "
          "tolerance %.3f" % (toks.size, e_big, counts[e_big], worst))


def test_prefill125b_48_layer_stack_teacher_forced(cuda_device):
    """The 8192-token chunk through the 48-layer 125B-shaped stack (pre-norm
    residual, fused layer boundaries).  On five layers spread over the stack
    (teacher forced: the oracle takes the GPU's input of the layer): the RMS
    norm of every token, every token's top-k against the oracle's logits,
    and 32 tokens' y at the stated tolerance with their residual; every
    layer's output finite."""
    cfg = W.CONFIGS["prefill125b"].replace(n_layers=48)
    T, L = cfg.n_tokens, cfg.n_layers
    layers = [make_layer_device(cfg, l, max_tokens=T) for l in range(L)]
    try:
        x = W.activations(cfg, 2)
        y, h_trace, in_trace, y_trace, ids_trace = moe.stack_forward(layers, to_dev(x), trace=True)
        assert moe.moe_status_sync(layers[0].handle) == moe.MOE_OK
        check = [0, 1, 23, 46, 47]
        y_last = to_host_bits(y)
        h_in = {l: (x if l == 0 else to_host_bits(h_trace[l - 1])) for l in check}
        h_out = {l: to_host_bits(h_trace[l]) for l in check}
        u_tr = {l: to_host_bits(in_trace[l]) for l in check}
        y_tr = {l: to_host_bits(y_trace[l]) for l in check}
        ids_tr = {l: ids_trace[l].cpu().numpy() for l in check}
        finite = bool(torch.isfinite(y_trace.view(torch.bfloat16).float()).all())
        assert np.array_equal(y_last, to_host_bits(h_trace[L - 1]))
    finally:
        for l in layers:
            l.close()
        del layers
        gc.collect()
        torch.cuda.empty_cache()
    assert finite
    rng = np.random.default_rng(1)
    for l in check:
        u = u_tr[l]
        u_ref = bf16_f64(oracle.rmsnorm(h_in[l]))
        assert np.all(np.abs(bf16_f64(u) - u_ref) <= 2.0 ** -7 * np.abs(u_ref) + 1e-30), l
        Wr, b = W.router(cfg, l)
        slices = np.array_split(np.arange(T), 64)

        def topk_slice(ts):
            zs = oracle.router_logits(Wr, b, u[ts])
            return sum(check_topk(ids_tr[l][t], zs[i], cfg.top_k) for i, t in enumerate(ts))

        parallel_map(topk_slice, slices)
        toks = np.sort(rng.choice(T, 32, replace=False))
        sh = W.shared_expert(cfg, l)
        need = sorted(set(ids_tr[l][toks].ravel().tolist()))
        cache = dict(zip(((l, e) for e in need), parallel_map(lambda e: W.expert(cfg, l, e), need)))

        def y_ref_of(t):
            return oracle_token(cfg, l, u[t], gpu_ids=ids_tr[l][t], router=(Wr, b), shared=sh,
                                expert_cache=cache)[0]

        y_ref = np.stack(parallel_map(y_ref_of, toks))
        check_stack_outputs(h_in[l][toks], y_tr[l][toks], h_out[l][toks], y_ref, where=l)
