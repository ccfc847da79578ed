"""Why the stack is a pre-norm residual (the stack reading): with the oracle
alone, a plain residual stack h_{l+1} = bf16(h_l + bf16(MoE_l(h_l))) of the
35B-A3B-shaped layers diverges -- the SwiGLU output grows with the square of
its input, so every layer feeds the next a larger input -- and reaches
non-finite values within 30 layers, while the pre-norm stack
u_l = rmsnorm(h_l), h_{l+1} = bf16(h_l + bf16(MoE_l(u_l))) on the same
layers and input stays finite with an RMS that grows slowly.  Only the
selected experts of each layer are drawn, so this runs on CPU in seconds."""
import numpy as np

import oracle
import workload as W


def _run(cfg, x, n_layers, pre_norm):
    h = x.copy()
    rms = []
    for l in range(n_layers):
        Wr, b = W.router(cfg, l)
        u = oracle.rmsnorm(h) if pre_norm else h
        z = oracle.router_logits(Wr, b, u)
        ids, w, _ = oracle.topk_softmax(z, cfg.top_k)
        exs = [W.expert(cfg, l, int(e)) for e in ids[0]]
        y = oracle.combine_token(exs, w[0], W.shared_expert(cfg, l), u[0])
        h = oracle.residual(h, y[None, :])
        hf = W.bf16_bits_to_f32(h).astype(np.float64)
        if not np.all(np.isfinite(hf)):
            return l, rms
        rms.append(float(np.sqrt(np.mean(hf ** 2))))
    return None, rms


def test_plain_residual_stack_diverges_and_pre_norm_stays_finite():
    cfg = W.CONFIGS["decode35b"]
    x = W.activations(cfg, 0)
    blew_up_at, rms_plain = _run(cfg, x, 30, pre_norm=False)
    assert blew_up_at is not None and blew_up_at < 30, rms_plain
    # before the overflow the growth is faster than geometric
    assert rms_plain[-1] > 1e6 * rms_plain[0]
    finite_until, rms_norm = _run(cfg, x, blew_up_at + 1, pre_norm=True)
    assert finite_until is None
    assert rms_norm[-1] < 4.0 * rms_norm[0], rms_norm
