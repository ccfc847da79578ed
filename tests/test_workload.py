"""The seeded input generator: determinism, recipe statistics, structure."""
import numpy as np

import workload as W


def test_same_seed_same_bytes_and_streams_differ():
    cfg = W.CONFIGS["tiny"]
    a = W.expert(cfg, 0, 3)
    b = W.expert(cfg, 0, 3)
    c = W.expert(cfg, 0, 4)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["gate_q"], c["gate_q"])
    assert not np.array_equal(a["gate_q"], a["up_q"])


def test_thread_count_does_not_change_bytes():
    cfg = W.CONFIGS["tiny"]
    lib = W._hostlib()
    out = []
    for nt in (1, 3, 8):
        q = np.empty((96, 64), np.uint8)
        s = np.empty((96, 4), np.uint16)
        lib.gen_quant_matrix(0, 1, 0, W.T_DOWN, 2, 96, 128, 0.02, q.ctypes.data, s.ctypes.data, nt)
        out.append((q, s))
    for q, s in out[1:]:
        assert np.array_equal(q, out[0][0]) and np.array_equal(s, out[0][1])


def test_normal_sampler_moments():
    key = W._hostlib().gen_key_u64(0, 9, 0, 1, 0)
    z = np.array([W._hostlib().gen_normal_f(key, i) for i in range(100000)])
    assert abs(z.mean()) < 0.02 and abs(z.std() - 1) < 0.02
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(kurt - 3) < 0.1


def test_slot_table_is_a_permutation_and_bias_is_log_zipf():
    cfg = W.CONFIGS["decode125b"]
    t = W.slot_table(cfg, 5)
    assert sorted(t) == list(range(cfg.n_experts)) and not np.array_equal(t, np.arange(512))
    _, b = W.router(cfg, 5)
    # b_e = -1.1 ln(rank_e) with ranks a permutation of 1..E
    ranks = np.exp(-b.astype(np.float64) / 1.1)
    assert np.allclose(np.sort(ranks), np.arange(1, 513), rtol=1e-5)
    assert np.array_equal(W.slot_table(W.CONFIGS["decode35b"], 0), np.arange(256))


def test_drafts_are_token0_plus_noise():
    cfg = W.CONFIGS["mtp35b"]
    x = W.bf16_bits_to_f32(W.activations(cfg, 2)).astype(np.float64)
    d = x[1:] - x[0]
    assert abs(d.std() - cfg.draft_sigma) < 0.05 * cfg.draft_sigma
    x2 = W.activations(W.CONFIGS["decode35b"], 2)
    assert x2.shape == (1, 2048)
