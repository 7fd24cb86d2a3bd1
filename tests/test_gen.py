"""The seeded generator: determinism, row addressability, distributions."""
import numpy as np

from gen import inputs as G
from gen.workloads import CONFIGS


def test_rows_are_addressable_and_deterministic():
    a = G.normal_block_bf16(3, G.S_LATENT, 5, 0, 64, 512)
    b = G.normal_rows_bf16(3, G.S_LATENT, 5, [10, 3, 63], 512)
    assert np.array_equal(a[[10, 3, 63]], b)
    assert np.array_equal(a, G.normal_block_bf16(3, G.S_LATENT, 5, 0, 64, 512))
    assert not np.array_equal(a, G.normal_block_bf16(3, G.S_LATENT, 6, 0, 64, 512))


def test_normal_moments_and_table():
    t = G.bf16_bits_to_f32(G.normal_table()).astype(np.float64)
    assert np.all(np.diff(t) >= 0) and np.allclose(t, -t[::-1])       # monotone, symmetric
    x = G.bf16_bits_to_f32(G.normal_block_bf16(0, G.S_LATENT, 0, 0, 2048, 512)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_zipf_rank_is_permutation():
    for n in (1000, 4096, 1 << 16):
        r = G.zipf_rank(4, 1, n, np.arange(n))
        assert np.array_equal(np.sort(r), np.arange(1, n + 1))


def test_zipf_key_norms_follow_rank():
    n = 4096
    k = G.bf16_bits_to_f32(G.zipf_keys_bf16(4, 0, n, np.arange(n))).astype(np.float64)
    r = G.zipf_rank(4, 0, n, np.arange(n))
    ratio = np.linalg.norm(k, axis=1) * r / np.sqrt(128)
    assert 0.8 < np.median(ratio) < 1.2


def test_weights_variance():
    w = G.weights_f32(0, G.S_W, 0, np.arange(4096), 32).astype(np.float64)
    assert abs(w.var() - 1 / 32) < 0.002


def test_workload_descriptors():
    c4 = CONFIGS[4]
    assert c4.n_vis()[0] == 1 << 20 and c4.pos()[0] == (1 << 20) - 1
    assert c4.swa_cnt()[0] == 128 and c4.swa_first()[0] == ((1 << 20) - 128) % 128
    c1 = CONFIGS[1]
    assert np.array_equal(c1.q_seq(), np.arange(32))
