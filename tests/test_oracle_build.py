"""Pins of the oracle's indexer-key projection (the indexer's key is a 512 ->
128 projection of the latent the main cache stores: "An infra-oriented diagram
of the DeepSeek-V4.1-Flash architecture", reading notes on the Full layer's
global KV) against constructed cases whose results follow without the
oracle's own sum: selection matrices, exact small-integer sums, a single
rounding of an inexact sum, and sign symmetry."""
import numpy as np

from gen import inputs as G


def _bf16(x):
    return G._f32_to_bf16_bits(np.asarray(x, np.float32))


def test_projection_by_a_selection_matrix_picks_channels(oracle_lib):
    """W with one 1 per row at channel perm[n]: key n is latent channel perm[n]
    exactly.  A transposed or misindexed W picks other channels."""
    rng = np.random.default_rng(1)
    x = G.normal_rows_bf16(5, 1, 0, np.arange(6), 512)
    perm = rng.permutation(512)[:128]
    w = np.zeros((128, 512), np.float32)
    w[np.arange(128), perm] = 1.0
    got = oracle_lib.project_keys(x, _bf16(w))
    assert np.array_equal(got, x[:, perm])


def test_projection_of_small_integers_is_their_exact_sum(oracle_lib):
    """Rows of W with +1 at two channels and -2 at a third, small-integer
    latents: every key is the integer sum, exact in bf16."""
    rng = np.random.default_rng(2)
    xi = rng.integers(-8, 9, size=(4, 512)).astype(np.float32)
    w = np.zeros((128, 512), np.float32)
    a, b, c = rng.integers(0, 512, 128), rng.integers(0, 512, 128), rng.integers(0, 512, 128)
    for n in range(128):
        w[n, a[n]] += 1.0
        w[n, b[n]] += 1.0
        w[n, c[n]] -= 2.0
    want = xi[:, a] + xi[:, b] - 2.0 * xi[:, c]
    got = G.bf16_bits_to_f32(oracle_lib.project_keys(_bf16(xi), _bf16(w)))
    assert np.array_equal(got, want.astype(np.float32))


def test_projection_rounds_once(oracle_lib):
    """1 + 2^-8 + 2^-9 lies 0.75 of a bf16 step above 1: one rounding gives
    1 + 2^-7; rounding after each addition would give 1 (the tie 1 + 2^-8 goes
    to even, then 2^-9 is lost)."""
    x = np.zeros((1, 512), np.float32)
    x[0, :3] = [1.0, 2.0 ** -8, 2.0 ** -9]
    w = np.zeros((128, 512), np.float32)
    w[:, :3] = 1.0
    got = G.bf16_bits_to_f32(oracle_lib.project_keys(_bf16(x), _bf16(w)))
    assert np.all(got == np.float32(1.0 + 2.0 ** -7))


def test_projection_is_odd_in_the_weights(oracle_lib):
    """Negating W negates every key exactly (round to nearest even is
    symmetric), and zero weights give +0 keys."""
    x = G.normal_rows_bf16(6, 1, 0, np.arange(3), 512)
    w = G.normal_rows_bf16(6, 2, 0, np.arange(128), 512)
    pos = oracle_lib.project_keys(x, w)
    neg = oracle_lib.project_keys(x, w ^ np.uint16(0x8000))
    nz = (pos & 0x7FFF) != 0
    assert np.array_equal(neg[nz], pos[nz] ^ np.uint16(0x8000))
    assert np.all(oracle_lib.project_keys(x, np.zeros((128, 512), np.uint16)) == 0)


def test_cache_build_composes_pool_pack_and_projection(oracle_lib):
    """m = 2: the main-cache records equal packing the pooled latents, and a
    gate that selects the first token of each pair (a dominant logit) makes
    the entries' keys those of the first tokens alone."""
    toks = G.normal_rows_bf16(7, 1, 0, np.arange(8), 512)
    w = G.normal_rows_bf16(7, 2, 0, np.arange(128), 512)
    z = np.zeros((8, 512), np.float32)
    z[0::2] = 200.0                                      # exp(-200) vanishes against 1 in fp64 rounding to bf16
    b = oracle_lib.build_cache(toks, z, w, 2)
    assert np.array_equal(b["latent"], toks[0::2])
    assert np.array_equal(b["kv"], oracle_lib.pack_kv(toks[0::2]))
    assert np.array_equal(b["keys"], oracle_lib.project_keys(toks[0::2], w))
    assert np.array_equal(b["idx"], oracle_lib.pack_idx(b["keys"]))
    b1 = oracle_lib.build_cache(toks, None, w, 1)
    assert np.array_equal(b1["latent"], toks) and b1["kv"].shape == (8, 288) and b1["idx"].shape == (8, 68)
