"""Pins of the oracle's path steps: indexer-score special cases, top-k and
pool against brute force and invariants, sparse attention against textbook
dense attention (torch SDPA in fp64) and RoPE closed forms."""
import numpy as np
import pytest
import torch

from gen import inputs as G
from gen.workloads import Workload, small, CONFIGS

OCP_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _decode_idx_np(rec):
    """Independent decode of logical 68-byte records (nibbles + E8M0)."""
    rec = np.asarray(rec, np.uint8).reshape(-1, 68)
    nib = np.stack([rec[:, :64] & 15, rec[:, :64] >> 4], axis=2).reshape(-1, 128)
    v = OCP_E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    return v * np.repeat(2.0 ** (rec[:, 64:].astype(np.float64) - 127), 32, axis=1)


def _decode_kv_np(rec):
    rec = np.asarray(rec, np.uint8).reshape(-1, 288)
    nib = np.stack([rec[:, :256] & 15, rec[:, :256] >> 4], axis=2).reshape(-1, 512)
    v = OCP_E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    s = torch.from_numpy(rec[:, 256:].copy()).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(s, 16, axis=1)


def _decode_swa_np(rec):
    rec = np.asarray(rec, np.uint8).reshape(-1, 528)
    v = torch.from_numpy(rec[:, :512].copy()).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(2.0 ** (rec[:, 512:].astype(np.float64) - 127), 32, axis=1)


@pytest.fixture(scope="module")
def idx_data(oracle_lib):
    keys = oracle_lib.pack_idx(G.normal_block_bf16(21, G.S_MISC, 0, 0, 300, 128))
    q = oracle_lib.pack_idx(G.normal_block_bf16(21, G.S_MISC, 1, 0, 32, 128))
    return keys, q


# ------------------------------------------------------------ indexer score
def test_score_one_head_is_relu_of_dot(oracle_lib, idx_data):
    keys, q = idx_data
    kd, qd = _decode_idx_np(keys), _decode_idx_np(q)
    for h in (0, 7, 31):
        w = np.zeros(32, np.float32)
        w[h] = 1.0
        s = oracle_lib.index_score(keys, q, w)
        assert np.array_equal(s, np.maximum(0.0, kd @ qd[h]))


def test_score_relu_kills_negative_heads(oracle_lib, idx_data):
    keys, _ = idx_data
    # every query head is the negated key 0 -> every head's dot with key 0 is < 0
    neg = keys[0].copy()
    neg[:64] ^= 0x88                           # flip the sign bit of every nibble
    q = np.tile(neg, (32, 1))
    w = G.weights_f32(21, G.S_W, 0, [0])[0]
    s = oracle_lib.index_score(keys[:1], q, w)
    assert s[0] == 0.0
    pos = np.tile(keys[0], (32, 1))            # all heads equal key 0 -> sum(w) * |k|^2
    s = oracle_lib.index_score(keys[:1], pos, w)
    k = _decode_idx_np(keys[:1])[0]
    assert np.isclose(s[0], float(np.sum(w.astype(np.float64))) * float(k @ k), rtol=1e-14)


def test_score_linear_in_weights_and_head_permutation(oracle_lib, idx_data):
    keys, q = idx_data
    w1 = G.weights_f32(22, G.S_W, 0, [0])[0]
    w2 = G.weights_f32(22, G.S_W, 1, [0])[0]
    s1, s2 = oracle_lib.index_score(keys, q, w1), oracle_lib.index_score(keys, q, w2)
    assert np.array_equal(oracle_lib.index_score(keys, q, 2 * w1), 2 * s1)      # exact scaling
    s12 = oracle_lib.index_score(keys, q, (w1 + w2).astype(np.float32))
    assert np.allclose(s12, s1 + s2, rtol=1e-6, atol=1e-6 * np.abs(s1 + s2).max())
    perm = np.random.default_rng(0).permutation(32)
    sp = oracle_lib.index_score(keys, q[perm], w1[perm])
    assert np.allclose(sp, s1, rtol=1e-13, atol=1e-13)


def test_score_uses_weight_per_head_not_per_channel(oracle_lib, idx_data):
    keys, q = idx_data
    kd, qd = _decode_idx_np(keys), _decode_idx_np(q)
    w = G.weights_f32(23, G.S_W, 0, [0])[0]
    s = oracle_lib.index_score(keys, q, w)
    want = np.maximum(0.0, kd @ qd.T) @ w.astype(np.float64)   # [n,32] relu'd dots times w
    assert np.allclose(s, want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ top-k
def _brute_topk(s, k):
    order = sorted(range(len(s)), key=lambda j: (-s[j], j))[:k]
    out = sorted(order) + [-1] * (k - min(k, len(s)))
    return np.array(out, np.int32)


@pytest.mark.parametrize("n,k,levels", [(2000, 512, 0), (2000, 512, 37), (300, 512, 5), (0, 512, 0),
                                        (513, 512, 0), (512, 512, 3), (5000, 64, 2)])
def test_topk_vs_full_sort(oracle_lib, n, k, levels):
    s = G.uniform_f32_scores(31, n, n, levels).astype(np.float64)
    assert np.array_equal(oracle_lib.topk(s, k), _brute_topk(list(s), k))


def test_topk_negative_zero_ties_positive_zero(oracle_lib):
    s = np.array([0.0, -0.0, 0.0, -1.0, -0.0])
    assert np.array_equal(oracle_lib.topk(s, 2), np.array([0, 1], np.int32))


def test_pool_blocks_brute_force_and_superset(oracle_lib):
    n = 20000 + 5                                  # ragged last block
    s = G.uniform_f32_scores(32, 0, n).astype(np.float64)
    blocks = oracle_lib.pool_blocks(s, 8, 2048)
    bmax = [max(s[8 * b: min(n, 8 * b + 8)]) for b in range((n + 7) // 8)]
    assert np.array_equal(blocks, _brute_topk(bmax, 2048))
    top = oracle_lib.topk(s, 512)
    assert set((top // 8).tolist()) <= set(blocks.tolist())      # pool contains the Full top-512


def test_pool_is_whole_cache_when_small(oracle_lib):
    n = 16384 - 3
    s = G.uniform_f32_scores(33, 0, n).astype(np.float64)
    blocks = oracle_lib.pool_blocks(s, 8, 2048)
    assert np.array_equal(blocks, np.arange(2048, dtype=np.int32))


# ------------------------------------------------------------ attention
def _rope_forward(o, pos, base=10000.0, off=448, rdim=64):
    """Textbook RoPE (RoFormer): rotate adjacent pairs by +pos * base^(-2i/d)."""
    o = o.copy()
    for i in range(rdim // 2):
        th = pos * base ** (-2.0 * i / rdim)
        a, b = o[..., off + 2 * i].copy(), o[..., off + 2 * i + 1].copy()
        o[..., off + 2 * i] = a * np.cos(th) - b * np.sin(th)
        o[..., off + 2 * i + 1] = a * np.sin(th) + b * np.cos(th)
    return o


def _attn_inputs(oracle_lib, seed, n_sel, n_swa):
    q = G.normal_block_bf16(seed, G.S_MISC, 0, 0, 64, 512)
    kv = oracle_lib.pack_kv(G.normal_block_bf16(seed, G.S_MISC, 1, 0, max(n_sel, 1), 512))[:n_sel]
    sw = oracle_lib.pack_swa(G.normal_block_bf16(seed, G.S_MISC, 2, 0, max(n_swa, 1), 512))[:n_swa]
    return q, kv, sw


@pytest.mark.parametrize("n_sel,n_swa,pos", [(512, 128, 1000), (37, 0, 5), (0, 17, 99), (300, 128, 0)])
def test_sparse_attn_equals_dense_sdpa(oracle_lib, n_sel, n_swa, pos):
    q, kv, sw = _attn_inputs(oracle_lib, 40 + n_sel, n_sel, n_swa)
    got = oracle_lib.sparse_attn(q, kv, sw, pos)
    K = np.concatenate([_decode_kv_np(kv), _decode_swa_np(sw)], axis=0)
    qf = torch.from_numpy(G.bf16_bits_to_f32(q).astype(np.float64)).view(1, 64, 1, 512)
    Kt = torch.from_numpy(K).view(1, 1, -1, 512).expand(1, 64, -1, 512)
    o = torch.nn.functional.scaled_dot_product_attention(qf, Kt, Kt, scale=1 / np.sqrt(512)).view(64, 512).numpy()
    assert np.allclose(_rope_forward(got, pos), o, rtol=1e-10, atol=1e-12)


def test_single_entry_returns_unrotated_entry(oracle_lib):
    q, kv, _ = _attn_inputs(oracle_lib, 50, 1, 0)
    for pos in (0, 1, 4095, 1048575):
        got = oracle_lib.sparse_attn(q, kv, np.zeros((0, 528), np.uint8), pos)
        k = _decode_kv_np(kv)[0]
        assert np.allclose(_rope_forward(got, pos), np.tile(k, (64, 1)), rtol=0, atol=1e-9 * np.abs(k).max())
        if pos == 0:
            assert np.array_equal(got, np.tile(k, (64, 1)))       # position 0: identity, exact
        # dims outside the RoPE range are untouched and exact
        assert np.array_equal(got[:, :448], np.tile(k[:448], (64, 1)))


def test_attention_order_of_entries_irrelevant(oracle_lib):
    q, kv, sw = _attn_inputs(oracle_lib, 51, 100, 20)
    a = oracle_lib.sparse_attn(q, kv, sw, 77)
    p = np.random.default_rng(1).permutation(100)
    b = oracle_lib.sparse_attn(q, kv[p], sw, 77)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ compositions
def test_decode_query_small_full_cache_is_dense(oracle_lib):
    """N <= 512: the top-512 is every entry, so decode == dense attention over
    the whole cache + window (the textbook case)."""
    wl = small(n_seq=1, n_entries=400, seed=60)
    r = oracle_lib.decode_query(wl, 0)
    assert np.array_equal(r["sel"][:400], np.arange(400)) and np.all(r["sel"][400:] == -1)


def test_reindex_small_cache_pool_equals_full(oracle_lib):
    """N <= 16,384: the pool is the whole cache, so reindex top-k == top-k of
    the Reindex layer's scores over all entries."""
    wl = small(n_seq=1, n_entries=5000, seed=61, pool=True)
    r = oracle_lib.reindex_query(wl, 0)
    s = oracle_lib.full_scores(wl, 0, reindex=True)
    assert np.array_equal(r["sel"], oracle_lib.topk(s, 512))


def test_reindex_pool_superset_of_full_topk(oracle_lib):
    wl = small(n_seq=1, n_entries=40000, seed=62, pool=True)
    r = oracle_lib.reindex_query(wl, 0)
    top = oracle_lib.topk(r["scores_full"], 512)
    assert set(top.tolist()) <= set(r["pool_pos"].tolist())
    assert len(r["pool_pos"]) == 16384 and np.all(np.diff(r["pool_pos"]) > 0)


def test_prefill_visibility_recipe():
    wl = CONFIGS[2]
    nv, pos, f, c = wl.n_vis(), wl.pos(), wl.swa_first(), wl.swa_cnt()
    assert nv[0] == 0 and nv[1] == 1 and nv[2] == 1 and nv[3] == 2 and nv[8191] == 4096
    assert c[0] == 1 and c[127] == 128 and c[8191] == 128 and f[8191] == 8191 - 127 and f[5] == 0


@pytest.mark.parametrize("pos,delta", [(0, 1), (1000, 37), (4095, 1_000_000), (1_048_575, 123_457)])
def test_rope_shift_invariance_fp64(oracle_lib, pos, delta):
    """RoPE's relative-position property, on unquantised fp64 data: rotating
    the query and every key forward by delta (textbook RoPE on dims 448..511)
    and moving the query to pos + delta leaves every logit unchanged, so after
    the output is rotated back by -(pos + delta) it equals the unshifted result.
    A wrong rotation direction, pairing or frequency fails this."""
    rng = np.random.default_rng(pos + delta)
    q = rng.standard_normal((64, 512))
    k = rng.standard_normal((200, 512))
    base = oracle_lib.attn_f64(q, k, pos)
    shifted = oracle_lib.attn_f64(_rope_forward(q, delta), _rope_forward(k, delta), pos + delta)
    assert np.allclose(shifted, base, rtol=0, atol=1e-9 * np.abs(base).max())
    # the rotation matters: shifting only the keys changes the output
    other = oracle_lib.attn_f64(q, _rope_forward(k, delta), pos + delta)
    assert np.abs(other - base).max() > 1e-6 * np.abs(base).max()


def test_attn_f64_is_sparse_attn_on_dequantised_records(oracle_lib):
    q, kv, sw = _attn_inputs(oracle_lib, 52, 90, 30)
    K = np.concatenate([_decode_kv_np(kv), _decode_swa_np(sw)], axis=0)
    a = oracle_lib.sparse_attn(q, kv, sw, 321)
    b = oracle_lib.attn_f64(G.bf16_bits_to_f32(q).astype(np.float64), K, 321)
    assert np.array_equal(a, b)


def test_decoder_step_roles(oracle_lib):
    """The decoder step's composition: every Reindex selection lies inside the
    Full layer's pool; a Reuse layer attending with its selecting layer's own
    query reproduces that layer's output exactly; and when the cache fits the
    pool (16,384 positions or fewer) a Reindex layer given the Full layer's
    indexer query selects exactly the Full layer's entries."""
    from gen.workloads import small, DECODER_LAYERS
    wl = small(n_seq=1, n_entries=40_000, seed=61)
    r = oracle_lib.decoder_step_query(wl, 0, DECODER_LAYERS)
    pool = r["pool"][r["pool"] >= 0].astype(np.int64)
    in_pool = set((pool[:, None] * 8 + np.arange(8)).reshape(-1).tolist())
    for k in range(1, 5):
        s = r["sel"][k]
        assert set(s[s >= 0].tolist()) <= in_pool
    # a Reuse layer (layer 1 borrows layer 0's selection) with layer 0's query
    a = oracle_lib.layer_attention(wl, 0, 0, r["sel"][0])
    assert np.array_equal(a, r["out"][0])
    # pool = whole cache: Reindex with the Full layer's indexer query = Full selection
    wl2 = small(n_seq=1, n_entries=12_000, seed=62)
    wl2.qidx_reindex = lambda qi, layer: wl2.qidx(qi)
    wl2.w_reindex = lambda qi, layer: wl2.w(qi)
    r2 = oracle_lib.decoder_step_query(wl2, 0, DECODER_LAYERS[:5])
    assert np.array_equal(r2["sel"][1], r2["sel"][0])
