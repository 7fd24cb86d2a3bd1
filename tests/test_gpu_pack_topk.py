"""GPU parity: generator twin, cache packing (bit-exact) and top-k (bit-exact
on identical fp32 inputs), through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen import inputs as G  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _dev_bf16(bits: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _edge_rows(width, n=12):
    """Rows with zeros, -0, bf16 subnormals, tiny/huge magnitudes, exact ties."""
    rows = np.zeros((n, width), np.float32)
    rows[1, :] = -0.0
    rows[2, :] = np.float32(2.0**-133) * np.arange(width)                  # bf16 subnormals
    rows[3, :] = np.float32(3e38) * np.cos(np.arange(width))               # near bf16 max
    rows[4, :] = np.where(np.arange(width) % 2, 1e-30, -1e-25)
    rows[5, :] = (np.arange(width) % 16) * 0.25 - 2.0                      # many exact ties
    rows[6, :] = 6.0 * 2.0 ** (np.arange(width) % 40 - 20)
    rows[7, :] = 448.0 * 2.0 ** (np.arange(width) % 7)
    rows[8, 0] = 1.0
    rows[9, :] = -1e-6
    rows[10, :] = np.linspace(-3, 3, width)
    rows[11, :] = 2.0**-126 * np.linspace(-1, 1, width)
    return G._f32_to_bf16_bits(rows)


def test_device_generator_matches_host():
    from gen.device import DeviceGen
    g = DeviceGen()
    a = g.normal_bf16(9, G.S_LATENT, 3, 100, 50, 512).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(a, G.normal_block_bf16(9, G.S_LATENT, 3, 100, 50, 512))
    for n in (1 << 20, 1000):
        k = g.zipf_keys_bf16(4, 2, n, 7, 64).view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(k, G.zipf_keys_bf16(4, 2, n, np.arange(7, 71)))
    w = g.weights_f32(5, G.S_W, 1, 0, 3).cpu().numpy()
    assert np.array_equal(w, G.weights_f32(5, G.S_W, 1, [0, 1, 2]))


@pytest.mark.parametrize("rows", [1, 37, 1000 + 3])
def test_pack_kv_bit_exact(lib, oracle_lib, rows):
    x = np.concatenate([_edge_rows(512), G.normal_block_bf16(70, G.S_MISC, rows, 0, rows, 512)])
    dst = torch.zeros((x.shape[0], 288), dtype=torch.uint8, device="cuda")
    lib.csa2_fp4_pack(lib.CSA2_KV_NVFP4, _dev_bf16(x), x.shape[0], 1, None, dst)
    assert np.array_equal(dst.cpu().numpy(), oracle_lib.pack_kv(x))


def test_pack_kv_m2_bit_exact(lib, oracle_lib):
    n = 2 * 515
    x = G.normal_block_bf16(71, G.S_MISC, 0, 0, n, 512)
    z = G.gate_logits_f32(71, 0, np.arange(n), 512)
    z[:40] = 0.0                      # equal logits: the pooled value is the exact mean (ties in bf16)
    z[40:80:2] = 90.0                 # a dominant logit
    dst = torch.zeros((n // 2, 288), dtype=torch.uint8, device="cuda")
    lib.csa2_fp4_pack(lib.CSA2_KV_NVFP4, _dev_bf16(x), n, 2, torch.from_numpy(z).cuda(), dst)
    want = oracle_lib.pack_kv(oracle_lib.pool_m2(x, z))
    assert np.array_equal(dst.cpu().numpy(), want)


@pytest.mark.parametrize("rows", [1, 33, 4096 + 5])
def test_pack_idx_bit_exact(lib, oracle_lib, rows):
    x = np.concatenate([_edge_rows(128), G.normal_block_bf16(72, G.S_MISC, rows, 0, rows, 128)])
    n = x.shape[0]
    nib = torch.zeros((n, 64), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((n, 4), dtype=torch.uint8, device="cuda")
    lib.csa2_fp4_pack(lib.CSA2_IDX_MXFP4, _dev_bf16(x), n, 1, None, nib, sc)
    from tests.parity import unswizzle_idx_nibbles
    got = np.concatenate([unswizzle_idx_nibbles(nib.cpu().numpy()), sc.cpu().numpy()], axis=1)
    assert np.array_equal(got, oracle_lib.pack_idx(x))


@pytest.mark.parametrize("rows", [1, 129])
def test_pack_swa_bit_exact(lib, oracle_lib, rows):
    x = np.concatenate([_edge_rows(512), G.normal_block_bf16(73, G.S_MISC, rows, 0, rows, 512)])
    dst = torch.zeros((x.shape[0], 528), dtype=torch.uint8, device="cuda")
    lib.csa2_fp4_pack(lib.CSA2_SWA_MXFP8, _dev_bf16(x), x.shape[0], 1, None, dst)
    assert np.array_equal(dst.cpu().numpy(), oracle_lib.pack_swa(x))


# ------------------------------------------------------------------ top-k
def _run_topk(lib, s_rows, n_valid, k, block=1, pool=None, n_max=None):
    n_q, stride = s_rows.shape
    n_max = stride if n_max is None else n_max
    scores = torch.from_numpy(np.ascontiguousarray(s_rows, np.float32)).cuda()
    nv = torch.tensor(n_valid, dtype=torch.int32, device="cuda")
    out = torch.empty((n_q, k), dtype=torch.int32, device="cuda")
    items = 16384 if pool is not None else (n_max if block == 1 else (n_max + 7) // 8)
    wsb = lib.csa2_workspace_size(lib.CSA2_OP_TOPK, n_q, items, k)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    pl = None if pool is None else torch.from_numpy(np.ascontiguousarray(pool, np.int32)).cuda()
    lib.csa2_topk(scores, stride, n_q, nv, n_max, k, block, pl, out, ws, wsb)
    assert lib.csa2_get_device_status() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("n,levels,k", [(4096, 0, 512), (5000, 7, 512), (300, 3, 512), (16384, 0, 512),
                                        (3000, 5, 512), (7000, 0, 1024),
                                        (100_000, 0, 512), (100_000, 50, 512), (1 << 20, 0, 512),
                                        (70_000, 0, 2048), (20_000, 1000, 1)])
def test_topk_bit_exact(lib, oracle_lib, n, levels, k):
    rows = np.stack([G.uniform_f32_scores(80 + i, n + levels, n, levels) for i in range(3)])
    rows[1, ::7] = -0.0 if levels else rows[1, ::7]          # negative zeros tie with +0
    nv = [n, n - 17 if n > 17 else n, max(0, n // 3)]
    got = _run_topk(lib, rows, nv, k)
    for i in range(3):
        want = oracle_lib.topk(rows[i, :nv[i]].astype(np.float64), k)
        assert np.array_equal(got[i], want), i


def test_topk_long_rows_odd_stride(lib, oracle_lib):
    """Row starts not 16-B aligned and ragged lengths: element-wise loads."""
    n, stride = 70_001, 70_003
    base = np.stack([G.uniform_f32_scores(95 + i, 1, stride, 0) for i in range(3)])
    scores = torch.from_numpy(np.ascontiguousarray(base, np.float32)).cuda()
    nv = torch.tensor([n, n - 2, 65_537], dtype=torch.int32, device="cuda")
    out = torch.empty((3, 512), dtype=torch.int32, device="cuda")
    wsb = lib.csa2_workspace_size(lib.CSA2_OP_TOPK, 3, n, 512)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    lib.csa2_topk(scores, stride, 3, nv, n, 512, 1, None, out, ws, wsb)
    assert lib.csa2_get_device_status() == 0
    got = out.cpu().numpy()
    for i, m in enumerate([n, n - 2, 65_537]):
        assert np.array_equal(got[i], oracle_lib.topk(base[i, :m].astype(np.float64), 512))


@pytest.mark.parametrize("n", [100_000, 1 << 20])
def test_topk_long_rows_negative_and_zero_thresholds(lib, oracle_lib, n):
    """Long rows whose threshold is a negative score or exactly zero (the
    streaming pass then compares order keys, not raw bits), next to an
    ordinary row; -0 and +0 tie and ties go to the smaller index."""
    neg = G.uniform_f32_scores(97, 0, n, 0) * 0.5 - 1.5               # all in [-2, -1)
    zero = np.zeros(n, np.float32)
    zero[1::2] = -0.0
    rng = np.random.default_rng(5)
    zero[rng.choice(n, 300, replace=False)] = rng.random(300).astype(np.float32) + 0.5
    rows = np.stack([neg, zero, G.uniform_f32_scores(98, 0, n, 0)])
    got = _run_topk(lib, rows, [n, n, n], 512)
    for i in range(3):
        assert np.array_equal(got[i], oracle_lib.topk(rows[i].astype(np.float64), 512)), i


def test_topk_all_equal_row_uses_exact_fallback(lib, oracle_lib):
    n = 200_000                                            # candidates overflow the filter buffer
    rows = np.zeros((2, n), np.float32)
    rows[1, 5000:] = 1.0
    got = _run_topk(lib, rows, [n, n], 512)
    assert np.array_equal(got[0], np.arange(512))
    assert np.array_equal(got[1], np.arange(5000, 5512))


@pytest.mark.parametrize("n", [1000, 20_003, 1 << 20])
def test_topk_block_mode_bit_exact(lib, oracle_lib, n):
    rows = np.stack([G.uniform_f32_scores(90, n, n, 0), G.uniform_f32_scores(91, n, n, 9)])
    got = _run_topk(lib, rows, [n, n - 3], 2048, block=8)
    for i, nv in enumerate([n, n - 3]):
        want = oracle_lib.pool_blocks(rows[i, :nv].astype(np.float64), 8, 2048)
        assert np.array_equal(got[i], want)


def test_topk_pool_mode_bit_exact(lib, oracle_lib):
    n_entries = 50_001
    rng = np.random.default_rng(3)
    pool = np.sort(rng.choice((n_entries + 7) // 8, 2048, replace=False)).astype(np.int32)
    pool2 = pool.copy()
    pool2[-100:] = -1
    s = np.stack([G.uniform_f32_scores(92, 0, 16384, 0), G.uniform_f32_scores(93, 0, 16384, 11)])
    got = _run_topk(lib, s, [n_entries, n_entries], 512, pool=np.stack([pool, pool2]), n_max=n_entries + 7)
    for i, pl in enumerate([pool, pool2]):
        pos = (pl[:, None].astype(np.int64) * 8 + np.arange(8)).reshape(-1)
        ok = (np.repeat(pl, 8) >= 0) & (pos < n_entries)
        loc = oracle_lib.topk(s[i][ok].astype(np.float64), 512)
        want = np.where(loc >= 0, pos[ok][np.maximum(loc, 0)], -1)
        assert np.array_equal(got[i], want)


def test_bad_pool_block_sets_bounds_status(lib):
    s = np.zeros((1, 16384), np.float32)
    pool = np.full((1, 2048), -1, np.int32)
    pool[0, 0] = 10**8                                      # beyond the cache
    out = torch.empty((1, 512), dtype=torch.int32, device="cuda")
    lib.csa2_topk(torch.from_numpy(s).cuda(), 16384, 1, torch.tensor([1000], dtype=torch.int32, device="cuda"), 1024,
                  512, 1, torch.from_numpy(pool).cuda(), out, None, 0)
    assert lib.csa2_get_device_status() == 4               # CSA2_ERR_BOUNDS
    assert np.all(out.cpu().numpy() == -1)
    assert lib.csa2_get_device_status() == 0               # cleared by the read
