"""GPU parity of the cache build: the indexer-key projection (512 -> 128 of an
entry's latent) on the tensor cores against the oracle, and csa2_build_cache
(pooling, main-cache records, keys and key records, in chunks) against the
oracle's composition, through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen import inputs as G  # noqa: E402
from tests.parity import unswizzle_idx_nibbles  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _dev(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16, np.uint16).view(np.int16)).cuda()


def _host_bits(t):
    return t.cpu().numpy().view(np.uint16)


def _weights(seed):
    # N(0, 1/512) weights in bf16, so that keys are of the latents' size
    w = G.bf16_bits_to_f32(G.normal_rows_bf16(seed, 9, 0, np.arange(128), 512)) / np.float32(np.sqrt(512.0))
    return G._f32_to_bf16_bits(w)


def _within_one_ulp(got, ref, x, w):
    """bf16 keys from fp32 accumulation against the oracle's single rounding of
    the exact sum: at most one bf16 step apart, plus the fp32 accumulation
    error bound over the 512 products (2^-14 of the sum of their magnitudes,
    which matters where the products cancel).  Returns the share of keys that
    are equal."""
    g = G.bf16_bits_to_f32(got).astype(np.float64)
    r = G.bf16_bits_to_f32(ref).astype(np.float64)
    mag = np.abs(G.bf16_bits_to_f32(x).astype(np.float64)) @ np.abs(G.bf16_bits_to_f32(w).astype(np.float64)).T
    tol = np.maximum(np.abs(r), np.abs(g)) * 2.0 ** -7 + mag * 2.0 ** -14
    assert np.all(np.abs(g - r) <= tol), float(np.max(np.abs(g - r) - tol))
    return float(np.mean(got == ref))


@pytest.mark.parametrize("rows", [1, 1000, 40_003])
def test_index_key_projection_parity(lib, oracle_lib, rows):
    """Ragged tiles (rows not a multiple of 128) and more tiles than SMs."""
    x = G.normal_rows_bf16(81, 1, 0, np.arange(rows), 512)
    w = _weights(81)
    out = torch.full((rows, 128), -1, dtype=torch.int16, device="cuda")
    lib.csa2_index_key_proj(_dev(x), rows, _dev(w), out)
    assert lib.csa2_get_device_status() == 0
    got = _host_bits(out)
    same = _within_one_ulp(got, oracle_lib.project_keys(x, w), x, w)
    assert same > 0.99, same


def test_index_key_projection_exact_cases(lib, oracle_lib):
    """A selection matrix picks channels exactly (one nonzero product per key),
    and small-integer sums are exact in fp32, so their one rounding to bf16 is
    the only one: bit for bit."""
    rng = np.random.default_rng(3)
    x = G.normal_rows_bf16(82, 1, 0, np.arange(300), 512)
    perm = rng.permutation(512)[:128]
    w = np.zeros((128, 512), np.float32)
    w[np.arange(128), perm] = 1.0
    out = torch.empty((300, 128), dtype=torch.int16, device="cuda")
    lib.csa2_index_key_proj(_dev(x), 300, _dev(G._f32_to_bf16_bits(w)), out)
    assert np.array_equal(_host_bits(out), x[:, perm])
    xi = rng.integers(-8, 9, size=(300, 512)).astype(np.float32)
    wi = rng.integers(-2, 3, size=(128, 512)).astype(np.float32)
    lib.csa2_index_key_proj(_dev(G._f32_to_bf16_bits(xi)), 300, _dev(G._f32_to_bf16_bits(wi)), out)
    assert np.array_equal(_host_bits(out), G._f32_to_bf16_bits((xi @ wi.T).astype(np.float32)))
    assert lib.csa2_get_device_status() == 0


def _build(lib, toks, z, w, m):
    n_tok = toks.shape[0]
    n_e = n_tok // m
    kv = torch.zeros((n_e, 288), dtype=torch.uint8, device="cuda")
    nib = torch.zeros((n_e, 64), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((n_e, 4), dtype=torch.uint8, device="cuda")
    wsb = lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, n_tok, m)
    ws = torch.full((wsb,), 0xA5, dtype=torch.uint8, device="cuda")
    zd = torch.from_numpy(np.ascontiguousarray(z, np.float32)).cuda() if z is not None else None
    lib.csa2_build_cache(toks, n_tok, m, zd, w, kv, nib, sc, ws, wsb)
    assert lib.csa2_get_device_status() == 0
    idx = np.concatenate([unswizzle_idx_nibbles(nib.cpu().numpy()), sc.cpu().numpy()], axis=1)
    return kv.cpu().numpy(), idx


@pytest.mark.parametrize("m", [1, 2])
def test_build_cache_parity(lib, oracle_lib, m):
    """A prompt of 2 x 140,008 / 140,008 tokens: two chunks of entries, the
    second ragged.  Main-cache records bit for bit against the oracle; keys within one
    bf16 step of the oracle's, and their records exactly the packing of the
    keys this GPU computes for the same latents."""
    n_e = 140_008
    n_tok = n_e * m
    toks = G.normal_rows_bf16(83, 1, 0, np.arange(n_tok), 512)
    z = G.gate_logits_f32(83, 0, np.arange(n_tok)) if m == 2 else None
    w = _weights(83)
    kv, idx = _build(lib, _dev(toks), z, _dev(w), m)
    ref = oracle_lib.build_cache(toks, z, w, m)
    assert np.array_equal(kv, ref["kv"])
    keys = torch.empty((n_e, 128), dtype=torch.int16, device="cuda")
    lib.csa2_index_key_proj(_dev(ref["latent"]), n_e, _dev(w), keys)   # the pooled latents are bit-exact
    gk = _host_bits(keys)
    assert _within_one_ulp(gk, ref["keys"], ref["latent"], w) > 0.99
    assert np.array_equal(idx, oracle_lib.pack_idx(gk))


def test_build_cache_of_a_million_token_prompt_sampled(lib, oracle_lib):
    """A 1,048,576-token encoder prompt (m = 2: 524,288 entries, 4 chunks) on
    the device; entries sampled across the chunks and at both ends checked
    against the oracle's composition of their own tokens."""
    n_tok = 1 << 20
    g = torch.Generator(device="cuda").manual_seed(84)
    toks = torch.randn((n_tok, 512), generator=g, device="cuda").to(torch.bfloat16)
    z = torch.randn((n_tok, 512), generator=g, device="cuda")
    w = _weights(84)
    n_e = n_tok // 2
    kv = torch.zeros((n_e, 288), dtype=torch.uint8, device="cuda")
    nib = torch.zeros((n_e, 64), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((n_e, 4), dtype=torch.uint8, device="cuda")
    wsb = lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, n_tok, 2)
    ws = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
    lib.csa2_build_cache(toks, n_tok, 2, z, _dev(w), kv, nib, sc, ws, wsb)
    assert lib.csa2_get_device_status() == 0
    ents = np.unique(np.concatenate([[0, 1, 7, 8, 131071, 131072, 131079, 262144, n_e - 8, n_e - 1],
                                     np.random.default_rng(84).integers(0, n_e, 48)]))
    # whole 8-row groups of the key plane, so that the swizzle undoes exactly
    groups = np.unique(ents // 8)
    rows = (groups[:, None] * 8 + np.arange(8)).reshape(-1)
    tok_rows = np.stack([2 * rows, 2 * rows + 1], axis=1).reshape(-1)
    t_idx = torch.from_numpy(tok_rows).cuda()
    tb = toks.index_select(0, t_idx).cpu().view(torch.int16).numpy().view(np.uint16)
    zb = z.index_select(0, t_idx).cpu().numpy()
    ref = oracle_lib.build_cache(tb, zb, w, 2)
    r_idx = torch.from_numpy(rows).cuda()
    assert np.array_equal(kv.index_select(0, r_idx).cpu().numpy(), ref["kv"])
    keys = torch.empty((rows.size, 128), dtype=torch.int16, device="cuda")
    lib.csa2_index_key_proj(_dev(ref["latent"]), rows.size, _dev(w), keys)
    gk = _host_bits(keys)
    assert _within_one_ulp(gk, ref["keys"], ref["latent"], w) > 0.99
    got = np.concatenate([unswizzle_idx_nibbles(nib.index_select(0, r_idx).cpu().numpy()),
                          sc.index_select(0, r_idx).cpu().numpy()], axis=1)
    assert np.array_equal(got, oracle_lib.pack_idx(gk))
