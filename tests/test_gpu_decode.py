"""GPU parity of the decode path (indexer score -> top-512 -> sparse attention)
against the CPU oracle, through the C ABI, on the pages' workload shapes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen.workloads import CONFIGS, Workload, small  # noqa: E402
from tests.parity import (ATTN_TOL_BF16, ATTN_TOL_F32, check_scores, check_selection,  # noqa: E402
                          row_norm_err)


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _dw(wl, n_q=None):
    from gen.device import build_device_workload
    return build_device_workload(wl, n_q=n_q)


def _bufs(dw, pool=False, out_dtype=None):
    from compressed_sparse_attention_index_gb300 import decode, CSA2_OUT_F32
    return decode.DecodeBuffers(dw.q.shape[0], dw.n_max, pool=pool,
                                out_dtype=CSA2_OUT_F32 if out_dtype is None else out_dtype)


@pytest.mark.parametrize("zipf", [False, True])
def test_index_score_full_parity(lib, oracle_lib, zipf):
    wl = small(n_seq=2, n_entries=1000, zipf=zipf, seed=200 + zipf)
    dw = _dw(wl)
    buf = _bufs(dw)
    lib.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, 2, dw.q_nib, dw.q_scale, dw.w, dw.q_seq, dw.n_vis, 2,
                         None, buf.scores, dw.n_max)
    s = buf.scores.cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    for qi in range(2):
        check_scores(s[qi, :1000], oracle_lib.full_scores(wl, qi))


def test_index_score_runs_of_units_across_queries(lib, oracle_lib):
    """More units than SMs and nothing claimed: each CTA takes runs of
    consecutive units (here 40 queries x 10 units over at most 152 CTAs, runs
    of 3 that cross from one query into the next), with ragged visible
    lengths (the last unit of every query partly visible)."""
    wl = small(n_seq=4, n_entries=5000, seed=207, q_per_seq=10)
    dw = _dw(wl)
    buf = _bufs(dw)
    n_q = dw.q.shape[0]
    lib.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, 4, dw.q_nib, dw.q_scale, dw.w, dw.q_seq, dw.n_vis, n_q,
                         None, buf.scores, dw.n_max)
    s = buf.scores.cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    nv = wl.n_vis()
    for qi in range(n_q):
        check_scores(s[qi, :nv[qi]], oracle_lib.full_scores(wl, qi))


def test_index_score_pool_mode_gather(lib, oracle_lib):
    """Pool mode: each 512-entry unit is 64 gathered 8-entry blocks, moved by
    four warps of 16 blocks each.  Empty slots (-1) fall in every warp's share,
    the last block of the cache is ragged (entries past n_vis score -inf), and
    a block beyond the cache is skipped and reported."""
    wl = small(n_seq=2, n_entries=40_003, seed=240)
    dw = _dw(wl)
    n_blocks = (40_003 + 7) // 8
    rng = np.random.default_rng(11)
    pool = np.stack([np.sort(rng.choice(n_blocks, 2048, replace=False)) for _ in range(2)]).astype(np.int32)
    pool[0, -1] = n_blocks - 1                          # the ragged last block
    pool[1, 3::7] = -1                                  # holes in every 16-block share
    pool[1, 2047] = n_blocks + 100                      # beyond the cache: skipped, reported
    scores = torch.empty((2, 16384), dtype=torch.float32, device="cuda")
    lib.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, 2, dw.q_nib, dw.q_scale, dw.w, dw.q_seq, dw.n_vis, 2,
                         torch.from_numpy(pool).cuda(), scores, 16384)
    assert lib.csa2_get_device_status() == 4            # CSA2_ERR_BOUNDS, then cleared
    got = scores.cpu().numpy()
    for qi in range(2):
        ref = oracle_lib.full_scores(wl, qi)
        pos = (pool[qi].astype(np.int64)[:, None] * 8 + np.arange(8)).reshape(-1)
        ok = (np.repeat(pool[qi], 8) >= 0) & (pos < 40_003)
        assert np.all(np.isneginf(got[qi][~ok])), qi
        check_scores(got[qi][ok], ref[pos[ok]])


@pytest.mark.parametrize("out_f32", [True, False])
def test_sparse_attn_parity_on_oracle_selection(lib, oracle_lib, out_f32):
    from compressed_sparse_attention_index_gb300 import decode, CSA2_OUT_F32, CSA2_OUT_BF16
    wl = small(n_seq=3, n_entries=3000, seed=210)
    dw = _dw(wl)
    buf = _bufs(dw, out_dtype=CSA2_OUT_F32 if out_f32 else CSA2_OUT_BF16)
    refs = [oracle_lib.decode_query(wl, qi) for qi in range(3)]
    sel = np.stack([r["sel"] for r in refs])
    sel[1, 100:] = -1                                   # ragged selection with holes
    sel[1, 40:60] = -1
    buf.sel.copy_(torch.from_numpy(sel))
    decode.attend(dw, buf)
    out = buf.out.float().cpu().numpy()
    tol = ATTN_TOL_F32 if out_f32 else ATTN_TOL_BF16
    from oracle.compose import kv_records, swa_records
    for qi in range(3):
        s = sel[qi][sel[qi] >= 0]
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, qi, s),
                                     swa_records(wl, qi, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])),
                                     int(wl.pos()[qi]))
        assert row_norm_err(out[qi], ref) <= tol


@pytest.mark.parametrize("n_seq,stride", [(3, 1), (3, 129), (3, 300), (48, 511)])
def test_sparse_attn_ragged_selection_stride(lib, oracle_lib, n_seq, stride):
    """sel_stride not a multiple of 128: the chunk that holds the last selected
    entries and the first window entries dequantises its FP4 latents to bf16
    (the chunks of FP4 latents only run in f16), and Q is staged in both types;
    with 48 queries a CTA takes two chunks, f16 then that bf16 one, and
    restages Q between them."""
    import compressed_sparse_attention_index_gb300 as C
    wl = small(n_seq=n_seq, n_entries=3000 if n_seq == 3 else 1500, seed=270 + stride)
    dw = _dw(wl)
    n_q = dw.q.shape[0]
    full = np.stack([oracle_lib.decode_query(wl, qi)["sel"] for qi in range(n_q)])
    sel = np.ascontiguousarray(full[:, :stride])
    sel[1, ::3] = -1                                    # holes as well
    out = torch.empty((n_q, 64, 512), dtype=torch.float32, device="cuda")
    ws_bytes = C.csa2_workspace_size(C.CSA2_OP_SPARSE_ATTN, n_q, stride + 128)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    C.csa2_sparse_attn(dw.q, dw.kv, dw.n_max, dw.kv.shape[0], torch.from_numpy(sel).cuda(), stride, dw.swa,
                       dw.swa.shape[1], dw.q_seq, dw.pos, dw.swa_first, dw.swa_cnt, n_q, out, C.CSA2_OUT_F32, None,
                       ws, ws_bytes)
    got = out.cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    from oracle.compose import kv_records, swa_records
    for qi in range(n_q):
        s_ = sel[qi][sel[qi] >= 0]
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, qi, s_),
                                     swa_records(wl, qi, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])),
                                     int(wl.pos()[qi]))
        assert row_norm_err(got[qi], ref) <= ATTN_TOL_F32


@pytest.mark.parametrize("e", [-40, 40])
def test_sparse_attn_query_scale_invariance(lib, oracle_lib, e):
    """q x 2^e with sm_scale x 2^-e gives the same logits.  The selected
    (FP4-only) chunks run in f16 with Q shifted by the power of two that puts
    max |q| in [2^14, 2^15), the window chunk in bf16 with Q as given: both must
    undo the shift, for huge and for tiny queries alike."""
    from compressed_sparse_attention_index_gb300 import decode, default_params
    wl = small(n_seq=2, n_entries=3000, seed=260)
    dw = _dw(wl)
    buf = _bufs(dw)
    sel = np.stack([oracle_lib.decode_query(wl, qi)["sel"] for qi in range(2)])
    buf.sel.copy_(torch.from_numpy(sel))
    decode.attend(dw, buf)
    base = buf.out.float().cpu().numpy()
    dw.q.mul_(2.0 ** e)                                 # exact in bf16 at this range
    p = default_params()
    p.sm_scale = p.sm_scale * 2.0 ** -e
    decode.attend(dw, buf, params=p)
    out = buf.out.float().cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    from oracle.compose import kv_records, swa_records
    for qi in range(2):
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, qi, sel[qi][sel[qi] >= 0]),
                                     swa_records(wl, qi, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])),
                                     int(wl.pos()[qi]))
        assert row_norm_err(out[qi], ref) <= ATTN_TOL_F32
        assert row_norm_err(out[qi], base[qi]) <= 1e-6


def _check_full(lib, oracle_lib, wl, dw, buf, queries, fused=False):
    from compressed_sparse_attention_index_gb300 import decode
    (decode.fused_decode if fused else decode.full_decode)(dw, buf)
    sel = buf.sel.cpu().numpy()
    out = buf.out.float().cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    worst = 0.0
    for qi in queries:
        r = oracle_lib.decode_query(wl, qi)
        check_selection(sel[qi], r["sel"], r["scores"])
        # attention is compared on the GPU's own selection (equal up to near-ties)
        from oracle.compose import kv_records, swa_records
        s = sel[qi][sel[qi] >= 0]
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, int(wl.q_seq()[qi]), s),
                                     swa_records(wl, int(wl.q_seq()[qi]), int(wl.swa_first()[qi]),
                                                 int(wl.swa_cnt()[qi])), int(wl.pos()[qi]))
        worst = max(worst, row_norm_err(out[qi], ref))
    assert worst <= ATTN_TOL_F32, worst
    return worst


def test_full_decode_config0(lib, oracle_lib):
    wl = CONFIGS[0]
    dw = _dw(wl)
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0])


@pytest.mark.parametrize("n_entries", [300, 1000, 5003])
def test_full_decode_small_ragged(lib, oracle_lib, n_entries):
    wl = small(n_seq=2, n_entries=n_entries, seed=220 + n_entries)
    dw = _dw(wl)
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0, 1])


def test_full_decode_config1_sampled(lib, oracle_lib):
    wl = CONFIGS[1]
    dw = _dw(wl)
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0, 17, 31])


def test_full_decode_config4_full_size_sampled(lib, oracle_lib):
    wl = CONFIGS[4]
    dw = _dw(wl)
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0, 7])
    # the one-call decode, whose attention starts from the candidate handoff
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0, 3, 7], fused=True)


def test_fused_decode_small_batch_of_64k_rows(lib, oracle_lib):
    """Four queries over 65,536-entry caches: the one-call decode on the
    32-entry group plan, whose attention takes the candidates when they fit
    (and the final selection otherwise), against the oracle."""
    wl = small(n_seq=4, n_entries=65536, zipf=True, seed=254)
    dw = _dw(wl)
    _check_full(lib, oracle_lib, wl, dw, _bufs(dw), [0, 1, 2, 3], fused=True)


def _check_reindex(lib, oracle_lib, wl, blocks, sel, out, qi):
    """The pool (blocks of 8) against the oracle's under the near-tie rule on
    block scores; the Reindex selection against the oracle's Reindex step run
    on the GPU's own pool (so a legal near-tie swap of a pool block cannot hide
    the selection from the check); the attention on the GPU's selection."""
    from oracle.compose import kv_records, swa_records
    r = oracle_lib.reindex_query(wl, qi)
    n = int(wl.n_vis()[qi])
    bscore = lambda b: max(r["scores_full"][8 * b:min(n, 8 * b + 8)])
    check_selection(blocks, r["blocks"], None, pos_to_score=bscore)
    rp = r if np.array_equal(blocks, r["blocks"]) else oracle_lib.reindex_on_pool(wl, qi, blocks)
    pos_score = dict(zip(rp["pool_pos"].tolist(), rp["scores_pool"].tolist()))
    check_selection(sel, rp["sel"], None, pos_to_score=lambda p: pos_score[p])
    if out is not None:
        seq = int(wl.q_seq()[qi])
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, seq, sel[sel >= 0]),
                                     swa_records(wl, seq, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])),
                                     int(wl.pos()[qi]))
        assert row_norm_err(out, ref) <= ATTN_TOL_F32


def test_reindex_decode_small(lib, oracle_lib):
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=2, n_entries=40_000, pool=True, seed=230)
    dw = _dw(wl)
    buf = _bufs(dw, pool=True)
    decode.reindex_decode(dw, buf)
    blocks, sel, out = buf.blocks.cpu().numpy(), buf.sel.cpu().numpy(), buf.out.float().cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    for qi in range(2):
        _check_reindex(lib, oracle_lib, wl, blocks[qi], sel[qi], out[qi], qi)


def test_reindex_on_a_pool_with_near_ties_swapped(lib, oracle_lib):
    """The Reindex step is checked on whatever pool it is given: here the
    GPU's pool with its last-ranked block replaced by another one, as a legal
    near-tie swap would, and the selection still matches the oracle's Reindex
    step on that same pool."""
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=2, n_entries=40_000, pool=True, seed=231)
    dw = _dw(wl)
    buf = _bufs(dw, pool=True)
    decode.reindex_decode(dw, buf)
    blocks = buf.blocks.cpu().numpy()
    r = oracle_lib.reindex_query(wl, 1)
    s_full = r["scores_full"]
    bs = np.array([s_full[8 * b:8 * b + 8].max() for b in blocks[1]])
    outside = np.setdiff1d(np.arange(5000), blocks[1])
    swapped = blocks[1].copy()
    swapped[int(np.argmin(bs))] = outside[0]
    swapped = np.sort(swapped)
    buf.blocks[1].copy_(torch.from_numpy(swapped))
    decode.reindex_decode(dw, buf, build_pool=False)
    sel, out = buf.sel.cpu().numpy(), buf.out.float().cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    rp = oracle_lib.reindex_on_pool(wl, 1, swapped)
    pos_score = dict(zip(rp["pool_pos"].tolist(), rp["scores_pool"].tolist()))
    check_selection(sel[1], rp["sel"], None, pos_to_score=lambda p: pos_score[p])
    from oracle.compose import kv_records, swa_records
    ref = oracle_lib.sparse_attn(wl.q(1), kv_records(wl, 1, sel[1][sel[1] >= 0]),
                                 swa_records(wl, 1, int(wl.swa_first()[1]), int(wl.swa_cnt()[1])), int(wl.pos()[1]))
    assert row_norm_err(out[1], ref) <= ATTN_TOL_F32


def test_reindex_decode_config3_full_size_sampled(lib, oracle_lib):
    """64 x 1,048,576 Reindex decode: the pool, the Reindex selection and the
    attention output (64 queries: the split plan with several chunks per CTA,
    FP4-only chunks in f16 beside the window's chunk in bf16) for sampled
    queries."""
    from compressed_sparse_attention_index_gb300 import decode
    wl = CONFIGS[3]
    dw = _dw(wl)
    buf = _bufs(dw, pool=True)
    decode.reindex_decode(dw, buf)
    blocks, sel, out = buf.blocks.cpu().numpy(), buf.sel.cpu().numpy(), buf.out.float().cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    for qi in (5, 63):
        _check_reindex(lib, oracle_lib, wl, blocks[qi], sel[qi], out[qi], qi)


@pytest.mark.parametrize("case", ["pool_40k", "short_3000", "equal_scores", "config3"])
def test_fused_reindex_equals_chain(lib, oracle_lib, case):
    """csa2_decode_reindex (the pool-mode indexer writing block maxima, the
    selection reading only the blocks that reach the 512th largest of them,
    the attention staged during the selection) against the chain
    csa2_index_score -> csa2_topk -> csa2_sparse_attn on the same pool:
    selection bit for bit, output bit for bit where the split plans agree.  short_3000: a pool of 375 valid blocks
    (fewer than 512 blocks: every valid block is read); equal_scores: zero
    head weights, every score equal, all 2,048 block maxima tie (more items
    than the candidate buffer: the whole row is read); config3: 64 x 1M, with
    sampled queries also against the oracle."""
    from compressed_sparse_attention_index_gb300 import decode
    wl = {"pool_40k": small(n_seq=2, n_entries=40_000, pool=True, seed=232),
          "short_3000": small(n_seq=2, n_entries=3000, pool=True, seed=233),
          "equal_scores": small(n_seq=2, n_entries=40_000, pool=True, seed=234),
          "config3": CONFIGS[3]}[case]
    dw = _dw(wl)
    if case == "equal_scores":
        dw.w_re.zero_()
    buf = _bufs(dw, pool=True)
    decode.reindex_decode(dw, buf)                      # the pool, then the chain on it
    sel_c, out_c = buf.sel.clone(), buf.out.clone()
    buf.sel.fill_(-7)
    buf.out.fill_(7.0)
    decode.fused_reindex_decode(dw, buf)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(buf.sel, sel_c)
    if case == "config3":
        # 64 queries: the call's attention, whose inputs are settled, runs each
        # query's window chunk first in its last split (two splits of two
        # chunks of selected entries instead of the chain's three and two), so
        # its numerators are rounded against other running maxima and its
        # partial sums merge in another grouping: equal to rounding
        for qi in range(0, 64, 9):
            assert row_norm_err(buf.out[qi].float().cpu().numpy(), out_c[qi].double().cpu().numpy()) <= 1e-3
    else:
        assert torch.equal(buf.out, out_c)
    if case == "equal_scores":                          # ties: the lowest pool positions win
        assert (buf.sel >= 0).sum().item() == 2 * 512
    if case == "config3":
        blocks, sel, out = buf.blocks.cpu().numpy(), buf.sel.cpu().numpy(), buf.out.float().cpu().numpy()
        for qi in (7, 40):
            _check_reindex(lib, oracle_lib, wl, blocks[qi], sel[qi], out[qi], qi)


def test_prefill_m2_config2_sampled(lib, oracle_lib):
    wl = CONFIGS[2]
    dw = _dw(wl)
    buf = _bufs(dw)
    _check_full(lib, oracle_lib, wl, dw, buf, [0, 1, 2, 3, 127, 128, 1023, 1024, 4095, 8191])


def test_out_of_range_selection_is_skipped_and_reported(lib, oracle_lib):
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=1, n_entries=1000, seed=240)
    dw = _dw(wl)
    buf = _bufs(dw)
    sel = np.full((1, 512), -1, np.int32)
    sel[0, :3] = [5, 10**7, 7]                          # 10**7 is beyond the cache
    buf.sel.copy_(torch.from_numpy(sel))
    decode.attend(dw, buf)
    assert lib.csa2_get_device_status() == 4
    from oracle.compose import kv_records, swa_records
    ref = oracle_lib.sparse_attn(wl.q(0), kv_records(wl, 0, [5, 7]), swa_records(wl, 0, int(wl.swa_first()[0]),
                                                                                 int(wl.swa_cnt()[0])),
                                 int(wl.pos()[0]))
    assert row_norm_err(buf.out.float().cpu().numpy()[0], ref) <= ATTN_TOL_F32


def test_empty_query_gives_zeros(lib):
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=1, n_entries=256, seed=241)
    dw = _dw(wl)
    buf = _bufs(dw)
    buf.sel.fill_(-1)
    dw.swa_cnt.zero_()
    decode.attend(dw, buf)
    assert lib.csa2_get_device_status() == 0
    assert torch.count_nonzero(buf.out).item() == 0


HAND_CAP = 640
HAND_FALLBACK = 0xFFFFFFFF


def _handoff(buf):
    """What the selection handed to the attention in the last csa2_decode call
    on buf, read from the workspace's last two regions (each 256-B aligned):
    32 words per query (0: selection CTAs that published, P; 1: selection
    final; 2-3: the smallest selected key; 8 + p: CTA p's candidate count or
    0xFFFFFFFF), then 16 x 256 candidate keys per query.  Returns
    [(counts, key)] per query."""
    r256 = lambda b: (b + 255) // 256 * 256
    n_q = buf.n_q
    start = buf.ws_decode_bytes - r256(n_q * 16 * 256 * 8) - r256(n_q * 128)
    w = buf.ws[start:start + n_q * 128].cpu().numpy().view(np.uint32).reshape(n_q, 32)
    assert np.all(w[:, 1] == 1)
    return [(w[qi, 8:8 + int(w[qi, 0])], int(w[qi, 2]) | (int(w[qi, 3]) << 32)) for qi in range(n_q)]


def _order_key(x):
    """The selection's order key of fp32 scores: unsigned order equals float order."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return np.where(b >> np.uint64(31), b ^ np.uint64(0xFFFFFFFF), b | np.uint64(0x80000000))


@pytest.mark.parametrize("case", ["small_direct", "ragged_standalone", "config1_groups", "config4_units"])
def test_fused_decode_equals_call_chain(lib, case):
    """csa2_decode (score epilogue feeds the selection) selects exactly what
    csa2_index_score -> csa2_topk selects, for each of its selection plans: one
    CTA per row, the standalone passes, 32-entry groups and 512-entry units.
    Where the attention takes the selection's candidates (8 x 1M: every query
    hands over at most 640, and the smallest selected key published is the
    512th largest key of the row), the entries sit in other chunks than in
    csa2_sparse_attn, so the output agrees with the chain's to rounding;
    elsewhere bit for bit.  Repeated calls and a garbage workspace give the
    same bits."""
    from compressed_sparse_attention_index_gb300 import decode
    wl = {"small_direct": small(n_seq=2, n_entries=1000, seed=250),
          "ragged_standalone": small(n_seq=3, n_entries=20_000, seed=251),
          "config1_groups": CONFIGS[1], "config4_units": CONFIGS[4]}[case]
    dw = _dw(wl)
    chain, fused = _bufs(dw), _bufs(dw)
    decode.full_decode(dw, chain)
    fused.sel.fill_(-7)
    fused.out.fill_(7)
    decode.fused_decode(dw, fused)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(chain.sel, fused.sel)
    handoff = case == "config4_units"
    if handoff:
        hand = _handoff(fused)
        sel = chain.sel.cpu().numpy()
        scores = chain.scores.cpu().numpy()
        for qi in range(fused.n_q):
            counts, kth = hand[qi]
            assert len(counts) >= 2 and np.all(counts != HAND_FALLBACK), counts
            assert 512 <= counts.sum() <= HAND_CAP, counts
            j = sel[qi][sel[qi] >= 0].astype(np.int64)
            keys = (_order_key(scores[qi, j]) << np.uint64(32)) | (~j.astype(np.uint64) & np.uint64(0xFFFFFFFF))
            assert kth == int(keys.min())
        err = max(row_norm_err(fused.out[qi].cpu().numpy(), chain.out[qi].cpu().numpy()) for qi in range(fused.n_q))
        assert err <= 1e-3, err
    else:
        assert torch.equal(chain.out.view(torch.int32), fused.out.view(torch.int32))
    first = fused.out.clone()
    decode.fused_decode(dw, fused)                       # second call: nothing left over from the first
    assert torch.equal(chain.sel, fused.sel)
    fused.ws.fill_(0xA5)                                 # a workspace of garbage: nothing in it is
    fused.out.fill_(7)                                   # read before this call writes it
    decode.fused_decode(dw, fused)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(chain.sel, fused.sel)
    assert torch.equal(first.view(torch.int32), fused.out.view(torch.int32))


def test_fused_decode_falls_back_to_the_final_selection(lib):
    """Rows whose candidates cannot be handed over (all scores equal: every
    entry reaches the threshold, the row is selected exactly from its scores)
    are flagged so, and the attention reads the final selection: the output
    is the chain's, bit for bit.  A query seeing fewer entries than k hands all
    of them over with the key 1 (every candidate selected)."""
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=2, n_entries=65536, seed=255)
    dw = _dw(wl)
    dw.w.zero_()                                         # every score is +0
    chain, fused = _bufs(dw), _bufs(dw)
    decode.full_decode(dw, chain)
    decode.fused_decode(dw, fused)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(chain.sel, fused.sel)
    assert all(np.any(counts == HAND_FALLBACK) for counts, _ in _handoff(fused))
    assert torch.equal(chain.out.view(torch.int32), fused.out.view(torch.int32))
    dw = _dw(wl)
    dw.n_vis[1] = 300                                    # fewer entries than k
    chain, fused = _bufs(dw), _bufs(dw)
    decode.full_decode(dw, chain)
    decode.fused_decode(dw, fused)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(chain.sel, fused.sel)
    counts, kth = _handoff(fused)[1]
    assert np.all(counts != HAND_FALLBACK) and counts.sum() == 300 and kth == 1, (counts, kth)
    err = max(row_norm_err(fused.out[qi].cpu().numpy(), chain.out[qi].cpu().numpy()) for qi in range(2))
    assert err <= 1e-3, err


def test_window_longer_than_ring_is_rejected(lib, oracle_lib):
    """A window count above the ring's capacity would wrap the ring and attend
    to some window entries twice: the query is skipped (zeros) and reported,
    while a query whose window fits the ring is served as usual."""
    import compressed_sparse_attention_index_gb300 as C
    wl = small(n_seq=2, n_entries=1000, seed=242)
    dw = _dw(wl)
    cap = 64
    swa = dw.swa[:, :cap].contiguous()                  # a 64-slot ring
    sel = np.stack([oracle_lib.decode_query(wl, qi)["sel"] for qi in range(2)])
    swa_first = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    swa_cnt = torch.tensor([128, 64], dtype=torch.int32, device="cuda")    # query 0: 128 > 64
    out = torch.full((2, 64, 512), 7.0, dtype=torch.float32, device="cuda")
    ws_bytes = C.csa2_workspace_size(C.CSA2_OP_SPARSE_ATTN, 2, 512 + 128)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    C.csa2_sparse_attn(dw.q, dw.kv, dw.n_max, 2, torch.from_numpy(sel).cuda(), 512, swa, cap, dw.q_seq, dw.pos,
                       swa_first, swa_cnt, 2, out, C.CSA2_OUT_F32, None, ws, ws_bytes)
    assert lib.csa2_get_device_status() == 4            # CSA2_ERR_BOUNDS
    got = out.cpu().numpy()
    assert np.count_nonzero(got[0]) == 0
    from oracle.compose import kv_records
    ring = oracle_lib.pack_swa(wl.swa_rows(1, np.arange(cap)))
    win = ring[(5 + np.arange(64)) % cap]
    ref = oracle_lib.sparse_attn(wl.q(1), kv_records(wl, 1, sel[1][sel[1] >= 0]), win, int(wl.pos()[1]))
    assert row_norm_err(got[1], ref) <= ATTN_TOL_F32


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("pinned", [True, False])
def test_decode_host_equals_device_call(lib, out_f32, pinned):
    """csa2_decode_host (inputs and outputs in host memory: page-locked,
    read in place by the staging kernel, or pageable, copied) gives exactly
    csa2_decode's selection and output, on a garbage-filled workspace and on a
    second call with changed inputs."""
    import compressed_sparse_attention_index_gb300 as C
    from gen import inputs as G
    wl = small(n_seq=3, n_entries=65536, seed=252)
    dw = _dw(wl)
    n_q = dw.q.shape[0]
    dt = C.CSA2_OUT_F32 if out_f32 else C.CSA2_OUT_BF16
    ref = _bufs(dw, out_dtype=dt)
    from compressed_sparse_attention_index_gb300 import decode
    decode.fused_decode(dw, ref)
    qidx = np.concatenate([G.normal_block_bf16(wl.seed, G.S_QIDX, qi, 0, 32, 128) for qi in range(n_q)])
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    h_q = pin(dw.q.cpu())
    h_qidx = pin(torch.from_numpy(qidx.view(np.int16)))
    h_w = pin(dw.w.cpu())
    h_desc = pin(torch.stack([dw.q_seq, dw.n_vis, dw.pos, dw.swa_first, dw.swa_cnt]).cpu().contiguous())
    h_sel = pin(torch.full((n_q, 512), -7, dtype=torch.int32))
    h_out = pin(torch.full(tuple(ref.out.shape), 7, dtype=ref.out.dtype))
    wsb = C.csa2_workspace_size(C.CSA2_OP_DECODE_HOST, n_q, dw.n_max, 512)
    ws = torch.full((wsb,), 0xA5, dtype=torch.uint8, device="cuda")
    q_true = h_q.clone()
    for it in range(3):
        # the first call sees a zero attention query (its output is not
        # compared); the later ones the true one, so that a stale read of the
        # host buffer would show
        h_q.copy_(torch.zeros_like(q_true) if it == 0 else q_true)
        C.csa2_decode_host(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.kv, dw.swa, dw.swa.shape[1], h_q,
                           h_qidx, h_w, h_desc, n_q, h_sel, h_out, dt, None, ws, wsb)
        torch.cuda.synchronize()
        assert lib.csa2_get_device_status() == 0
        assert torch.equal(h_sel, ref.sel.cpu())
        if it > 0:
            assert torch.equal(h_out.view(torch.int16 if not out_f32 else torch.int32),
                               ref.out.cpu().view(torch.int16 if not out_f32 else torch.int32))
        h_out.fill_(7)


def test_bounded_wait_runs_out_cleanly(lib):
    """A wait that nothing completes ends after its limit with
    CSA2_ERR_TIMEOUT in the status word (no trap, no hang), and the context
    stays usable: a decode afterwards is exact."""
    import time
    t0 = time.time()
    lib.csa2_check_bounded_wait(2000)                    # 2 ms
    assert lib.csa2_get_device_status() == 5            # CSA2_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    assert lib.csa2_get_device_status() == 0            # read and cleared
    from compressed_sparse_attention_index_gb300 import decode
    wl = small(n_seq=2, n_entries=20_000, seed=253)
    dw = _dw(wl)
    chain, fused = _bufs(dw), _bufs(dw)
    decode.full_decode(dw, chain)
    decode.fused_decode(dw, fused)
    assert lib.csa2_get_device_status() == 0
    assert torch.equal(chain.sel, fused.sel)
    assert torch.equal(chain.out.view(torch.int32), fused.out.view(torch.int32))
