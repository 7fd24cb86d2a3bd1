"""GPU parity of the multi-query decode (several draft positions of one
sequence decoded together, their keys scored once per group) against the CPU
oracle, query by query, through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen.workloads import MQ_DECODE, small  # noqa: E402
from tests.parity import ATTN_TOL_F32, check_scores, check_selection, row_norm_err  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _dw(wl):
    from gen.device import build_device_workload
    return build_device_workload(wl)


@pytest.mark.parametrize("g,n_entries", [(1, 3000), (2, 3000), (5, 5003), (6, 20_000)])
def test_index_score_mq_matches_oracle_and_single_query(lib, oracle_lib, g, n_entries):
    """Every query of every group scores as the oracle does (and as the
    single-query kernel does); columns at or past a query's visible length
    are left untouched."""
    wl = small(n_seq=2, n_entries=n_entries, seed=280 + g, q_per_seq=g)
    dw = _dw(wl)
    n_q, n_max = dw.q.shape[0], dw.n_max
    mq = torch.full((n_q, n_max), 7.0, dtype=torch.float32, device="cuda")
    sq = torch.full((n_q, n_max), 7.0, dtype=torch.float32, device="cuda")
    lib.csa2_index_score_mq(dw.key_nib, dw.key_scale, n_max, 2, dw.q_nib, dw.q_scale, dw.w, dw.q_seq, dw.n_vis, n_q,
                            g, mq, n_max)
    lib.csa2_index_score(dw.key_nib, dw.key_scale, n_max, 2, dw.q_nib, dw.q_scale, dw.w, dw.q_seq, dw.n_vis, n_q,
                         None, sq, n_max)
    assert lib.csa2_get_device_status() == 0
    got, single = mq.cpu().numpy(), sq.cpu().numpy()
    n_vis = wl.n_vis()
    for qi in range(n_q):
        nv = int(n_vis[qi])
        check_scores(got[qi, :nv], oracle_lib.full_scores(wl, qi))
        m = np.abs(single[qi, :nv]).max()
        assert np.abs(got[qi, :nv] - single[qi, :nv]).max() <= 1e-6 * m
        assert np.all(got[qi, nv:] == 7.0)


def test_index_score_mq_group_across_sequences_is_skipped(lib):
    """A group whose queries name two sequences is skipped and reported."""
    wl = small(n_seq=2, n_entries=2000, seed=290, q_per_seq=2)
    dw = _dw(wl)
    q_seq = torch.tensor([0, 1, 1, 1], dtype=torch.int32, device="cuda")   # group 0 mixes sequences
    out = torch.full((4, dw.n_max), 7.0, dtype=torch.float32, device="cuda")
    lib.csa2_index_score_mq(dw.key_nib, dw.key_scale, dw.n_max, 2, dw.q_nib, dw.q_scale, dw.w, q_seq, dw.n_vis, 4, 2,
                            out, dw.n_max)
    assert lib.csa2_get_device_status() == 4                # CSA2_ERR_BOUNDS
    got = out.cpu().numpy()
    assert np.all(got[:2] == 7.0) and not np.any(got[2:, :1000] == 7.0)


def _check_mq_decode(lib, oracle_lib, wl, dw, queries):
    from compressed_sparse_attention_index_gb300 import decode, CSA2_OUT_F32
    from oracle.compose import kv_records, swa_records
    buf = decode.DecodeBuffers(dw.q.shape[0], dw.n_max, out_dtype=CSA2_OUT_F32, q_group=wl.q_per_seq)
    decode.mq_decode(dw, buf)
    sel, out = buf.sel.cpu().numpy(), buf.out.cpu().numpy()
    assert lib.csa2_get_device_status() == 0
    for qi in queries:
        r = oracle_lib.decode_query(wl, qi)
        check_selection(sel[qi], r["sel"], r["scores"])
        seq = int(wl.q_seq()[qi])
        s = sel[qi][sel[qi] >= 0]
        ref = oracle_lib.sparse_attn(wl.q(qi), kv_records(wl, seq, s),
                                     swa_records(wl, seq, int(wl.swa_first()[qi]), int(wl.swa_cnt()[qi])),
                                     int(wl.pos()[qi]))
        assert row_norm_err(out[qi], ref) <= ATTN_TOL_F32


def test_decode_mq_five_drafts(lib, oracle_lib):
    """Five draft positions per sequence (each sees the cache up to itself):
    selection and attention of every query match the oracle."""
    wl = small(n_seq=2, n_entries=30_011, seed=291, q_per_seq=5)
    _check_mq_decode(lib, oracle_lib, wl, _dw(wl), range(10))


def test_decode_mq_full_size_sampled(lib, oracle_lib):
    """8 sequences x 1,048,576 Zipf entries, five drafts each (40 queries)."""
    wl = MQ_DECODE
    _check_mq_decode(lib, oracle_lib, wl, _dw(wl), [0, 4, 37])
