"""GPU parity of the decoder's twenty layers in one step (one Full layer,
four Reindex layers, fifteen Reuse layers borrowing the selections) against
the CPU oracle's composition of the same roles, through the C ABI."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen.workloads import CONFIGS, DECODER_LAYERS, small  # noqa: E402
from tests.parity import ATTN_TOL_F32, check_selection, row_norm_err  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _run(wl):
    from compressed_sparse_attention_index_gb300 import decode, CSA2_OUT_F32
    from gen.device import build_device_workload, build_decoder_layers
    dw = build_device_workload(wl)
    dl = build_decoder_layers(wl, dw, DECODER_LAYERS)
    step = decode.DecoderStep(dw.q.shape[0], dw.n_max, DECODER_LAYERS, out_dtype=CSA2_OUT_F32)
    step.run(dw, dl)
    return step


def _check(lib, oracle_lib, wl, step, qi):
    blocks = step.buf.blocks.cpu().numpy()[qi]
    sels = {r: step.sels[r].cpu().numpy()[qi] for r in range(step.sels.shape[0])}
    outs = step.outs.cpu().numpy()[:, qi]
    ref = oracle_lib.decoder_step_query(wl, qi, DECODER_LAYERS)
    n = int(wl.n_vis()[qi])
    s_full = ref["scores"][0][1]
    check_selection(sels[0], ref["sel"][0], s_full)
    bscore = lambda b: max(s_full[8 * b:min(n, 8 * b + 8)])
    check_selection(blocks, ref["pool"], None, pos_to_score=bscore)
    # each Reindex layer on the GPU's own pool
    for r in range(1, 5):
        rp = oracle_lib.reindex_on_pool(wl, qi, blocks, layer=r)
        ps = dict(zip(rp["pool_pos"].tolist(), rp["scores_pool"].tolist()))
        check_selection(sels[r], rp["sel"], None, pos_to_score=lambda p: ps[p])
    # every layer's attention on the GPU's selections
    for l, (role, r) in enumerate(DECODER_LAYERS):
        att = oracle_lib.layer_attention(wl, qi, l, sels[r])
        assert row_norm_err(outs[l], att) <= ATTN_TOL_F32, (l, role, r)


def test_decoder_step_small(lib, oracle_lib):
    wl = small(n_seq=2, n_entries=40_000, seed=300)
    step = _run(wl)
    assert lib.csa2_get_device_status() == 0
    for qi in range(2):
        _check(lib, oracle_lib, wl, step, qi)


def test_decoder_step_full_size_sampled(lib, oracle_lib):
    """The 8 x 1,048,576 Zipf caches, every layer of one sampled query."""
    wl = CONFIGS[4]
    step = _run(wl)
    assert lib.csa2_get_device_status() == 0
    _check(lib, oracle_lib, wl, step, 3)
