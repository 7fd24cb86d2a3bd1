"""csa2_topk_noalloc: the top-k selection for callers that may not allocate
device memory (code that runs where cudaMalloc is unavailable or forbidden,
e.g. a plugin whose host application owns all device memory, or a serving
process that must keep a fixed footprint after start-up).  Its scratch is a
fixed array inside the library, so these checks compare it with csa2_topk,
which takes a caller-allocated workspace, on two different calls in a row
(the second call must not see anything left over from the first).

Kept in a file of its own that runs last, and written to pass both alone in a
fresh process and after the other tests."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gen import inputs as G  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def _both(lib, rows, n_valid, k, block=1):
    n_q, n = rows.shape
    scores = torch.from_numpy(np.ascontiguousarray(rows, np.float32)).cuda()
    nv = torch.tensor(n_valid, dtype=torch.int32, device="cuda")
    items = n if block == 1 else (n + 7) // 8
    wsb = lib.csa2_workspace_size(lib.CSA2_OP_TOPK, n_q, items, k)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    ref = torch.full((n_q, k), -7, dtype=torch.int32, device="cuda")
    got = torch.full((n_q, k), -7, dtype=torch.int32, device="cuda")
    lib.csa2_topk(scores, n, n_q, nv, n, k, block, None, ref, ws, wsb)
    lib.csa2_topk_noalloc(scores, n, n_q, nv, n, k, block, None, got)
    assert lib.csa2_get_device_status() == 0
    return got.cpu().numpy(), ref.cpu().numpy(), wsb


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    # call 1: eight 1,048,576-entry rows (1.6 MiB of scratch), Zipf-like skew and ties
    n = 1 << 20
    rows = np.stack([G.uniform_f32_scores(300 + i, i, n, 0 if i % 2 else 97) for i in range(8)])
    rows[1] = np.sign(rows[1]) * np.abs(rows[1]) ** 9
    got, ref, wsb = _both(lib, rows, [n, n - 5, n // 3, n, n, 17, n, n - 1000], 512)
    assert wsb > 0 and np.array_equal(got, ref)
    # call 2: a different shape and mode (262,144-entry rows, blocks of 8, k = 2048)
    n2 = 262_144
    rows2 = np.stack([G.uniform_f32_scores(310 + i, i, n2, 5) for i in range(3)])
    got2, ref2, wsb2 = _both(lib, rows2, [n2, n2 - 3, 140_000], 2048, block=8)
    assert wsb2 > 0 and np.array_equal(got2, ref2)
    # call 3 repeats call 1's inputs: same answer after another call used the scratch
    got3, _, _ = _both(lib, rows, [n, n - 5, n // 3, n, n, 17, n, n - 1000], 512)
    assert np.array_equal(got3, ref)


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    n = 1 << 20
    scratch = 4 << 20                        # CSA2_TOPK_NOALLOC_SCRATCH_BYTES
    per_query = lib.csa2_workspace_size(lib.CSA2_OP_TOPK, 1, n, 512)
    too_many = scratch // per_query + 1      # one query more than the array holds
    assert lib.csa2_workspace_size(lib.CSA2_OP_TOPK, too_many, n, 512) > scratch
    assert lib.csa2_workspace_size(lib.CSA2_OP_TOPK, too_many - 1, n, 512) <= scratch
    dummy = 1 << 20                          # never dereferenced: the call is rejected first
    with pytest.raises(lib.CSA2Error) as e:
        lib.csa2_topk_noalloc(dummy, n, too_many, dummy, n, 512, 1, None, dummy)
    assert e.value.code == 6                 # CSA2_ERR_WORKSPACE
