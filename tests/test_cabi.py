"""The C-ABI library loads, exports every symbol include/csa2.h declares, and
rejects bad arguments on the host before touching a GPU (no compute here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "csa2.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    import compressed_sparse_attention_index_gb300 as c
    return c


def test_exports_match_header(lib):
    L = lib.load()
    decl = _declared()
    assert "csa2_index_score" in decl and "csa2_topk" in decl and "csa2_sparse_attn" in decl
    assert "csa2_fp4_pack" in decl
    for name in decl:
        assert hasattr(L, name), name
    assert sorted(lib.EXPORTS) == decl


def test_entry_bytes_and_params(lib):
    assert [lib.csa2_entry_bytes(k) for k in (0, 1, 2)] == [288, 68, 528]
    assert lib.csa2_entry_bytes(7) == 0
    p = lib.default_params()
    assert (p.heads, p.dim, p.rope_dim, p.rope_off, p.idx_heads, p.idx_dim, p.topk, p.swa, p.block,
            p.pool_blocks) == (64, 512, 64, 448, 32, 128, 512, 128, 8, 2048)
    assert abs(p.sm_scale - 512 ** -0.5) < 1e-8 and p.rope_base == 10000.0


def _code(fn, *args):
    return fn(*args)


def test_host_validation_rejects_before_launch(lib):
    L = lib.load()
    INVALID, UNSUP, WS = 1, 2, 6
    fake = 1 << 20                                   # never dereferenced: rejected first
    assert L.csa2_fp4_pack(9, fake, 4, 1, None, fake, None, None) == INVALID
    assert L.csa2_fp4_pack(0, fake, 3, 2, fake, fake, None, None) == INVALID           # odd rows with m=2
    assert L.csa2_fp4_pack(1, fake, 4, 1, None, fake, None, None) == INVALID           # IDX needs scales
    assert L.csa2_fp4_pack(0, fake + 8, 4, 1, None, fake, None, None) == INVALID       # misaligned src
    assert L.csa2_fp4_pack(0, None, 0, 1, None, None, None, None) == 0                 # empty: nothing to do
    p = lib.default_params()
    p.heads = 32
    assert L.csa2_index_score(fake, fake, 1024, 1, fake, fake, fake, fake, fake, 1, None, fake, 1024,
                              ctypes.byref(p), None) == UNSUP
    assert L.csa2_index_score(fake, fake, 1000, 1, fake, fake, fake, fake, fake, 1, None, fake, 1000,
                              None, None) == INVALID                                    # n_max % 128
    assert L.csa2_index_score(fake, fake, 1024, 1, fake, fake, fake, fake, fake, 1, fake, fake, 1024,
                              None, None) == INVALID                                    # pool stride < 16384
    assert L.csa2_topk(fake, 1024, 1, fake, 1024, 0, 1, None, fake, None, 0, None) == UNSUP
    assert L.csa2_topk(fake, 1024, 1, fake, 1024, 4096, 1, None, fake, None, 0, None) == UNSUP
    assert L.csa2_topk(fake, 1024, 1, fake, 1024, 512, 3, None, fake, None, 0, None) == INVALID
    assert L.csa2_topk(fake, 1 << 20, 1, fake, 1 << 20, 512, 1, None, fake, None, 0, None) == WS
    assert L.csa2_sparse_attn(fake, fake, 1024, 1, fake, 513, fake, 128, fake, fake, fake, fake, 1, fake, 0,
                              None, None, 0, None) == INVALID
    assert L.csa2_sparse_attn(fake, fake, 1024, 1, fake, 512, fake, 128, fake, fake, fake, fake, 1, fake, 5,
                              None, None, 0, None) == INVALID
    assert L.csa2_sparse_attn(fake, fake, 1024, 1, fake, 512, fake, 128, fake, fake, fake, fake, 8, fake, 0,
                              None, None, 0, None) == WS
    # csa2_decode_host: a missing host buffer, a workspace without room for the staging
    args = (fake, fake, 1024, 1, fake, fake, 128)
    assert L.csa2_decode_host(*args, fake, fake, fake, None, 1, None, fake, 0, None, fake, 1 << 30, None) == INVALID
    assert L.csa2_decode_host(*args, fake, fake, fake, fake, 1, None, fake, 0, None, fake, 1024, None) == WS
    assert L.csa2_decode_host(*args, fake, fake, fake, fake, 1, None, fake, 7, None, fake, 1 << 30, None) == INVALID
    # csa2_index_key_proj / csa2_build_cache: negative or ragged sizes, a gate
    # that does not match m, an unaligned key plane, a short workspace
    assert L.csa2_index_key_proj(fake, -1, fake, fake, None) == INVALID
    assert L.csa2_index_key_proj(fake, 0, None, None, None) == 0                         # nothing to do
    assert L.csa2_index_key_proj(fake + 8, 4, fake, fake, None) == INVALID
    assert L.csa2_build_cache(fake, 24, 2, fake, fake, fake, fake, fake, fake, 1 << 30, None) == INVALID
    assert L.csa2_build_cache(fake, 32, 2, None, fake, fake, fake, fake, fake, 1 << 30, None) == INVALID
    assert L.csa2_build_cache(fake, 32, 1, fake, fake, fake, fake, fake, fake, 1 << 30, None) == INVALID
    assert L.csa2_build_cache(fake, 32, 1, None, fake, fake, fake + 256, fake, fake,
                              1 << 30, None) == INVALID
    assert L.csa2_build_cache(fake, 32, 2, fake, fake, fake, fake, fake, fake, 1024, None) == WS
    # csa2_decode_reindex: no pool, a misaligned pool, n_max not a multiple of 128, a short workspace
    def reindex(n_max, pool, ws_bytes):
        return L.csa2_decode_reindex(fake, fake, n_max, 1, fake, fake, fake, fake, fake, 8, pool, fake, fake, fake,
                                     128, fake, fake, fake, fake, fake, 0, None, fake, ws_bytes, None)
    assert reindex(1024, None, 1 << 30) == INVALID
    assert reindex(1024, fake + 2, 1 << 30) == INVALID
    assert reindex(1000, fake, 1 << 30) == INVALID
    assert reindex(1024, fake, 1024) == WS
    assert L.csa2_profile_events(fake, None) == INVALID                                  # both or neither
    assert L.csa2_profile_events(None, None) == 0
    assert L.csa2_check_bounded_wait(0, None) == INVALID                                 # limit out of range
    assert L.csa2_check_bounded_wait(2_000_001, None) == INVALID
    assert L.csa2_get_device_status(None, None) == INVALID


def test_workspace_sizes(lib):
    # the host-buffer decode stages the step's inputs and outputs after the decode workspace
    dec = lib.csa2_workspace_size(lib.CSA2_OP_DECODE, 8, 1 << 20, 512)
    host = lib.csa2_workspace_size(lib.CSA2_OP_DECODE_HOST, 8, 1 << 20, 512)
    staged = 8 * (65536 + 8192 + 2048 + 128 + 128 + 20 + 2048 + 131072)
    assert staged <= host - dec <= staged + 8 * 256
    assert lib.csa2_workspace_size(lib.CSA2_OP_TOPK, 8, 4096, 512) == 0          # one CTA per row
    # per row: the 2,048 maxima of 512-item supergroups (candidates stay on chip)
    assert lib.csa2_workspace_size(lib.CSA2_OP_TOPK, 8, 1 << 20, 512) == 8 * 2048 * 4
    assert lib.csa2_workspace_size(lib.CSA2_OP_SPARSE_ATTN, 8192, 640) == 0      # no split for big batches
    # the Reindex step: the pool's scores and block maxima come first
    assert lib.csa2_workspace_size(lib.CSA2_OP_DECODE_REINDEX, 8, 1 << 20, 512) >= 8 * (16384 + 2048) * 4
    # the cache build's scratch: one chunk of at most 131,072 entries (keys; for m = 2 the pooled
    # latents, two counts and the pooling's fix-up list of four words per entry)
    assert lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, 1 << 20, 2) == \
        131072 * (128 + 512) * 2 + 256 + 131072 * 4 * 4
    assert lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, 1 << 20, 1) == 131072 * 128 * 2
    assert lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, 64, 2) == 32 * (128 + 512) * 2 + 256 + 512
    with pytest.raises(lib.CSA2Error):
        lib.csa2_workspace_size(lib.CSA2_OP_BUILD_CACHE, 0, 64, 3)
    with pytest.raises(lib.CSA2Error):
        lib.csa2_workspace_size(lib.CSA2_OP_SPARSE_ATTN, 8, 100)
