"""Decode-step compositions over the C ABI (one CUDA stream, no host sync).

* Full layer: csa2_index_score over every visible entry -> csa2_topk (k=512)
  -> csa2_sparse_attn over the selected entries + the SWA window.
* Reindex layer: Full-layer scores -> csa2_topk in block mode (2,048 blocks of
  8) -> csa2_index_score over the 16,384 pool slots with the Reindex layer's
  own indexer query -> csa2_topk over the pool -> csa2_sparse_attn.
  (An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture,
  lightning-indexer note: decoder Reindex layers score only a 16,384-position
  pool picked earlier as blocks of 8; perchy.ai/models/deepseek, card "Full.
  Reindex. Reuse.": the pool feeds the top-512 that attention reads.)
"""
from __future__ import annotations

import torch

from . import _lib as L

TOPK, POOL_BLOCKS, POOL_SLOTS, SWA = 512, 2048, 16384, 128


class DecodeBuffers:
    """Device buffers of one decode step for n_q queries over caches of n_max entries."""

    def __init__(self, n_q: int, n_max: int, pool: bool = False, out_dtype=L.CSA2_OUT_BF16, device="cuda",
                 q_group: int = 1):
        self.n_q, self.n_max, self.pool, self.out_dtype = n_q, n_max, pool, out_dtype
        self.scores = torch.empty((n_q, n_max), dtype=torch.float32, device=device)
        self.sel = torch.empty((n_q, TOPK), dtype=torch.int32, device=device)
        odt = torch.bfloat16 if out_dtype == L.CSA2_OUT_BF16 else torch.float32
        self.out = torch.empty((n_q, 64, 512), dtype=odt, device=device)
        ws_t = L.csa2_workspace_size(L.CSA2_OP_TOPK, n_q, n_max, TOPK)
        if pool:
            self.blocks = torch.empty((n_q, POOL_BLOCKS), dtype=torch.int32, device=device)
            self.pool_scores = torch.empty((n_q, POOL_SLOTS), dtype=torch.float32, device=device)
            ws_t = max(ws_t, L.csa2_workspace_size(L.CSA2_OP_TOPK, n_q, (n_max + 7) // 8, POOL_BLOCKS),
                       L.csa2_workspace_size(L.CSA2_OP_TOPK, n_q, POOL_SLOTS, TOPK))
        self.ws_topk_bytes = ws_t
        self.ws_attn_bytes = L.csa2_workspace_size(L.CSA2_OP_SPARSE_ATTN, n_q, TOPK + SWA)
        self.q_group = q_group
        self.ws_decode_bytes = L.csa2_workspace_size(L.CSA2_OP_DECODE_REINDEX, n_q, n_max, TOPK) if pool else \
            L.csa2_workspace_size(L.CSA2_OP_DECODE_MQ if q_group > 1 else L.CSA2_OP_DECODE, n_q, n_max, TOPK)
        self.ws = torch.empty(max(1, ws_t, self.ws_attn_bytes, self.ws_decode_bytes), dtype=torch.uint8,
                              device=device)


def full_decode(dw, buf: DecodeBuffers, params=None, stream=None):
    """Full-layer decode step of every query of a device workload (see gen.device)."""
    n_q = buf.n_q
    L.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w, dw.q_seq,
                       dw.n_vis, n_q, None, buf.scores, buf.n_max, params, stream)
    L.csa2_topk(buf.scores, buf.n_max, n_q, dw.n_vis, dw.n_max, TOPK, 1, None, buf.sel, buf.ws, buf.ws_topk_bytes,
                stream)
    attend(dw, buf, params, stream)
    return buf.out


def fused_decode(dw, buf: DecodeBuffers, params=None, stream=None):
    """The same Full-layer step as full_decode, as the single call csa2_decode
    (scores stay in the workspace; buf.sel and buf.out are written)."""
    L.csa2_decode(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w, dw.q_seq,
                  dw.n_vis, buf.n_q, dw.q, dw.kv, dw.swa, dw.swa.shape[1], dw.pos, dw.swa_first, dw.swa_cnt,
                  buf.sel, buf.out, buf.out_dtype, params, buf.ws, buf.ws_decode_bytes, stream)
    return buf.out


def mq_decode(dw, buf: DecodeBuffers, params=None, stream=None):
    """Full-layer decode of groups of buf.q_group queries per sequence (draft
    positions decoded together) as the single call csa2_decode_mq: each
    sequence's keys are scored once for its whole group."""
    L.csa2_decode_mq(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w, dw.q_seq,
                     dw.n_vis, buf.n_q, buf.q_group, dw.q, dw.kv, dw.swa, dw.swa.shape[1], dw.pos, dw.swa_first,
                     dw.swa_cnt, buf.sel, buf.out, buf.out_dtype, params, buf.ws, buf.ws_decode_bytes, stream)
    return buf.out


def reindex_decode(dw, buf: DecodeBuffers, params=None, stream=None, build_pool: bool = True):
    """Reindex-layer decode step.  With build_pool=False the candidate pool in
    buf.blocks (chosen earlier by the Full layer) is reused as it is."""
    n_q = buf.n_q
    if build_pool:
        L.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w,
                           dw.q_seq, dw.n_vis, n_q, None, buf.scores, buf.n_max, params, stream)
        L.csa2_topk(buf.scores, buf.n_max, n_q, dw.n_vis, dw.n_max, POOL_BLOCKS, 8, None, buf.blocks, buf.ws,
                    buf.ws_topk_bytes, stream)
    L.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib_re, dw.q_scale_re, dw.w_re,
                       dw.q_seq, dw.n_vis, n_q, buf.blocks, buf.pool_scores, POOL_SLOTS, params, stream)
    L.csa2_topk(buf.pool_scores, POOL_SLOTS, n_q, dw.n_vis, dw.n_max, TOPK, 1, buf.blocks, buf.sel, buf.ws,
                buf.ws_topk_bytes, stream)
    attend(dw, buf, params, stream)
    return buf.out


def fused_reindex_decode(dw, buf: DecodeBuffers, params=None, stream=None):
    """The Reindex-layer step over the pool in buf.blocks (chosen earlier by
    the Full layer) as the single call csa2_decode_reindex: the same selection
    and output as reindex_decode(build_pool=False); buf.sel and buf.out are
    written, the pool's scores stay in the workspace."""
    L.csa2_decode_reindex(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib_re, dw.q_scale_re, dw.w_re,
                          dw.q_seq, dw.n_vis, buf.n_q, buf.blocks, dw.q, dw.kv, dw.swa, dw.swa.shape[1], dw.pos,
                          dw.swa_first, dw.swa_cnt, buf.sel, buf.out, buf.out_dtype, params, buf.ws,
                          buf.ws_decode_bytes, stream)
    return buf.out


def attend(dw, buf: DecodeBuffers, params=None, stream=None):
    L.csa2_sparse_attn(dw.q, dw.kv, dw.n_max, dw.kv.shape[0], buf.sel, TOPK, dw.swa, dw.swa.shape[1], dw.q_seq,
                       dw.pos, dw.swa_first, dw.swa_cnt, buf.n_q, buf.out, buf.out_dtype, params, buf.ws,
                       buf.ws_attn_bytes, stream)
    return buf.out


class DecoderStep:
    """The decoder's layers in one step over the C ABI (layers as in
    gen.workloads.DECODER_LAYERS: (role, r) with role full / reindex / reuse):
    the Full layer scores every visible entry, keeps the top-512 and picks the
    pool of 2,048 blocks of 8 from the same scores; each Reindex layer r scores
    the pool with its own indexer query and keeps its top-512; every layer
    attends with its own query and window over the selection of the selecting
    layer it names (Reuse layers borrow it).  One stream, no host sync."""

    def __init__(self, n_q: int, n_max: int, layers, out_dtype=L.CSA2_OUT_F32, device="cuda"):
        self.layers, self.n_q, self.n_max = list(layers), n_q, n_max
        self.buf = DecodeBuffers(n_q, n_max, pool=True, out_dtype=out_dtype, device=device)
        n_sel = 1 + max(r for _, r in self.layers)
        self.sels = torch.empty((n_sel, n_q, TOPK), dtype=torch.int32, device=device)
        odt = torch.bfloat16 if out_dtype == L.CSA2_OUT_BF16 else torch.float32
        self.outs = torch.empty((len(self.layers), n_q, 64, 512), dtype=odt, device=device)
        self.out_dtype = out_dtype

    def run(self, dw, dl, params=None, stream=None):
        b, n_q = self.buf, self.n_q
        for l, (role, r) in enumerate(self.layers):
            if role == "full":
                L.csa2_index_score(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dw.q_nib, dw.q_scale, dw.w,
                                   dw.q_seq, dw.n_vis, n_q, None, b.scores, b.n_max, params, stream)
                L.csa2_topk(b.scores, b.n_max, n_q, dw.n_vis, dw.n_max, TOPK, 1, None, self.sels[r], b.ws,
                            b.ws_topk_bytes, stream)
                L.csa2_topk(b.scores, b.n_max, n_q, dw.n_vis, dw.n_max, POOL_BLOCKS, 8, None, b.blocks, b.ws,
                            b.ws_topk_bytes, stream)
            elif role == "reindex":
                # scoring the pool, its top-512 and the attention: one call
                L.csa2_decode_reindex(dw.key_nib, dw.key_scale, dw.n_max, dw.kv.shape[0], dl.q_nib_re[r],
                                      dl.q_scale_re[r], dl.w_re[r], dw.q_seq, dw.n_vis, n_q, b.blocks, dl.q[l], dw.kv,
                                      dl.swa[l], dl.swa.shape[2], dw.pos, dw.swa_first, dw.swa_cnt, self.sels[r],
                                      self.outs[l], self.out_dtype, params, b.ws, b.ws_decode_bytes, stream)
                continue
            L.csa2_sparse_attn(dl.q[l], dw.kv, dw.n_max, dw.kv.shape[0], self.sels[r], TOPK, dl.swa[l],
                               dl.swa.shape[2], dw.q_seq, dw.pos, dw.swa_first, dw.swa_cnt, n_q, self.outs[l],
                               self.out_dtype, params, b.ws, b.ws_attn_bytes, stream)
        return self.outs
