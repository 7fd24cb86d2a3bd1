"""The five synthetic workloads of the CSA2 decode path, as input recipes.

Only shapes, seeds and which generator stream feeds which tensor live here; no
packing, scoring or attention arithmetic.  Sizes follow the pages:

* 512-wide k=v latent per cache entry, 64 query heads (DeepSeek-V4.1-Flash
  study, reading notes on the attention enclosure);
* 32 indexer heads of 128 dims, top-512, candidate pool of 2,048 blocks of 8
  (same study, lightning-indexer note; perchy.ai "Full. Reindex. Reuse." card);
* 128-token sliding window (helix.ml, "CSA2 makes long context cheaper to retain");
* m=2 gated pooling for encoder caches (study, Full-layer global KV note).

Config index = seed.  Per-sequence tensors use the sequence index as sub-stream,
per-query tensors the query index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import inputs as G

H, D, HI, DI = 64, 512, 32, 128
TOPK, SWA, BLOCK, POOL_BLOCKS = 512, 128, 8, 2048


@dataclass
class Workload:
    name: str
    seed: int
    n_seq: int              # B: independent caches
    n_entries: int          # N: cache entries per sequence (after m-pooling)
    n_q: int                # queries in one step
    m: int = 1              # tokens pooled per entry
    zipf: bool = False      # Zipf-skewed indexer key norms
    pool: bool = False      # Reindex layer over a 16,384-position pool
    prefill: bool = False   # causal prefill: all queries on sequence 0
    swa_cap: int = SWA      # SWA ring capacity per sequence
    q_per_seq: int = 1      # draft positions decoded together: queries [b*G, b*G + G) of sequence b
    extra: dict = field(default_factory=dict)

    # ---- per-query descriptors (host int32 arrays) ----
    def q_seq(self) -> np.ndarray:
        if self.prefill:
            return np.zeros(self.n_q, np.int32)
        if self.q_per_seq > 1:
            return (np.arange(self.n_q) // self.q_per_seq % self.n_seq).astype(np.int32)
        return (np.arange(self.n_q) % self.n_seq).astype(np.int32)

    def pos(self) -> np.ndarray:
        if self.prefill:
            return np.arange(self.n_q, dtype=np.int32)
        if self.q_per_seq > 1:
            # draft position t of G sits at n_entries - G + t: the cache holds
            # the G drafted tokens' entries, each query sees up to its own
            t = np.arange(self.n_q) % self.q_per_seq
            return (self.n_entries - self.q_per_seq + t).astype(np.int32)
        return np.full(self.n_q, self.n_entries * self.m - 1, np.int32)

    def n_vis(self) -> np.ndarray:
        if self.prefill:   # entry j (tokens 2j, 2j+1) visible to query t iff 2j+1 <= t
            t = np.arange(self.n_q, dtype=np.int64)
            return ((t + 1) // self.m).astype(np.int32)
        if self.q_per_seq > 1:
            return (self.pos().astype(np.int64) + 1).astype(np.int32)
        return np.full(self.n_q, self.n_entries, np.int32)

    def swa_first(self) -> np.ndarray:
        p = self.pos().astype(np.int64)
        return (np.maximum(0, p - (SWA - 1)) % self.swa_cap).astype(np.int32)

    def swa_cnt(self) -> np.ndarray:
        return np.minimum(SWA, self.pos().astype(np.int64) + 1).astype(np.int32)

    # ---- tensors (bf16 as uint16 bit patterns, fp32 as float32) ----
    def latent_rows(self, seq: int, rows) -> np.ndarray:
        """[len(rows), 512] bf16: cache latents (m=1) or token latents (m=2)."""
        return G.normal_rows_bf16(self.seed, G.S_LATENT, seq, rows, D)

    def gate_rows(self, seq: int, rows) -> np.ndarray:
        return G.gate_logits_f32(self.seed, seq, rows, D)

    def key_rows(self, seq: int, rows) -> np.ndarray:
        """[len(rows), 128] bf16 indexer keys."""
        if self.zipf:
            return G.zipf_keys_bf16(self.seed, seq, self.n_entries, rows, DI)
        return G.normal_rows_bf16(self.seed, G.S_IDX_KEY, seq, rows, DI)

    def swa_rows(self, seq: int, slots) -> np.ndarray:
        return G.normal_rows_bf16(self.seed, G.S_SWA, seq, slots, D)

    def q(self, qi: int) -> np.ndarray:
        return G.normal_block_bf16(self.seed, G.S_Q, qi, 0, H, D)

    def qidx(self, qi: int, reindex: bool = False) -> np.ndarray:
        return G.normal_block_bf16(self.seed, G.S_QIDX_RE if reindex else G.S_QIDX, qi, 0, HI, DI)

    def w(self, qi: int, reindex: bool = False) -> np.ndarray:
        return G.weights_f32(self.seed, G.S_W_RE if reindex else G.S_W, qi, [0], HI)[0]

    # ---- the decoder step's layers (see DECODER_LAYERS): layer 0 is the Full
    # layer and uses the tensors above; layer l > 0 has its own attention query
    # and window, Reindex layer r its own indexer query and weights
    def q_layer(self, qi: int, layer: int) -> np.ndarray:
        if layer == 0:
            return self.q(qi)
        return G.normal_block_bf16(self.seed, G.S_LQ, layer * G.LAYER_SUB + qi, 0, H, D)

    def swa_rows_layer(self, seq: int, slots, layer: int) -> np.ndarray:
        if layer == 0:
            return self.swa_rows(seq, slots)
        return G.normal_rows_bf16(self.seed, G.S_LSWA, layer * G.LAYER_SUB + seq, slots, D)

    def qidx_reindex(self, qi: int, r: int) -> np.ndarray:
        return G.normal_block_bf16(self.seed, G.S_QIDX_RE, r * G.LAYER_SUB + qi, 0, HI, DI)

    def w_reindex(self, qi: int, r: int) -> np.ndarray:
        return G.weights_f32(self.seed, G.S_W_RE, r * G.LAYER_SUB + qi, [0], HI)[0]


CONFIGS = {
    0: Workload("tiny_full_decode_N4096_B1", 0, 1, 4096, 1),
    1: Workload("full_decode_N65536_B32", 1, 32, 65536, 32),
    2: Workload("m2_prefill_T8192", 2, 1, 4096, 8192, m=2, prefill=True, swa_cap=8192),
    3: Workload("reindex_decode_N1M_B64", 3, 64, 1 << 20, 64, pool=True),
    4: Workload("long_full_decode_N1M_B8_zipf", 4, 8, 1 << 20, 8, zipf=True),
}

# The decoder's twenty layers in one step (perchy.ai card "Full. Reindex.
# Reuse."; the study's reading notes): the Full layer (layer 0: it scores the
# whole cache, selects 512 entries and picks the 2,048-block pool), four
# Reindex layers (each scores the pool with its own indexer query and selects
# 512), and fifteen Reuse layers, each borrowing the selection of the nearest
# Full or Reindex layer before it (20 decoder layers = 1 + 4 + 15; the order
# within the decoder is not given on the pages: three Reuse layers follow each
# selecting layer).  Entries: (role, r) with r the selecting layer's number
# (0 = Full, 1..4 = Reindex r).
DECODER_LAYERS = [("full", 0)] + [("reuse", 0)] * 3
for _r in range(1, 5):
    DECODER_LAYERS += [("reindex", _r)] + [("reuse", _r)] * 3

# Multi-query decode (the next row after the five workloads above): the 8 x 1M
# Zipf caches with five draft positions per sequence decoded in one step.
MQ_DECODE = Workload("mq_decode_N1M_B8_G5_zipf", 4, 8, 1 << 20, 40, zipf=True, q_per_seq=5)


def small(n_seq=2, n_entries=1000, zipf=False, pool=False, seed=100, q_per_seq=1) -> Workload:
    """A small decode workload for tests (ragged N allowed)."""
    return Workload(f"small_N{n_entries}_B{n_seq}_G{q_per_seq}", seed, n_seq, n_entries, n_seq * q_per_seq,
                    zipf=zipf, pool=pool, q_per_seq=q_per_seq)
