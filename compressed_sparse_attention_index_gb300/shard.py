"""Sequence sharding of one long cache over R ranks: the two merge steps.

A layout the decode path admits for caches too long for one GPU (every box
here has one GPU, so nothing runs it on GPUs; the tests run it on CPU ranks).
Rank r holds entries [lo_r, hi_r) of the cache (contiguous ranges), scores
them and keeps its local top-k of (score, index).  Every entry of the global
top-k is in the local top-k of the rank holding it, so one all-gather of the R
local lists and a top-k of their union give the global top-k.  Each rank then
attends over the selected entries it holds (the window on one rank only) and
returns its normalised output with the log-sum-exp of its logits per head;
the outputs combine as the softmax over all the entries would:
o = sum_r exp(lse_r - LSE) o_r with LSE = log sum_r exp(lse_r).  RoPE's
un-rotation is linear, so it commutes with that combination.
"""
import numpy as np


def shard_ranges(n: int, ranks: int):
    """Contiguous entry ranges [lo, hi) of `ranks` near-equal shards of n entries."""
    return [(r * n // ranks, (r + 1) * n // ranks) for r in range(ranks)]


def merge_topk(scores, indices, k: int) -> np.ndarray:
    """Top k of the union of the local lists by (score descending, index
    ascending), as ascending indices with -1 padding.  scores / indices: one
    array per rank (global indices; -1 marks an empty slot)."""
    s = np.concatenate([np.asarray(x, np.float64).ravel() for x in scores])
    i = np.concatenate([np.asarray(x, np.int64).ravel() for x in indices])
    keep = i >= 0
    s, i = s[keep], i[keep]
    order = np.lexsort((i, -s))                    # score descending, then index ascending
    top = np.sort(i[order[:k]])
    out = np.full(k, -1, np.int32)
    out[:top.size] = top
    return out


def lse_merge(outs, lses) -> np.ndarray:
    """Normalised partial outputs outs [R][H][D] with their per-head
    log-sum-exp lses [R][H] -> the output over all the entries [H][D] (zeros
    for a head no rank attended)."""
    outs = np.asarray(outs, np.float64)
    lses = np.asarray(lses, np.float64)
    m = lses.max(axis=0)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - m)                           # exp(-inf) = 0: a rank with no entries
    total = w.sum(axis=0)
    o = np.einsum("rh,rhd->hd", w, outs)
    return np.where((total > 0)[:, None], o / np.where(total > 0, total, 1.0)[:, None], 0.0)
