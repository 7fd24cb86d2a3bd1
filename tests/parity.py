"""Comparison rules shared by the GPU parity tests.

* Packing, indices, pool blocks: bit-exact.
* Selected sets: equal, except at entries whose oracle score is within 1e-5
  (relative) of the oracle's k-th score (the near-tie rule).
* Attention output: row-normalised max error  max_c|o - r| / max_c|r|  per
  (query, head) <= 2e-3 on the fp32 output; bf16 output <= 2e-3 + 2^-8.
* Indexer scores (diagnostic): |s - r| <= 1e-5 * max|r| per query.
"""
import numpy as np

ATTN_TOL_F32 = 2e-3
ATTN_TOL_BF16 = 2e-3 + 2.0**-8
SCORE_TOL = 1e-5
NEAR_TIE = 1e-5


def row_norm_err(out, ref) -> float:
    out = np.asarray(out, np.float64).reshape(-1, 512)
    ref = np.asarray(ref, np.float64).reshape(-1, 512)
    den = np.abs(ref).max(axis=1)
    num = np.abs(out - ref).max(axis=1)
    zero = den == 0
    assert np.all(num[zero] == 0), "nonzero output where the reference row is all zero"
    return float((num[~zero] / den[~zero]).max()) if np.any(~zero) else 0.0


def check_selection(sel_gpu, sel_orc, scores_orc, tol=NEAR_TIE, pos_to_score=None):
    """Near-tie rule.  scores_orc[i] is the oracle score of entry i (or use
    pos_to_score to map a selected index to its score)."""
    g = set(int(x) for x in np.asarray(sel_gpu) if x >= 0)
    o = set(int(x) for x in np.asarray(sel_orc) if x >= 0)
    assert len(g) == len(o), (len(g), len(o))
    sc = (lambda i: scores_orc[i]) if pos_to_score is None else pos_to_score
    if not o:
        return 0
    s_k = min(sc(i) for i in o)
    diff = g ^ o
    for i in diff:
        assert abs(sc(i) - s_k) <= tol * abs(s_k), (i, sc(i), s_k)
    g_sorted = np.asarray(sel_gpu)
    valid = g_sorted[g_sorted >= 0]
    assert np.all(np.diff(valid) > 0), "selection not ascending"
    assert np.all(g_sorted[len(valid):] == -1)
    return len(diff)


def check_scores(s_gpu, s_orc, tol=SCORE_TOL):
    s_gpu = np.asarray(s_gpu, np.float64)
    s_orc = np.asarray(s_orc, np.float64)
    m = np.abs(s_orc).max() if s_orc.size else 0.0
    err = np.abs(s_gpu - s_orc).max() if s_orc.size else 0.0
    assert err <= tol * m + 1e-30, (err, m)
    return err / m if m else 0.0


def unswizzle_idx_nibbles(nib):
    """Logical order of IDX nibble rows stored 64B-swizzled (include/csa2.h):
    16-B chunk c of row r (row 0 at a 512-B aligned address) sits at chunk
    c ^ ((r >> 1) & 3).  The permutation is its own inverse."""
    nib = np.asarray(nib, np.uint8).reshape(-1, 4, 16)
    r = np.arange(nib.shape[0])
    out = np.empty_like(nib)
    for c in range(4):
        out[:, c] = nib[r, c ^ ((r >> 1) & 3)]
    return out.reshape(-1, 64)
