"""Block-map prediction in fp64 (test infrastructure; see the package header).

Follows the block-map pipeline of the "Sparge Attention (Composable Kernel)"
README (intro: "mean-pool -> cosine sim -> pooled QK -> top-k LUT"; 'Status vs
Upstream': per-block mean-pool, cosine similarity, pooled QK, top-k /
cdfthreshd block selection, per-head topk / simthreshd1 / cdfthreshd; 'Not yet
ported': the causal mask in the pooled score and the attention sink that forces
kv-block column 0 on).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

from synth import bits_to_f64


def pool_blocks(x: np.ndarray, blk: int) -> np.ndarray:
    """Mean of the rows of every ``blk``-row block of ``x`` [s, d] -> [nb, d].

    A partial last block averages the rows it holds.  (README intro:
    per-block mean-pool.)"""
    s, d = x.shape
    nb = (s + blk - 1) // blk
    out = np.empty((nb, d), dtype=np.float64)
    for j in range(nb):
        rows = x[j * blk:min((j + 1) * blk, s)]
        out[j] = rows.sum(axis=0) / rows.shape[0]
    return out


def self_similarity(block: np.ndarray) -> float:
    """Mean cosine similarity over all ordered row pairs (self-pairs included).

    With unit rows u_t = x_t / ||x_t|| (a zero row gives u_t = 0) the mean of
    u_a . u_b over the n^2 ordered pairs is ||sum_t u_t||^2 / n^2.  (README
    intro: cosine similarity of a block, compared with simthreshd1.)"""
    n = block.shape[0]
    norms = np.sqrt((block * block).sum(axis=1))
    unit = np.zeros_like(block)
    nz = norms > 0.0
    unit[nz] = block[nz] / norms[nz, None]
    tot = unit.sum(axis=0)
    return float(tot @ tot) / float(n * n)


def eligible_mask(nq: int, nk: int, blkq: int, blkk: int, causal: bool) -> np.ndarray:
    """Block pairs that hold at least one visible (query, key) pair.

    Causal: kv block j is eligible for q block i when its first key position
    j*blkk is at or before the last query position (i+1)*blkq - 1 ('Not yet
    ported': the causal mask applied to the pooled score)."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return j * blkk <= (i + 1) * blkq - 1


def topk_count(topk: float, n_elig: int) -> int:
    """K_i = ceil(topk * n_elig), the product taken in float32 (the precision
    in which topk is passed), so that CPU and GPU take the same decision."""
    prod = np.float32(topk) * np.float32(n_elig)
    return int(math.ceil(float(prod)))


def select_row(score: np.ndarray, topk: Optional[float], cdf: Optional[float],
               n_elig: int) -> np.ndarray:
    """Selected kv blocks of one q block from its pooled scores.

    ``score`` [nk] holds scale * qbar . kbar, or -inf where the block may not
    be chosen (masked).  The finite entries are ordered by pooled softmax
    probability, descending, with the lower block index first on ties; the
    softmax is monotone, so this is the order of the scores.  topk mode keeps
    the first min(K_i, #finite) of them; cdf mode keeps the shortest prefix
    whose probability mass reaches ``cdf`` (the crossing entry included), or
    every finite entry when the total stays below it.  ('Status vs Upstream':
    top-k / cdfthreshd block selection; 'Not yet ported': sort-based top-k.)"""
    nk = score.shape[0]
    sel = np.zeros(nk, dtype=bool)
    finite = np.isfinite(score)
    nf = int(finite.sum())
    if nf == 0:
        return sel
    idx = np.nonzero(finite)[0]
    sc = score[idx]
    # pooled softmax over the finite entries
    m = sc.max()
    e = np.exp(sc - m)
    p = e / e.sum()
    order = np.lexsort((idx, -p))  # primary: p descending; ties: index ascending
    if topk is not None:
        kcount = min(topk_count(topk, n_elig), nf)
        sel[idx[order[:kcount]]] = True
        return sel
    cum = np.cumsum(p[order])
    hit = np.nonzero(cum >= cdf)[0]
    take = int(hit[0]) + 1 if hit.size else nf
    sel[idx[order[:take]]] = True
    return sel


def smooth_keys(kg: np.ndarray) -> np.ndarray:
    """K smoothing: every key row minus the mean key row of the sequence,
    k - km with km = mean over the s_k rows ("Sparge Attention (Composable
    Kernel)" README, 'Not yet ported': pre-pool k -= km)."""
    return kg - kg.mean(axis=0, keepdims=True)


def block_map_head(qh: np.ndarray, kg: np.ndarray, theta: float, topk: Optional[float],
                   cdf: Optional[float], scale: float, causal: bool, sink: bool,
                   blkq: int = 64, blkk: int = 64, smooth_k: bool = False) -> dict:
    """Block map of one query head ``qh`` [s_q, d] against its KV head ``kg``
    [s_k, d] (steps 1-7 of the package header).  With ``smooth_k`` every step
    runs on the smoothed keys (``smooth_keys``); the queries are unchanged."""
    if smooth_k:
        kg = smooth_keys(kg)
    qbar = pool_blocks(qh, blkq)
    kbar = pool_blocks(kg, blkk)
    nq, nk = qbar.shape[0], kbar.shape[0]
    simq_val = np.array([self_similarity(qh[i * blkq:(i + 1) * blkq]) for i in range(nq)])
    simk_val = np.array([self_similarity(kg[j * blkk:(j + 1) * blkk]) for j in range(nk)])
    simq = simq_val > theta
    simk = simk_val > theta
    elig = eligible_mask(nq, nk, blkq, blkk, causal)
    raw = scale * (qbar @ kbar.T)
    score = np.where(elig & simk[None, :], raw, -np.inf)
    selected = np.zeros((nq, nk), dtype=bool)
    for i in range(nq):
        selected[i] = select_row(score[i], topk, cdf, int(elig[i].sum()))
    forced = np.zeros((nq, nk), dtype=bool)
    forced[:, ~simk] = True
    forced[~simq, :] = True
    if sink:
        forced[:, 0] = True
    bmap = (selected | forced) & elig
    lut = np.full((nq, nk), -1, dtype=np.int32)
    count = np.zeros(nq, dtype=np.int32)
    for i in range(nq):
        cols = np.nonzero(bmap[i])[0]
        lut[i, :cols.size] = cols
        count[i] = cols.size
    return {"block_map": bmap, "lut": lut, "count": count, "score": score, "raw": raw,
            "simq": simq_val, "simk": simk_val, "elig": elig, "selected": selected,
            "qbar": qbar, "kbar": kbar}


def _head(x: np.ndarray, bi: int, h: int, dtype: Optional[str]) -> np.ndarray:
    if dtype is None:
        return np.asarray(x[bi, h], dtype=np.float64)
    return bits_to_f64(x[bi, h], dtype)


def sparge_block_map(q: np.ndarray, k: np.ndarray, topk: Optional[np.ndarray],
                     cdfthreshd: Optional[np.ndarray], simthreshd1: np.ndarray,
                     scale: float, causal: bool, attention_sink: bool,
                     blkq: int = 64, blkk: int = 64, keep_aux: bool = False,
                     dtype: Optional[str] = None, heads: Optional[list] = None,
                     smooth_k: bool = False) -> dict:
    """Block map of every (batch, query head): q [b, hq, s, d], k [b, hk, s, d],
    float64 values or, with ``dtype`` = "f16" / "bf16", their bit patterns
    (widened exactly one head at a time).  ``heads`` restricts the work to a
    list of (batch, head) pairs; the other rows stay empty.
    Query head h reads KV head h // (hq // hk) (the GQA mapping of ROCm/aiter
    pull 6841: query head j reads KV head j // (hq / hk)).  Per-head
    hyperparameters are arrays of length hq; exactly one of topk / cdfthreshd
    is given.  ``smooth_k`` applies K smoothing per KV head before pooling.
    Returns the LUT [b, hq, nq, nk] (ascending, -1 padded), the count
    [b, hq, nq] and the boolean block map."""
    b, hq, s_q, d = q.shape
    hk = k.shape[1]
    if (topk is None) == (cdfthreshd is None):
        raise ValueError("exactly one of topk / cdfthreshd")
    ratio = hq // hk
    nq = (s_q + blkq - 1) // blkq
    nk = (k.shape[2] + blkk - 1) // blkk
    lut = np.full((b, hq, nq, nk), -1, dtype=np.int32)
    count = np.zeros((b, hq, nq), dtype=np.int32)
    bmap = np.zeros((b, hq, nq, nk), dtype=bool)
    aux = {}
    todo = heads if heads is not None else [(bi, h) for bi in range(b) for h in range(hq)]
    for bi, h in todo:
        r = block_map_head(_head(q, bi, h, dtype), _head(k, bi, h // ratio, dtype),
                           float(simthreshd1[h]),
                           None if topk is None else float(topk[h]),
                           None if cdfthreshd is None else float(cdfthreshd[h]),
                           scale, causal, attention_sink, blkq, blkk, smooth_k)
        lut[bi, h] = r["lut"]
        count[bi, h] = r["count"]
        bmap[bi, h] = r["block_map"]
        if keep_aux:
            aux[(bi, h)] = r
    out = {"lut": lut, "count": count, "block_map": bmap}
    if keep_aux:
        out["aux"] = aux
    return out
