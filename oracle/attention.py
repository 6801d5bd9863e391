"""Sparse attention, split-KV partials, the LSE combine and sparse decode in
fp64 (test infrastructure; see the package header).

Sources:
* "Sparge Attention (Composable Kernel)" README, intro: the sparse FMHA stage
  visits only the kv blocks listed in each q block's LUT row.
* "Incremental_FlashAttention updating_log.md", Stage 1: reference attention
  returns (O, LSE) with a natural-log LSE; partials over disjoint key sets are
  merged with the lse_max trick, in any order, and an empty partial
  (LSE = -inf) is the identity.  Stage 3: an empty block list writes O = 0 and
  LSE = -inf.
* ROCm/aiter pull 6841: the exported LSE is the logsumexp of the scores that
  were actually computed (the selected blocks), -inf for an empty LUT row.
* ROCm/aiter pull 6841: the LSE is exported so that partial attentions over
  disjoint key sets can be merged across ranks (ring / context parallelism);
  here the kv blocks are cut into contiguous per-rank ranges.
* ROCm/aiter pull 4919: sparse MLA decode - each query lists top-k token
  positions, resolved through a page table into rows of a paged cache; a K row
  is 512 latent + 64 rotary values and V is its latent plane; the key list is
  split into chunks whose partials (O_s, LSE_s) an LSE reduce merges.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from synth import bits_to_f64


def row_keys(lut_row: Iterable[int], blkk: int, s_k: int) -> np.ndarray:
    """Key positions covered by a list of kv blocks, in list order."""
    parts = [np.arange(j * blkk, min((j + 1) * blkk, s_k)) for j in lut_row]
    if not parts:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(parts)


def _softmax_attend(scores: np.ndarray, vals: np.ndarray):
    """O = softmax(scores) @ vals and LSE = logsumexp(scores) per row, with
    rows whose scores are all -inf giving O = 0, LSE = -inf."""
    rows, dv = scores.shape[0], vals.shape[1]
    out = np.zeros((rows, dv), dtype=np.float64)
    lse = np.full(rows, -np.inf, dtype=np.float64)
    if scores.shape[1] == 0:
        return out, lse
    m = scores.max(axis=1)
    live = np.isfinite(m)
    if not live.any():
        return out, lse
    p = np.exp(scores[live] - m[live, None])
    l = p.sum(axis=1)
    out[live] = (p @ vals) / l[:, None]
    lse[live] = m[live] + np.log(l)
    return out, lse


def attention_unit(q: np.ndarray, k: np.ndarray, v: np.ndarray, lut_row: Iterable[int],
                   i: int, blkq: int, blkk: int, scale: float, causal: bool,
                   key_offset: int = 0):
    """Attention of the rows of q block ``i`` over the keys of the listed kv
    blocks.  q [s_q, d], k [s_k, d], v [s_k, dv] are one head's float64
    values.  Under ``causal`` the key at index u is visible to the query at
    index t only when u <= t + key_offset: key_offset = 0 when queries and keys
    start at the same position, s_k - s_q when the queries are the last s_q
    positions of the keys' sequence (the causal alignment of a speculative
    dense pass over caller-gathered keys, "Incremental_FlashAttention
    updating_log.md" Stage 5), -lo when a rank's keys start at position lo
    (causal context parallelism).  Returns (O [rows, dv], LSE [rows])."""
    s_q, s_k = q.shape[0], k.shape[0]
    t = np.arange(i * blkq, min((i + 1) * blkq, s_q))
    keys = row_keys(lut_row, blkk, s_k)
    scores = scale * (q[t] @ k[keys].T)
    if causal:
        scores = np.where(keys[None, :] <= t[:, None] + key_offset, scores, -np.inf)
    return _softmax_attend(scores, v[keys])


def _head(x: np.ndarray, bi: int, h: int, dtype: Optional[str]) -> np.ndarray:
    if dtype is None:
        return np.asarray(x[bi, h], dtype=np.float64)
    return bits_to_f64(x[bi, h], dtype)


def sparse_fmha(q: np.ndarray, k: np.ndarray, v: np.ndarray, lut: np.ndarray,
                count: np.ndarray, scale: float, causal: bool, units: Optional[list] = None,
                blkq: int = 64, blkk: int = 64, dtype: Optional[str] = None,
                key_offset: int = 0) -> dict:
    """Block-sparse attention of q [b, hq, s_q, d] over k, v [b, hk, s_k, *]
    with LUT [b, hq, nq, nk] / count [b, hq, nq] (values, or bit patterns when
    ``dtype`` is given).  Query head h reads KV head h // (hq // hk).  The
    causal mask takes ``key_offset`` as attention_unit does.  ``units`` lists
    (b, h, i) q blocks to compute (default: all).  Returns
    {(b, h, i): (O, LSE)}."""
    b, hq, s_q, _ = q.shape
    hk = k.shape[1]
    ratio = hq // hk
    nq = (s_q + blkq - 1) // blkq
    if units is None:
        units = [(bi, h, i) for bi in range(b) for h in range(hq) for i in range(nq)]
    res = {}
    cache = {}
    for bi, h, i in units:
        key = (bi, h)
        if key not in cache:
            cache.clear()
            cache[key] = (_head(q, bi, h, dtype), _head(k, bi, h // ratio, dtype),
                          _head(v, bi, h // ratio, dtype))
        qh, kg, vg = cache[key]
        row = lut[bi, h, i, :count[bi, h, i]]
        res[(bi, h, i)] = attention_unit(qh, kg, vg, row, i, blkq, blkk, scale, causal,
                                         key_offset)
    return res


def split_bounds(n: int, num_splits: int) -> list:
    """Contiguous chunks of an n-entry list: the first n mod S chunks hold
    ceil(n/S) entries, the others floor(n/S) (some may be empty)."""
    base, extra = divmod(n, num_splits)
    out, start = [], 0
    for s in range(num_splits):
        size = base + (1 if s < extra else 0)
        out.append((start, start + size))
        start += size
    return out


def split_partials_unit(qh: np.ndarray, kg: np.ndarray, vg: np.ndarray, lut_row,
                        i: int, num_splits: int, blkq: int, blkk: int, scale: float,
                        causal: bool):
    """Split-KV partials of one q block: attention over each contiguous chunk
    of its LUT row.  Returns (O_parts [S, rows, dv], LSE_parts [S, rows])."""
    lut_row = list(lut_row)
    outs, lses = [], []
    for lo, hi in split_bounds(len(lut_row), num_splits):
        o, l = attention_unit(qh, kg, vg, lut_row[lo:hi], i, blkq, blkk, scale, causal)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def combine(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge partials over disjoint key sets (the lse_max trick of the
    updating_log's Stage 1): m = max_s LSE_s, w_s = exp(LSE_s - m),
    O = sum_s w_s O_s / sum_s w_s, LSE = m + ln(sum_s w_s).  Rows whose
    partials are all empty (LSE = -inf) give O = 0, LSE = -inf.
    o_parts [S, rows, dv], lse_parts [S, rows]."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    rows, dv = o_parts.shape[1], o_parts.shape[2]
    out = np.zeros((rows, dv), dtype=np.float64)
    lse = np.full(rows, -np.inf, dtype=np.float64)
    live = np.isfinite(m)
    if live.any():
        w = np.exp(lse_parts[:, live] - m[None, live])
        wsum = w.sum(axis=0)
        out[live] = (w[:, :, None] * o_parts[:, live]).sum(axis=0) / wsum[:, None]
        lse[live] = m[live] + np.log(wsum)
    return out, lse


# ----------------------------------------------------------------------------
# PV skip (pv_threshold)
# ----------------------------------------------------------------------------

def attention_unit_pv_skip(q: np.ndarray, k: np.ndarray, v: np.ndarray, lut_row: Iterable[int],
                           i: int, blkq: int, blkk: int, scale: float, causal: bool,
                           pv_threshold: float, margins: Optional[list] = None):
    """Attention of q block ``i`` with the per-Q-tile PV skip ("Sparge
    Attention (Composable Kernel)" README, 'Not yet ported': pv_threshold
    per-Q-tile skip in the attention kernel, a pure performance feature).

    The kv blocks are visited in LUT order with a running row max m (the
    largest score of the blocks visited so far, -inf before the first).  A
    block whose every row has all its scores below m - pv_threshold (natural
    log units, the scores already scaled) contributes nothing to the P.V
    product; its probabilities still count in the softmax denominator, and the
    LSE is unchanged.  So every skipped probability is below e^-pv_threshold
    times the row's largest one.  Returns (O [rows, dv], LSE [rows], the list
    of skipped kv blocks).  ``margins``, if given, receives per visited block
    the smallest over rows of m - pv_threshold - (block max): the block is
    skipped when it is positive."""
    s_q, s_k = q.shape[0], k.shape[0]
    t = np.arange(i * blkq, min((i + 1) * blkq, s_q))
    rows, dv = len(t), v.shape[1]
    m = np.full(rows, -np.inf)
    l = np.zeros(rows)
    num = np.zeros((rows, dv))
    skipped = []
    for j in lut_row:
        keys = row_keys([j], blkk, s_k)
        s = scale * (q[t] @ k[keys].T)
        if causal:
            s = np.where(keys[None, :] <= t[:, None], s, -np.inf)
        tmax = s.max(axis=1)
        skip = bool(np.all(tmax < m - pv_threshold))
        if margins is not None:
            margins.append(float(np.min(m - pv_threshold - tmax)))
        m_new = np.maximum(m, tmax)
        live = np.isfinite(m_new)
        alpha = np.where(live, np.exp(np.where(live, m - m_new, 0.0)), 0.0)
        p = np.where(live[:, None], np.exp(s - np.where(live, m_new, 0.0)[:, None]), 0.0)
        l = l * alpha + p.sum(axis=1)
        num = num * alpha[:, None]
        if skip:
            skipped.append(int(j))
        else:
            num = num + p @ v[keys]
        m = m_new
    out = np.zeros((rows, dv))
    lse = np.full(rows, -np.inf)
    ok = l > 0
    out[ok] = num[ok] / l[ok, None]
    lse[ok] = m[ok] + np.log(l[ok])
    return out, lse, skipped


# ----------------------------------------------------------------------------
# Context parallelism over the kv blocks
# ----------------------------------------------------------------------------

def shard_lut_row(lut_row: Iterable[int], lo: int, hi: int) -> list:
    """The entries of a LUT row inside the kv-block range [lo, hi), in their
    order, re-based to the range (e - lo): the row as seen by the rank that
    holds K/V blocks lo .. hi - 1."""
    return [int(e) - lo for e in lut_row if lo <= int(e) < hi]


def context_parallel_unit(qh: np.ndarray, kg: np.ndarray, vg: np.ndarray, lut_row, i: int,
                          world: int, blkq: int, blkk: int, scale: float, causal: bool = False):
    """Partials of one q block under context parallelism over ``world`` ranks:
    rank r holds the kv blocks of split_bounds(nk, world)[r] (K/V rows
    [lo * blkk, min(hi * blkk, s_k))) and attends over its shard of the LUT
    row; under ``causal`` (queries and the full key sequence start at the same
    position) its local key index u is position lo * blkk + u, so the key
    offset of its mask is -lo * blkk.  Returns (O_parts [world, rows, dv],
    LSE_parts [world, rows]); ``combine`` of them is the attention of the
    whole row."""
    nk = (kg.shape[0] + blkk - 1) // blkk
    outs, lses = [], []
    for lo, hi in split_bounds(nk, world):
        r0, r1 = lo * blkk, min(hi * blkk, kg.shape[0])
        o, l = attention_unit(qh, kg[r0:r1], vg[r0:r1], shard_lut_row(lut_row, lo, hi), i,
                              blkq, blkk, scale, causal, key_offset=-lo * blkk)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


# ----------------------------------------------------------------------------
# Speculative two-pass attention
# ----------------------------------------------------------------------------

def speculative_two_pass_unit(qh: np.ndarray, k_spec: np.ndarray, v_spec: np.ndarray,
                              kg: np.ndarray, vg: np.ndarray, missed_row, i: int, blkq: int,
                              blkk: int, scale: float, causal_spec: bool = True):
    """The two-pass recipe of "Incremental_FlashAttention updating_log.md",
    Stage 5, for the rows of q block ``i``:
      pass 1 - dense attention over the caller-gathered speculative keys
               k_spec / v_spec [s_spec, *], causal with the queries aligned to
               the last s_q of them (key offset s_spec - s_q), so the block
               holding each query's own position is masked as usual;
      pass 2 - sparse attention over the missed kv blocks of the full K/V
               (``missed_row``: fully historical blocks, every key before the
               q block's first query, so no mask);
      combine - the Stage 1 merge of the two (O, LSE) partials.
    Returns (O [rows, dv], LSE [rows]) and the two partials."""
    s_q, s_spec = qh.shape[0], k_spec.shape[0]
    nspec = (s_spec + blkk - 1) // blkk
    o1, l1 = attention_unit(qh, k_spec, v_spec, range(nspec), i, blkq, blkk, scale, causal_spec,
                            key_offset=s_spec - s_q)
    o2, l2 = attention_unit(qh, kg, vg, missed_row, i, blkq, blkk, scale, False)
    o, l = combine(np.stack([o1, o2]), np.stack([l1, l2]))
    return o, l, (o1, l1), (o2, l2)


# ----------------------------------------------------------------------------
# Sparse decode (paged cache, token index lists)
# ----------------------------------------------------------------------------


def decode_rows(page_table: np.ndarray, idx: np.ndarray, page: int) -> np.ndarray:
    """Physical cache row of every listed token position: the row sits at
    offset pos mod page inside page page_table[c, pos div page] (paged KV
    addressing of ROCm/aiter pull 4919)."""
    pt = np.asarray(page_table, dtype=np.int64)
    pos = np.asarray(idx, dtype=np.int64)
    c = np.arange(pos.shape[0])[:, None]
    return pt[c, pos // page] * page + pos % page


def decode_attention(q: np.ndarray, kv: np.ndarray, dv: int, scale: float):
    """One query token per row of q [H, d] attending to the gathered rows kv
    [T, d]: K = kv, V = kv[:, :dv] (the latent plane).  Returns (O [H, dv],
    LSE [H])."""
    scores = scale * (q @ kv.T)
    return _softmax_attend(scores, kv[:, :dv])


def decode_partials(q: np.ndarray, kv: np.ndarray, dv: int, scale: float, num_splits: int):
    """Split-KV partials of one query: attention over each contiguous chunk of
    its gathered key list.  Returns (O_parts [S, H, dv], LSE_parts [S, H])."""
    outs, lses = [], []
    for lo, hi in split_bounds(kv.shape[0], num_splits):
        o, l = decode_attention(q, kv[lo:hi], dv, scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)
