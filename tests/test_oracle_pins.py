"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a closed form, a
brute-force enumeration on tiny inputs, a textbook / library routine
(torch scaled_dot_product_attention and logsumexp in float64), or an identity
the pages state (the combine identity of the Incremental_FlashAttention
updating_log, Stage 1).  The last tests plant mistakes in copies of oracle
functions and check that a pin catches each one.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import attention as oatt
from oracle import block_map as obm

RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------------------
# self-similarity and pooling
# ----------------------------------------------------------------------------


def brute_similarity(block):
    """Mean of cos(x_a, x_b) over all ordered pairs, in plain Python."""
    rows = [list(map(float, r)) for r in block]
    n = len(rows)
    norms = [math.sqrt(sum(v * v for v in r)) for r in rows]
    tot = 0.0
    for a in range(n):
        for b in range(n):
            if norms[a] == 0.0 or norms[b] == 0.0:
                continue
            tot += sum(x * y for x, y in zip(rows[a], rows[b])) / (norms[a] * norms[b])
    return tot / (n * n)


@pytest.mark.parametrize("n,d", [(64, 8), (5, 3), (17, 33)])
def test_self_similarity_matches_pairwise_cosines(n, d):
    for _ in range(3):
        blk = RNG.standard_normal((n, d)) + RNG.standard_normal(d)
        assert obm.self_similarity(blk) == pytest.approx(brute_similarity(blk), abs=1e-12)


def test_self_similarity_special_cases():
    row = RNG.standard_normal(16)
    same = np.tile(row, (64, 1))
    assert obm.self_similarity(same) == pytest.approx(1.0, abs=1e-14)
    half = RNG.standard_normal((32, 16))
    anti = np.empty((64, 16))
    anti[0::2], anti[1::2] = half, -half
    assert obm.self_similarity(anti) == pytest.approx(0.0, abs=1e-14)
    # a zero row contributes a zero unit vector: (n-1)^2 / n^2
    z = same.copy()
    z[3] = 0.0
    assert obm.self_similarity(z) == pytest.approx((63 / 64) ** 2, abs=1e-14)
    # independent noise averages out: E[sim] = 1/n for isotropic rows
    noise = RNG.standard_normal((64, 2048))
    assert obm.self_similarity(noise) == pytest.approx(1 / 64, abs=3e-3)


def test_pool_blocks_exact_means_with_partial_block():
    x = np.arange(7 * 2, dtype=np.float64).reshape(7, 2)  # 7 rows, blk = 3
    got = obm.pool_blocks(x, 3)
    want = []
    for j in range(3):
        rows = [list(map(Fraction, r)) for r in x[3 * j:3 * j + 3].astype(int)]
        want.append([sum(c) / len(rows) for c in zip(*rows)])
    assert got.shape == (3, 2)
    assert [[Fraction(v) for v in r] for r in got] == want


# ----------------------------------------------------------------------------
# eligibility, counts and selection
# ----------------------------------------------------------------------------


def test_eligibility_causal_is_lower_triangle():
    e = obm.eligible_mask(8, 8, 64, 64, True)
    assert (e == np.tril(np.ones((8, 8), dtype=bool))).all()
    assert (e.sum(axis=1) == np.arange(1, 9)).all()
    assert obm.eligible_mask(3, 5, 64, 64, False).all()
    # unequal blocks: q blocks of 128 see kv blocks of 64 up to 2i+1
    e2 = obm.eligible_mask(2, 4, 128, 64, True)
    assert e2.tolist() == [[True, True, False, False], [True, True, True, True]]


@pytest.mark.parametrize("topk,n,want", [(0.5, 8, 4), (0.1, 256, 26), (0.2, 256, 52),
                                         (0.4, 256, 103), (0.6, 256, 154), (1.0, 256, 256),
                                         (0.2, 5, 1), (0.2, 512, 103), (1e-6, 9, 1)])
def test_topk_count_table(topk, n, want):
    assert obm.topk_count(topk, n) == want


def _softmax(sc):
    fin = np.isfinite(sc)
    p = np.zeros_like(sc)
    e = np.exp(sc[fin] - sc[fin].max())
    p[fin] = e / e.sum()
    return p


def check_topk_bruteforce(select, sc, topk):
    """The chosen set is the lexicographically-first maximiser of total pooled
    probability among all sets of min(K, #finite) finite entries."""
    nk = sc.shape[0]
    fin = [j for j in range(nk) if np.isfinite(sc[j])]
    kk = min(obm.topk_count(topk, nk), len(fin))
    p = _softmax(sc)
    best, best_set = -1.0, None
    for comb in itertools.combinations(fin, kk):  # lexicographic order
        tot = sum(p[j] for j in comb)
        if tot > best + 1e-15:
            best, best_set = tot, comb
    got = tuple(np.nonzero(select(sc, topk, None, nk))[0])
    assert got == tuple(best_set), (got, best_set)


def check_cdf_bruteforce(select, sc, tau):
    """The chosen set has the smallest size m for which some m-subset of
    finite entries reaches mass tau, and is the top-m by probability (lower
    index on ties); everything finite when nothing reaches tau."""
    nk = sc.shape[0]
    fin = [j for j in range(nk) if np.isfinite(sc[j])]
    p = _softmax(sc)
    got = tuple(np.nonzero(select(sc, None, tau, nk))[0])
    want = tuple(fin)
    for m in range(1, len(fin) + 1):
        cands = [c for c in itertools.combinations(fin, m) if sum(p[j] for j in c) >= tau]
        if cands:
            bestmass = max(sum(p[j] for j in c) for c in cands)
            want = min(c for c in cands if sum(p[j] for j in c) >= bestmass - 1e-15)
            break
    assert got == tuple(sorted(want)), (got, want)


def _tiny_rows(seed):
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(40):
        nk = int(rng.integers(1, 9))
        sc = rng.standard_normal(nk) * 2.0
        if nk > 2:
            sc[rng.integers(0, nk)] = -np.inf
        if nk > 3 and rng.random() < 0.5:  # an exact tie
            a, b = rng.choice(nk, 2, replace=False)
            sc[b] = sc[a]
        rows.append(sc)
    return rows


@pytest.mark.parametrize("topk", [0.1, 0.25, 0.5, 0.75, 1.0])
def test_topk_selection_bruteforce(topk):
    for sc in _tiny_rows(1):
        check_topk_bruteforce(obm.select_row, sc, topk)


@pytest.mark.parametrize("tau", [0.3, 0.5, 0.8, 0.9, 0.99])
def test_cdf_selection_bruteforce(tau):
    for sc in _tiny_rows(2):
        check_cdf_bruteforce(obm.select_row, sc, tau)


def test_selection_special_cases():
    sc = np.array([0.3, 1.7, -np.inf, 1.7, -0.2])
    assert np.nonzero(obm.select_row(sc, 1e-6, None, 5))[0].tolist() == [1]  # argmax, low index
    assert np.nonzero(obm.select_row(sc, None, 1.0, 5))[0].tolist() == [0, 1, 3, 4]
    assert not obm.select_row(np.full(4, -np.inf), 0.5, None, 4).any()
    assert np.nonzero(obm.select_row(sc, 1.0, None, 5))[0].tolist() == [0, 1, 3, 4]


def test_block_map_hand_example():
    """A tiny worked example with exact rational pooled scores.

    blk = 2, d = 2.  q blocks pool to (1,0) and (0,1); k blocks pool to
    (2,0), (0,3), (1,1), (-1,0).  Scores (scale 1): row 0 = [2,0,1,-1],
    row 1 = [0,3,1,0].  topk 0.5 of 4 -> 2 per row: row 0 {0,2}, row 1 {1,2}.
    Every block is 'similar' (rows of a block are parallel, sim = 1 > 0.5).
    """
    q = np.array([[1, 0], [1, 0], [0, 1], [0, 1]], dtype=np.float64)
    k = np.array([[2, 0], [2, 0], [0, 3], [0, 3], [1, 1], [1, 1], [-1, 0], [-1, 0]],
                 dtype=np.float64)
    r = obm.block_map_head(q, k, 0.5, 0.5, None, 1.0, False, False, 2, 2)
    assert r["raw"].tolist() == [[2, 0, 1, -1], [0, 3, 1, 0]]
    assert r["lut"].tolist() == [[0, 2, -1, -1], [1, 2, -1, -1]]
    assert r["count"].tolist() == [2, 2]
    # causal + sink on the same data (q blocks and k blocks of equal size 2):
    # row 0 sees only kv block 0; row 1 sees 0,1 -> K = ceil(0.5*2) = 1 -> {1}, plus sink 0
    k2 = k[:4]
    r = obm.block_map_head(q, k2, 0.5, 0.5, None, 1.0, True, True, 2, 2)
    assert r["lut"].tolist() == [[0, -1], [0, 1]]
    # kv block 1 made dissimilar (antithetic rows): its column is forced on
    k3 = k2.copy()
    k3[2], k3[3] = [1.0, 0.0], [-1.0, 0.0]
    r = obm.block_map_head(q, k3, 0.5, 0.5, None, 1.0, False, False, 2, 2)
    assert r["simk"].tolist() == [1.0, 0.0]
    assert r["lut"].tolist() == [[0, 1], [0, 1]]
    # a dissimilar q block keeps every eligible column
    q3 = q.copy()
    q3[0], q3[1] = [0.0, 2.0], [0.0, -2.0]
    r = obm.block_map_head(q3, k, 0.5, 0.25, None, 1.0, False, False, 2, 2)
    assert r["lut"][0].tolist() == [0, 1, 2, 3]
    assert r["count"][1] == 1 and r["lut"][1, 0] == 1


def _gqa_hand_inputs():
    """b = 1, hq = 4 query heads on hk = 2 KV heads, blk = 2, d = 2, s = 4.

    Every query head pools to qbar_0 = (1, 0), qbar_1 = (0, 1).  KV head 0
    pools to kbar = (2, 0), (0, 3) -> scores [[2, 0], [0, 3]]; KV head 1 to
    (0, 1), (1, 0) -> scores [[0, 1], [1, 0]] (scale 1).  Rows of every block
    are parallel, so every self-similarity is exactly 1."""
    qh = np.array([[1, 0], [1, 0], [0, 1], [0, 1]], dtype=np.float64)
    q = np.stack([qh] * 4)[None]
    k0 = np.array([[2, 0], [2, 0], [0, 3], [0, 3]], dtype=np.float64)
    k1 = np.array([[0, 1], [0, 1], [1, 0], [1, 0]], dtype=np.float64)
    k = np.stack([k0, k1])[None]
    return q, k


# per query head h: KV head h // 2, topk, simthreshd1 and the LUT rows
GQA_TOPK = np.array([0.5, 1.0, 0.5, 0.5], dtype=np.float32)
GQA_THETA = np.array([0.5, 0.5, 0.5, 2.0], dtype=np.float32)
GQA_TOPK_LUT = [
    [[0, -1], [1, -1]],  # h0: KV head 0, one block per row: the row argmax
    [[0, 1], [0, 1]],    # h1: KV head 0, topk 1.0: both blocks
    [[1, -1], [0, -1]],  # h2: KV head 1, one block per row
    [[0, 1], [0, 1]],    # h3: KV head 1, theta 2 > sim 1: every row and column forced
]
GQA_CDF = np.array([0.5, 0.95, 0.5, 0.8], dtype=np.float32)
GQA_CDF_LUT = [
    [[0, -1], [1, -1]],  # h0: p = (0.881, 0.119) and (0.047, 0.953): the top entry reaches 0.5
    [[0, 1], [1, -1]],   # h1: 0.881 < 0.95 takes both; 0.953 >= 0.95 takes one
    [[1, -1], [0, -1]],  # h2: KV head 1, p = (0.269, 0.731): the top entry reaches 0.5
    [[0, 1], [0, 1]],    # h3: 0.731 < 0.8 takes both
]


def test_per_head_hyperparameters_and_gqa_mapping_hand_example():
    """Per-head topk / simthreshd1 / cdfthreshd ("Sparge Attention (Composable
    Kernel)" README, 'Status vs Upstream') and the GQA mapping query head
    j -> KV head j / (hq / hk) (ROCm/aiter pull 6841), on values worked by
    hand.  Query heads 0 and 1 share KV head 0, heads 2 and 3 share KV head 1;
    the two KV heads rank the kv blocks in opposite orders, so a wrong KV head
    changes a LUT, and every head's hyperparameters differ from head 0's where
    that changes its LUT."""
    q, k = _gqa_hand_inputs()
    r = oracle.sparge_block_map(q, k, GQA_TOPK, None, GQA_THETA, 1.0, False, False, 2, 2)
    assert r["lut"][0].tolist() == GQA_TOPK_LUT
    assert r["count"][0].tolist() == [[1, 1], [2, 2], [1, 1], [2, 2]]
    r = oracle.sparge_block_map(q, k, None, GQA_CDF, np.full(4, 0.5, np.float32), 1.0, False,
                                False, 2, 2)
    assert r["lut"][0].tolist() == GQA_CDF_LUT
    # the closed-form probabilities behind the cdf rows
    assert math.exp(2) / (math.exp(2) + 1) == pytest.approx(0.8808, abs=1e-4)
    assert math.exp(3) / (math.exp(3) + 1) == pytest.approx(0.9526, abs=1e-4)


def test_planted_gqa_and_per_head_mistakes_are_caught(monkeypatch):
    """Three plausible slips in sparge_block_map, each caught by the hand
    example: the KV head taken as h % hk instead of h // (hq / hk), head 0's
    topk (or cdfthreshd) used for every head, head 0's simthreshd1 used for
    every head."""
    real_head = obm.block_map_head

    def run(q, k, topk, cdf, theta):
        return oracle.sparge_block_map(q, k, topk, cdf, theta, 1.0, False, False, 2, 2)["lut"][0]

    q, k = _gqa_hand_inputs()
    # KV head h % hk: rebuild the call with the permuted KV heads
    hq, hk = 4, 2
    k_mod = np.stack([k[0, h % hk] for h in range(hq)])[None]
    q_one = q  # one KV head per query head: ratio 1 reads k_mod[h] for head h
    got = run(q_one, k_mod, GQA_TOPK, None, GQA_THETA)
    assert got.tolist() != GQA_TOPK_LUT
    # head 0's selection parameter for every head
    got = run(q, k, np.full(4, GQA_TOPK[0], np.float32), None, GQA_THETA)
    assert got.tolist() != GQA_TOPK_LUT
    got = run(q, k, None, np.full(4, GQA_CDF[0], np.float32), np.full(4, 0.5, np.float32))
    assert got.tolist() != GQA_CDF_LUT
    # head 0's threshold for every head, planted inside the per-head call
    calls = []

    def head_with_theta0(qh, kg, theta, *a, **kw):
        calls.append(theta)
        return real_head(qh, kg, float(GQA_THETA[0]), *a, **kw)

    monkeypatch.setattr(obm, "block_map_head", head_with_theta0)
    got = run(q, k, GQA_TOPK, None, GQA_THETA)
    assert calls == [float(t) for t in GQA_THETA]  # the oracle passes each head its own
    assert got.tolist() != GQA_TOPK_LUT


def test_smooth_k_hand_example():
    """K smoothing subtracts the mean key row of the sequence (README 'Not yet
    ported': pre-pool k -= km).  blk = 2, d = 2, two kv blocks whose rows are
    the constants a = (3, 1) and b = (1, 1): km = (2, 1), the smoothed rows are
    (1, 0) and (-1, 0), each block still parallel (sim 1), pooled to (1, 0)
    and (-1, 0).  With q pooled to (1, 1) and (-1, 3) the raw scores are
    [[4, 2], [0, 2]] without smoothing and [[1, -1], [-1, 1]] with it: each
    row moves by the constant -qbar_i . km, so the ranking, the softmax and the
    LUT are unchanged ([[0], [1]] at topk 0.5).  Smoothing changes the map
    through the self-similarity alone: identical blocks a = b smooth to zero
    rows, sim 0, and both columns are forced on."""
    q = np.array([[1, 1], [1, 1], [-1, 3], [-1, 3]], dtype=np.float64)
    k = np.array([[3, 1], [3, 1], [1, 1], [1, 1]], dtype=np.float64)
    assert obm.smooth_keys(k).tolist() == [[1, 0], [1, 0], [-1, 0], [-1, 0]]
    r0 = obm.block_map_head(q, k, 0.5, 0.5, None, 1.0, False, False, 2, 2)
    r1 = obm.block_map_head(q, k, 0.5, 0.5, None, 1.0, False, False, 2, 2, smooth_k=True)
    assert r0["raw"].tolist() == [[4, 2], [0, 2]]
    assert r1["raw"].tolist() == [[1, -1], [-1, 1]]
    assert r1["kbar"].tolist() == [[1, 0], [-1, 0]]
    assert r1["simk"].tolist() == [1.0, 1.0]
    assert r0["lut"].tolist() == r1["lut"].tolist() == [[0, -1], [1, -1]]
    same = np.array([[3, 1]] * 4, dtype=np.float64)
    r2 = obm.block_map_head(q, same, 0.5, 0.5, None, 1.0, False, False, 2, 2)
    r3 = obm.block_map_head(q, same, 0.5, 0.5, None, 1.0, False, False, 2, 2, smooth_k=True)
    assert np.allclose(r2["simk"], [1.0, 1.0], atol=1e-12)
    assert r2["lut"].tolist() == [[0, -1], [0, -1]]
    assert r3["simk"].tolist() == [0.0, 0.0] and r3["lut"].tolist() == [[0, 1], [0, 1]]


def test_smooth_k_invariant_to_a_common_key_offset():
    """Smoothed keys do not depend on a row c added to every key, so neither
    does the smoothed block map; the unsmoothed map does (through the
    self-similarity of the shifted rows)."""
    rng = np.random.default_rng(7)
    s, d, blk = 256, 16, 16
    q = rng.standard_normal((s, d))
    k = np.repeat(rng.standard_normal((s // blk, d)), blk, axis=0) + 0.8 * rng.standard_normal((s, d))
    c = 6.0 * rng.standard_normal(d)
    args = (0.3, 0.25, None, 0.25, False, False, blk, blk)
    a = obm.block_map_head(q, k, *args, smooth_k=True)
    b = obm.block_map_head(q, k + c, *args, smooth_k=True)
    assert np.array_equal(a["lut"], b["lut"]) and np.array_equal(a["count"], b["count"])
    assert np.allclose(a["raw"], b["raw"], atol=1e-9) and np.allclose(a["simk"], b["simk"], atol=1e-12)
    # the smoothed pooled means of equal-size blocks sum to zero
    assert np.abs(a["kbar"].sum(axis=0)).max() < 1e-12
    u = obm.block_map_head(q, k, *args)
    v = obm.block_map_head(q, k + c, *args)
    assert not np.allclose(u["simk"], v["simk"], atol=1e-3)


def test_all_dissimilar_gives_dense_map():
    cfg = synth.C1
    x = synth.prefill(cfg)
    r = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, 0.1), None,
                                synth.per_head(cfg, 2.0), cfg.scale, False, False,
                                dtype="f16")
    assert r["block_map"].all()
    assert (r["count"] == cfg.nq).all()


def test_generated_blocks_clear_the_threshold():
    """The centroid-plus-noise blocks (diffuse ones included) sit far above
    simthreshd1 = 0.001, so nothing is forced at the configured threshold;
    the antithetic variant drives diffuse blocks to exactly zero."""
    cfg = synth.C1
    x = synth.prefill(cfg)
    q = synth.bits_to_f64(x["q"], "f16")
    sims = [obm.self_similarity(q[0, 0, i * 64:(i + 1) * 64]) for i in range(cfg.nq)]
    assert min(sims) > 0.1
    xa = synth.prefill(cfg.replace(antithetic_diffuse=True))
    qa = synth.bits_to_f64(xa["q"], "f16")
    sa = sorted(obm.self_similarity(qa[0, 0, i * 64:(i + 1) * 64]) for i in range(cfg.nq))
    assert sa[0] == 0.0 and sa[1] == 0.0 and sa[2] > 0.5


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------


def _sdpa(q, k, v, scale, causal=False):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale,
                                                         is_causal=causal)
    return o[0, 0].numpy()


def _loop_row(qrow, k, v, scale, upto=None):
    """One query row, written as plain loops with math.exp."""
    n = k.shape[0] if upto is None else upto
    sc = [scale * float(qrow @ k[u]) for u in range(n)]
    m = max(sc)
    w = [math.exp(x - m) for x in sc]
    l = sum(w)
    o = sum(w[u] * v[u] for u in range(n)) / l
    return o, m + math.log(l)


def test_topk_one_is_dense_attention():
    cfg = synth.C1
    x = synth.prefill(cfg)
    q, k, v = (synth.bits_to_f64(x[t], "f16") for t in ("q", "k", "v"))
    bm = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, 1.0), None,
                                 synth.per_head(cfg, cfg.simthreshd1), cfg.scale, False,
                                 False, dtype="f16")
    assert (bm["count"] == cfg.nq).all()
    res = oracle.sparse_fmha(q, k, v, bm["lut"], bm["count"], cfg.scale, False)
    for h in range(cfg.hq):
        o_full = np.concatenate([res[(0, h, i)][0] for i in range(cfg.nq)])
        lse_full = np.concatenate([res[(0, h, i)][1] for i in range(cfg.nq)])
        ref = _sdpa(q[0, h], k[0, h], v[0, h], cfg.scale)
        assert np.abs(o_full - ref).max() < 1e-12
        for t in (0, 77, 511):
            o_t, lse_t = _loop_row(q[0, h, t], k[0, h], v[0, h], cfg.scale)
            assert np.abs(o_full[t] - o_t).max() < 1e-12
            assert abs(lse_full[t] - lse_t) < 1e-12
        sc = torch.from_numpy(q[0, h] @ k[0, h].T * cfg.scale)
        assert np.abs(lse_full - torch.logsumexp(sc, dim=-1).numpy()).max() < 1e-12


def test_causal_topk_one_is_causal_attention_with_sink():
    cfg = synth.C1.replace(causal=True, attention_sink=True, topk=1.0, hq=4, hk=2)
    x = synth.prefill(cfg)
    q, k, v = (synth.bits_to_f64(x[t], "f16") for t in ("q", "k", "v"))
    bm = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, 1.0), None,
                                 synth.per_head(cfg, cfg.simthreshd1), cfg.scale, True,
                                 True, dtype="f16")
    nq = cfg.nq
    assert (bm["count"] == np.arange(1, nq + 1)[None, None, :]).all()
    assert (bm["lut"][..., 0] == 0).all()
    res = oracle.sparse_fmha(q, k, v, bm["lut"], bm["count"], cfg.scale, True)
    for h in range(cfg.hq):
        g = h // 2
        o_full = np.concatenate([res[(0, h, i)][0] for i in range(nq)])
        ref = _sdpa(q[0, h], k[0, g], v[0, g], cfg.scale, causal=True)
        assert np.abs(o_full - ref).max() < 1e-12
        o_t, lse_t = _loop_row(q[0, h, 130], k[0, g], v[0, g], cfg.scale, upto=131)
        assert np.abs(o_full[130] - o_t).max() < 1e-12
        assert abs(res[(0, h, 2)][1][2] - lse_t) < 1e-12


def test_sink_column_under_small_topk():
    cfg = synth.C1.replace(causal=True, attention_sink=True, topk=0.1)
    x = synth.prefill(cfg)
    bm = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, 0.1), None,
                                 synth.per_head(cfg, cfg.simthreshd1), cfg.scale, True,
                                 True, dtype="f16")
    assert (bm["lut"][..., 0] == 0).all()
    for i in range(cfg.nq):
        row = bm["lut"][0, 0, i, :bm["count"][0, 0, i]]
        assert (row <= i).all() and (np.diff(row) > 0).all()


def test_sparse_lse_is_logsumexp_of_selected_scores():
    cfg = synth.C1
    x = synth.prefill(cfg)
    q, k, v = (synth.bits_to_f64(x[t], "f16") for t in ("q", "k", "v"))
    lut_row = [1, 4, 6]
    o, lse = oatt.attention_unit(q[0, 1], k[0, 1], v[0, 1], lut_row, 3, 64, 64, cfg.scale,
                                 False)
    keys = np.concatenate([np.arange(j * 64, j * 64 + 64) for j in lut_row])
    sc = torch.from_numpy(cfg.scale * q[0, 1, 192:256] @ k[0, 1, keys].T)
    assert np.abs(lse - torch.logsumexp(sc, -1).numpy()).max() < 1e-12
    ref = _sdpa(q[0, 1, 192:256], k[0, 1, keys], v[0, 1, keys], cfg.scale)
    assert np.abs(o - ref).max() < 1e-12


def test_empty_row_gives_zero_and_minus_inf():
    q = RNG.standard_normal((128, 8))
    o, lse = oatt.attention_unit(q, q, q, [], 1, 64, 64, 0.3, False)
    assert o.shape == (64, 8) and (o == 0).all() and np.isneginf(lse).all()


# ----------------------------------------------------------------------------
# split-KV and the combine identity
# ----------------------------------------------------------------------------


def _splits(nb):
    allb = list(range(nb))
    return {
        "interleaved": (allb[0::2], allb[1::2]),
        "spec_heavy": (allb[: nb - 2], allb[nb - 2:]),
        "miss_heavy": (allb[:2], allb[2:]),
        "contiguous_miss": ([b for b in allb if not 2 <= b < 5], [2, 3, 4]),
    }


@pytest.mark.parametrize("seqlen_q", [1, 4, 16])
@pytest.mark.parametrize("block_size", [32, 64, 128])
@pytest.mark.parametrize("split", ["interleaved", "spec_heavy", "miss_heavy",
                                   "contiguous_miss"])
def test_combine_identity(seqlen_q, block_size, split):
    """FA(A u B) == Combine(FA(A), FA(B)) to 1e-10 in fp64, on the grid of the
    updating_log's Stage 1 (seqlen_q x block_size x four splits)."""
    rng = np.random.default_rng(seqlen_q * 1000 + block_size)
    nb, d = 8, 32
    q = rng.standard_normal((seqlen_q, d))
    k = rng.standard_normal((nb * block_size, d))
    v = rng.standard_normal((nb * block_size, d))
    a, b = _splits(nb)[split]
    full = oatt.attention_unit(q, k, v, sorted(a + b), 0, seqlen_q, block_size, 0.2, False)
    pa = oatt.attention_unit(q, k, v, a, 0, seqlen_q, block_size, 0.2, False)
    pb = oatt.attention_unit(q, k, v, b, 0, seqlen_q, block_size, 0.2, False)
    o, lse = oracle.combine(np.stack([pa[0], pb[0]]), np.stack([pa[1], pb[1]]))
    assert np.abs(o - full[0]).max() < 1e-10
    assert np.abs(lse - full[1]).max() < 1e-10
    o2, lse2 = oracle.combine(np.stack([pb[0], pa[0]]), np.stack([pb[1], pa[1]]))
    assert np.abs(o2 - o).max() < 1e-10 and np.abs(lse2 - lse).max() < 1e-10


def test_combine_empty_partials():
    rng = np.random.default_rng(5)
    o1 = rng.standard_normal((4, 8))
    l1 = rng.standard_normal(4)
    empty_o, empty_l = np.zeros((4, 8)), np.full(4, -np.inf)
    o, l = oracle.combine(np.stack([o1, empty_o]), np.stack([l1, empty_l]))
    assert np.abs(o - o1).max() < 1e-15 and np.abs(l - l1).max() < 1e-15
    o, l = oracle.combine(np.stack([empty_o, empty_o]), np.stack([empty_l, empty_l]))
    assert (o == 0).all() and np.isneginf(l).all()
    # a row empty in one partial only
    l1b = l1.copy()
    l1b[2] = -np.inf
    o, l = oracle.combine(np.stack([o1, empty_o]), np.stack([l1b, empty_l]))
    assert (o[2] == 0).all() and np.isneginf(l[2])


def test_combine_closed_form_two_partials():
    """Two partials with LSE a, b: weights e^a/(e^a+e^b), LSE = ln(e^a+e^b)."""
    o1, o2 = np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]])
    a, b = math.log(3.0), math.log(1.0)
    o, l = oracle.combine(np.stack([o1, o2]), np.array([[a], [b]]))
    assert np.abs(o[0] - [0.75, 0.25]).max() < 1e-15
    assert abs(l[0] - math.log(4.0)) < 1e-15


@pytest.mark.parametrize("n,S,sizes", [(10, 4, [3, 3, 2, 2]), (3, 8, [1, 1, 1, 0, 0, 0, 0, 0]),
                                       (12, 3, [4, 4, 4]), (0, 2, [0, 0]), (7, 1, [7])])
def test_split_bounds_table(n, S, sizes):
    b = oracle.split_bounds(n, S)
    assert [hi - lo for lo, hi in b] == sizes
    assert b[0][0] == 0 and b[-1][1] == n
    assert all(b[s][1] == b[s + 1][0] for s in range(S - 1))


@pytest.mark.parametrize("S", [2, 3, 4, 8])
def test_split_partials_combine_to_the_full_row(S):
    rng = np.random.default_rng(S)
    q = rng.standard_normal((256, 32))
    k = rng.standard_normal((512, 32))
    v = rng.standard_normal((512, 16))
    row = [0, 2, 3, 5, 7]
    parts = oatt.split_partials_unit(q, k, v, row, 2, S, 64, 64, 0.25, True)
    o, l = oracle.combine(*parts)
    ref = oatt.attention_unit(q, k, v, row, 2, 64, 64, 0.25, True)
    assert np.abs(o - ref[0]).max() < 1e-10 and np.abs(l - ref[1]).max() < 1e-10


# ----------------------------------------------------------------------------
# PV skip (pv_threshold)
# ----------------------------------------------------------------------------

_PV_Q = np.array([[1.0]])
_PV_K = np.array([[2.0], [2.0], [-3.0], [-3.0]])       # block 0 scores 2, block 1 scores -3
_PV_V = np.array([[1.0], [1.0], [10.0], [10.0]])


def test_pv_skip_hand_example():
    den = 2 * math.exp(2) + 2 * math.exp(-3)
    o, l, sk = oatt.attention_unit_pv_skip(_PV_Q, _PV_K, _PV_V, [0, 1], 0, 1, 2, 1.0, False, 4.0)
    assert sk == [1]                                        # -3 < 2 - 4
    assert abs(o[0, 0] - 2 * math.exp(2) / den) < 1e-14
    assert abs(l[0] - math.log(den)) < 1e-14                # the denominator keeps block 1
    o, l, sk = oatt.attention_unit_pv_skip(_PV_Q, _PV_K, _PV_V, [0, 1], 0, 1, 2, 1.0, False, 6.0)
    assert sk == [] and abs(o[0, 0] - (2 * math.exp(2) + 20 * math.exp(-3)) / den) < 1e-14


def test_pv_skip_uses_the_running_max_in_lut_order():
    # block 1 first: nothing was visited before it, and block 0 raises the max
    o, _, sk = oatt.attention_unit_pv_skip(_PV_Q, _PV_K, _PV_V, [1, 0], 0, 1, 2, 1.0, False, 4.0)
    full = oatt.attention_unit(_PV_Q, _PV_K, _PV_V, [1, 0], 0, 1, 2, 1.0, False)
    assert sk == [] and abs(o[0, 0] - full[0][0, 0]) < 1e-14


def test_pv_skip_needs_every_row_of_the_q_tile():
    q = np.array([[1.0], [-1.0]])       # row 1 scores block 0 at -2 and block 1 at 3
    _, _, sk = oatt.attention_unit_pv_skip(q, _PV_K, _PV_V, [0, 1], 0, 2, 2, 1.0, False, 4.0)
    assert sk == []


@pytest.mark.parametrize("causal", [False, True])
def test_pv_skip_infinite_threshold_is_plain_attention(causal):
    rng = np.random.default_rng(11)
    q, k, v = (rng.standard_normal((256, 16)) for _ in range(3))
    row = [0, 1, 2, 3] if causal else [3, 0, 2]
    o, l, sk = oatt.attention_unit_pv_skip(q, k, v, row, 3, 64, 64, 0.5, causal, math.inf)
    ref = oatt.attention_unit(q, k, v, row, 3, 64, 64, 0.5, causal)
    assert sk == []
    assert np.abs(o - ref[0]).max() < 1e-12 and np.abs(l - ref[1]).max() < 1e-12


def test_pv_skip_error_bound():
    # large score spread: blocks whose every score is far below the running max
    rng = np.random.default_rng(12)
    q = rng.standard_normal((64, 16))
    k = rng.standard_normal((512, 16)) * np.repeat(rng.uniform(0.1, 3.0, 8), 64)[:, None]
    v = rng.standard_normal((512, 8))
    row = list(range(8))
    ref = oatt.attention_unit(q, k, v, row, 0, 64, 64, 1.0, False)
    for tau in (0.5, 2.0, 5.0):
        o, l, sk = oatt.attention_unit_pv_skip(q, k, v, row, 0, 64, 64, 1.0, False, tau)
        assert np.abs(l - ref[1]).max() < 1e-12                    # LSE unchanged
        bound = 64 * len(sk) * math.exp(-tau) * np.abs(v).max()
        assert np.abs(o - ref[0]).max() <= bound + 1e-12
    assert oatt.attention_unit_pv_skip(q, k, v, row, 0, 64, 64, 1.0, False, 0.5)[2]  # skips some


def test_planted_pv_skip_mistake_is_caught(monkeypatch):
    """Testing each block against the final row max instead of the running
    max skips block 1 even when it is visited first: the order pin fails."""
    real = oatt.attention_unit_pv_skip

    def final_max(q, k, v, lut_row, i, blkq, blkk, scale, causal, tau):
        t = np.arange(i * blkq, min((i + 1) * blkq, q.shape[0]))
        keys = oatt.row_keys(lut_row, blkk, k.shape[0])
        mfin = (scale * (q[t] @ k[keys].T)).max(axis=1)
        o, l, _ = real(q, k, v, lut_row, i, blkq, blkk, scale, causal, math.inf)
        sk = []
        for j in lut_row:
            kj = oatt.row_keys([j], blkk, k.shape[0])
            if np.all((scale * (q[t] @ k[kj].T)).max(axis=1) < mfin - tau):
                sk.append(j)
        return o, l, sk

    monkeypatch.setattr(oatt, "attention_unit_pv_skip", final_max)
    with pytest.raises(AssertionError):
        test_pv_skip_uses_the_running_max_in_lut_order()


# ----------------------------------------------------------------------------
# fp8 (e4m3) Q/K
# ----------------------------------------------------------------------------

from oracle import fp8 as ofp8  # noqa: E402


def test_e4m3_value_table():
    tab = oracle.e4m3_values()
    assert len(tab) == 127 and (np.diff(tab) > 0).all()
    assert tab[0] == 0.0 and tab[1] == 2.0 ** -9 and tab[7] == 7 * 2.0 ** -9
    assert tab[8] == 2.0 ** -6 and tab[-1] == 448.0 and tab[-2] == 416.0
    assert tab[np.searchsorted(tab, 1.0)] == 1.0 and tab[np.searchsorted(tab, 1.0) + 1] == 1.125


def test_e4m3_rounding_hand_cases():
    x = np.array([1.0625, 1.1875, 464.0, 500.0, 1e30, 2.0 ** -10, 3 * 2.0 ** -11, -1.0625,
                  -448.0, 0.0, 17.0, 18.0])
    want = [1.0, 1.25, 448.0, 448.0, 448.0, 0.0, 2.0 ** -9, -1.0, -448.0, 0.0, 16.0, 18.0]
    assert oracle.round_e4m3(x).tolist() == want


def test_e4m3_rounding_matches_torch_cast_in_range():
    # a library routine for the in-range case: ties, subnormals, every binade
    rng = np.random.default_rng(21)
    tab = oracle.e4m3_values()
    mids = (tab[1:] + tab[:-1]) / 2                     # exact ties
    x = np.concatenate([tab, mids, rng.uniform(-448, 448, 20000),
                        rng.uniform(-2.0 ** -5, 2.0 ** -5, 20000), -mids])
    x = x.astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x).float().to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(oracle.round_e4m3(x), want)


def test_e4m3_block_quantisation_is_lossless_on_representable_blocks():
    rng = np.random.default_rng(22)
    tab = oracle.e4m3_values()
    for k2 in (-12, 0, 5):
        codes = rng.choice(tab, (64, 32)) * rng.choice([-1.0, 1.0], (64, 32))
        codes[3, 7] = 448.0                                # amax = 448 * 2^k2
        x = codes * 2.0 ** k2
        vals, qs = oracle.quantize_block_e4m3(x)
        assert qs == 2.0 ** k2 and np.array_equal(vals * qs, x)


def test_e4m3_scales_are_per_block():
    # a tiny block next to a large one keeps its own relative precision
    rng = np.random.default_rng(23)
    x = rng.standard_normal((128, 16))
    x[64:] *= 2.0 ** -20
    vals, qs = oracle.quantize_blocks_e4m3(x, 64)
    rel = np.abs(vals * np.repeat(qs, 64)[:, None] - x) / np.abs(x)
    assert rel[np.abs(x) > 1e-3 * np.abs(x).max(axis=1, keepdims=True)].max() <= 2.0 ** -4


def _fp8_case(seed=24):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((256, 32)), rng.standard_normal((256, 32)), \
        rng.standard_normal((256, 16))
    return q, k, v


def test_fp8_attention_equals_plain_attention_on_representable_inputs():
    rng = np.random.default_rng(25)
    tab = oracle.e4m3_values()

    def rep(n):  # 64-row blocks of e4m3 values times a power of two, amax 448 * 2^k
        x = rng.choice(tab, (n, 32)) * rng.choice([-1.0, 1.0], (n, 32))
        for b0 in range(0, n, 64):
            x[b0, 0] = 448.0
            x[b0:b0 + 64] *= 2.0 ** int(rng.integers(-9, -5))
        return x

    q, k = rep(256), rep(256)
    v = rng.standard_normal((256, 16))
    for causal in (False, True):
        row = [0, 1, 2] if causal else [3, 0, 2]
        o8 = oracle.attention_unit_fp8(q, k, v, row, 2, 64, 64, 0.25, causal)
        ref = oracle.attention_unit(q, k, v, row, 2, 64, 64, 0.25, causal)
        assert np.abs(o8[0] - ref[0]).max() < 1e-12 and np.abs(o8[1] - ref[1]).max() < 1e-12


def test_fp8_score_and_lse_error_bound():
    q, k, v = _fp8_case()
    row = [0, 1, 3]
    cq, sq = oracle.quantize_block_e4m3(q[128:192])
    # |x - qscale * code| <= 2^-4 |x| for normal codes, <= 2^-10 qscale below them
    for x in (q[128:192], k[0:64]):
        c, s = oracle.quantize_block_e4m3(x)
        err = np.abs(c * s - x)
        assert (err <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s) * (1 + 1e-6)).all()
    o8, l8 = oracle.attention_unit_fp8(q, k, v, row, 2, 64, 64, 0.2, False)
    o, l = oracle.attention_unit(q, k, v, row, 2, 64, 64, 0.2, False)
    # score error bound from the element bounds; the LSE moves by at most the
    # largest score error (logsumexp is 1-Lipschitz in the max norm)
    keys = oatt.row_keys(row, 64, 256)
    dq = np.maximum(2.0 ** -4 * np.abs(q[128:192]), 2.0 ** -10 * sq)
    dk = np.concatenate([np.maximum(2.0 ** -4 * np.abs(k[j * 64:(j + 1) * 64]),
                                    2.0 ** -10 * oracle.quantize_block_e4m3(k[j * 64:(j + 1) * 64])[1])
                         for j in row])
    aq, ak = np.abs(q[128:192]), np.abs(k[keys])
    bound = 0.2 * (aq @ dk.T + dq @ ak.T + dq @ dk.T)
    assert np.abs(l8 - l).max() <= bound.max()
    assert np.abs(l8 - l).max() > 0                       # the quantisation does change it


def test_planted_fp8_mistakes_are_caught(monkeypatch):
    # one scale for the whole tensor instead of one per block
    real = ofp8.quantize_block_e4m3
    big = {}

    def per_tensor(x):
        vals, qs = real(x)
        qs_t = big.setdefault("s", qs)
        return oracle.round_e4m3(np.asarray(x, np.float64) / qs_t), qs_t

    monkeypatch.setattr(ofp8, "quantize_block_e4m3", per_tensor)
    with pytest.raises(AssertionError):
        test_e4m3_scales_are_per_block()
    monkeypatch.undo()
    # rounding ties toward zero (the first nearest value) instead of to the even code
    def ties_down(x):
        a = np.minimum(np.abs(np.asarray(x, np.float64)), oracle.E4M3_MAX)
        return np.copysign(ofp8._TABLE[np.abs(a[..., None] - ofp8._TABLE).argmin(-1)], x)

    monkeypatch.setattr(oracle, "round_e4m3", ties_down)
    with pytest.raises(AssertionError):
        test_e4m3_rounding_hand_cases()


# ----------------------------------------------------------------------------
# context parallelism over the kv blocks
# ----------------------------------------------------------------------------

def test_shard_lut_row_hand_example():
    row = [0, 2, 3, 5, 7]
    assert oatt.shard_lut_row(row, 0, 2) == [0]
    assert oatt.shard_lut_row(row, 2, 6) == [0, 1, 3]
    assert oatt.shard_lut_row(row, 6, 8) == [1]
    assert oatt.shard_lut_row(row, 8, 9) == []


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_shards_partition_every_row(world):
    rng = np.random.default_rng(world)
    nk = 13
    bounds = oracle.split_bounds(nk, world)
    for _ in range(200):
        row = sorted(rng.choice(nk, size=int(rng.integers(0, nk + 1)), replace=False).tolist())
        back = []
        for lo, hi in bounds:
            sh = oatt.shard_lut_row(row, lo, hi)
            assert all(0 <= e < hi - lo for e in sh)
            assert all(a < b for a, b in zip(sh, sh[1:]))
            back += [e + lo for e in sh]
        assert back == row


def _cp_case(world):
    rng = np.random.default_rng(100 + world)
    q = rng.standard_normal((256, 32))
    k = rng.standard_normal((1000, 32))       # 16 kv blocks, the last one 40 rows
    v = rng.standard_normal((1000, 16))
    row = [1, 4, 5, 6, 15]                      # no block of 7 .. 14: some ranks empty
    parts = oatt.context_parallel_unit(q, k, v, row, 3, world, 64, 64, 0.3)
    ref = oatt.attention_unit(q, k, v, row, 3, 64, 64, 0.3, False)
    return parts, ref


@pytest.mark.parametrize("world", [2, 3, 5])
def test_context_parallel_combines_to_the_full_row(world):
    (o_parts, l_parts), ref = _cp_case(world)
    assert o_parts.shape[0] == world
    o, l = oracle.combine(o_parts, l_parts)
    assert np.abs(o - ref[0]).max() < 1e-10 and np.abs(l - ref[1]).max() < 1e-10
    if world == 5:   # blocks 7 .. 9 and 10 .. 12 hold no entry: empty partials
        assert np.isneginf(l_parts[2]).all() and (o_parts[2] == 0).all()


def test_planted_cp_mistake_is_caught(monkeypatch):
    """A shard that keeps the global block index (no re-basing to the rank's
    own K rows) attends over the wrong keys: the combine pin fails."""
    monkeypatch.setattr(oatt, "shard_lut_row",
                        lambda row, lo, hi: [int(e) for e in row if lo <= int(e) < hi])
    with pytest.raises(AssertionError):
        test_context_parallel_combines_to_the_full_row(2)


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------


# ----------------------------------------------------------------------------
# causal key offset, speculative two-pass, causal context parallelism
# ----------------------------------------------------------------------------


def _masked_sdpa(q, k, v, scale, visible):
    """torch scaled_dot_product_attention (fp64) with an explicit boolean mask."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), attn_mask=torch.from_numpy(visible)[None, None], scale=scale)
    return o[0, 0].numpy()


@pytest.mark.parametrize("s_q,s_k,off", [(192, 192, 0), (100, 260, 160), (128, 320, -70),
                                          (150, 150, 35)])
def test_causal_key_offset_matches_masked_sdpa(s_q, s_k, off):
    """Key u visible to query t iff u <= t + key_offset, checked against sdpa
    with that mask written out; rows without a visible key give (0, -inf)."""
    rng = np.random.default_rng(s_q + s_k)
    d = 16
    q, k, v = (rng.standard_normal((n, d)) for n in (s_q, s_k, s_k))
    nk = (s_k + 63) // 64
    vis = np.arange(s_k)[None, :] <= np.arange(s_q)[:, None] + off
    ref = _masked_sdpa(q, k, v, 0.25, vis)
    for i in range((s_q + 63) // 64):
        o, l = oatt.attention_unit(q, k, v, range(nk), i, 64, 64, 0.25, True, key_offset=off)
        rows = np.arange(i * 64, min((i + 1) * 64, s_q))
        live = vis[rows].any(axis=1)
        if live.any():
            assert np.abs(o[live] - ref[rows][live]).max() < 1e-12
        assert (o[~live] == 0).all() and np.isneginf(l[~live]).all()
        assert np.isfinite(l[live]).all()


def test_causal_key_offset_hand_example():
    """One dimension, scale 1: queries q = (1, 1), keys k = (0, 1, 2), values
    v = (10, 20, 30), key offset 1.  Query 0 sees keys 0 and 1: weights
    (1, e) / (1 + e), O = (10 + 20 e) / (1 + e), LSE = ln(1 + e).  Query 1
    sees all three: O = (10 + 20 e + 30 e^2) / (1 + e + e^2)."""
    q = np.array([[1.0], [1.0]])
    k = np.array([[0.0], [1.0], [2.0]])
    v = np.array([[10.0], [20.0], [30.0]])
    o, l = oatt.attention_unit(q, k, v, [0], 0, 64, 64, 1.0, True, key_offset=1)
    e = math.e
    assert o[0, 0] == pytest.approx((10 + 20 * e) / (1 + e), abs=1e-12)
    assert l[0] == pytest.approx(math.log(1 + e), abs=1e-12)
    assert o[1, 0] == pytest.approx((10 + 20 * e + 30 * e * e) / (1 + e + e * e), abs=1e-12)
    # offset 0: query 0 sees key 0 alone
    o, l = oatt.attention_unit(q, k, v, [0], 0, 64, 64, 1.0, True, key_offset=0)
    assert o[0, 0] == 10.0 and l[0] == 0.0


def _spec_case(seed=3, n_blocks=6, s_q=64, window=2, d=16):
    rng = np.random.default_rng(seed)
    s = n_blocks * 64
    q = rng.standard_normal((s_q, d))   # the last s_q positions of the sequence
    k, v = rng.standard_normal((s, d)), rng.standard_normal((s, d))
    w0 = (n_blocks - window) * 64        # the speculative window: keys w0 .. s-1
    return q, k, v, w0, s


def test_speculative_two_pass_equals_causal_attention():
    """Stage 5 of the Incremental_FlashAttention updating_log: a dense causal
    pass over the speculative window (the last blocks, holding the queries'
    own positions) plus a sparse pass over every missed historical block,
    combined, is causal attention over the whole sequence (sdpa with the
    causal mask of queries placed at the end)."""
    q, k, v, w0, s = _spec_case()
    missed = list(range(w0 // 64))
    o, l, _, _ = oatt.speculative_two_pass_unit(q, k[w0:], v[w0:], k, v, missed, 0, 64, 64, 0.25)
    vis = np.arange(s)[None, :] <= np.arange(q.shape[0])[:, None] + (s - q.shape[0])
    assert np.abs(o - _masked_sdpa(q, k, v, 0.25, vis)).max() < 1e-12
    # a sparse miss set: attention over the window plus the listed blocks only
    some = [0, 2]
    o, l, _, _ = oatt.speculative_two_pass_unit(q, k[w0:], v[w0:], k, v, some, 0, 64, 64, 0.25)
    keep = np.zeros(s, dtype=bool)
    keep[w0:] = True
    for j in some:
        keep[j * 64:(j + 1) * 64] = True
    assert np.abs(o - _masked_sdpa(q, k, v, 0.25, vis & keep[None, :])).max() < 1e-12
    # no missed block: pass 2 is the empty partial, the result is pass 1 alone
    o, l, p1, p2 = oatt.speculative_two_pass_unit(q, k[w0:], v[w0:], k, v, [], 0, 64, 64, 0.25)
    assert np.isneginf(p2[1]).all() and np.abs(o - p1[0]).max() == 0.0


@pytest.mark.parametrize("world", [2, 3, 5])
def test_causal_context_parallel_combines_to_causal_attention(world):
    """Causal context parallelism: rank r's keys start at position lo * 64, so
    its mask is key index u <= t - lo * 64; the ranks' partials combine to the
    causal attention of the whole LUT row (a causal LUT: blocks <= i, the
    diagonal included)."""
    rng = np.random.default_rng(world)
    s, d = 5 * 64 + 17, 16
    qh, kg, vg = (rng.standard_normal((s, d)) for _ in range(3))
    for i in range(6):
        row = sorted(set(rng.choice(i + 1, size=max(1, (i + 1) // 2), replace=False).tolist())
                     | {i})
        parts = oatt.context_parallel_unit(qh, kg, vg, row, i, world, 64, 64, 0.25, causal=True)
        o, l = oatt.combine(*parts)
        o_ref, l_ref = oatt.attention_unit(qh, kg, vg, row, i, 64, 64, 0.25, True)
        assert np.abs(o - o_ref).max() < 1e-12 and np.abs(l - l_ref).max() < 1e-12


def test_planted_key_offset_mistake_is_caught(monkeypatch):
    """A rank mask that adds lo * 64 instead of subtracting it (a flipped
    sign) breaks the causal context-parallel pin."""
    real = oatt.attention_unit

    def flipped(q, k, v, row, i, blkq, blkk, scale, causal, key_offset=0):
        return real(q, k, v, row, i, blkq, blkk, scale, causal, -key_offset)

    monkeypatch.setattr(oatt, "attention_unit", flipped)
    with pytest.raises(AssertionError):
        test_causal_context_parallel_combines_to_causal_attention(3)


def test_decode_rows_hand_example():
    rows = oatt.decode_rows(np.array([[3, 1]]), np.array([[0, 5, 7]]), 4)
    assert rows.tolist() == [[12, 5, 7]]


SMALL_DEC = synth.C5.replace(n_queries=4, pages_per_query=8, topk=96)


@pytest.mark.parametrize("S", [2, 3, 4, 5, 8])
def test_decode_split_invariance(S):
    cfg = SMALL_DEC
    inp = synth.decode(cfg)
    q = synth.bits_to_f64(inp["q"], "bf16")
    rows = oatt.decode_rows(inp["page_table"], inp["idx"], cfg.page)
    for c in range(cfg.n_queries):
        kv = synth.bits_to_f64(synth.cache_rows(cfg, rows[c]), "bf16")
        full = oatt.decode_attention(q[c], kv, cfg.dv, cfg.sm_scale)
        o, l = oracle.combine(*oatt.decode_partials(q[c], kv, cfg.dv, cfg.sm_scale, S))
        assert np.abs(o - full[0]).max() < 1e-10 and np.abs(l - full[1]).max() < 1e-10
        ref = _sdpa(q[c], kv, kv[:, :cfg.dv], cfg.sm_scale)
        assert np.abs(full[0] - ref).max() < 1e-12


# ----------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# ----------------------------------------------------------------------------


def _select_high_index_ties(score, topk, cdf, n_elig):
    sel = np.zeros(score.shape[0], dtype=bool)
    fin = np.nonzero(np.isfinite(score))[0]
    order = fin[np.lexsort((-fin, -score[fin]))]  # planted: higher index first
    kk = min(obm.topk_count(topk, n_elig), fin.size)
    sel[order[:kk]] = True
    return sel


def _select_cdf_exclusive(score, topk, cdf, n_elig):
    sel = np.zeros(score.shape[0], dtype=bool)
    fin = np.nonzero(np.isfinite(score))[0]
    p = _softmax(score)[fin]
    order = np.lexsort((fin, -p))
    cum = np.cumsum(p[order])
    take = int((cum < cdf).sum())  # planted: crossing entry left out
    sel[fin[order[:take]]] = True
    return sel


def test_planted_mistakes_are_caught():
    rows = _tiny_rows(1)
    with pytest.raises(AssertionError):
        for sc in rows:
            check_topk_bruteforce(_select_high_index_ties, sc, 0.5)
    with pytest.raises(AssertionError):
        for sc in rows:
            check_cdf_bruteforce(_select_cdf_exclusive, sc, 0.8)

    def bad_combine(o_parts, lse_parts):  # planted: weights not renormalised
        m = lse_parts.max(axis=0)
        w = np.exp(lse_parts - m)
        return (w[:, :, None] * o_parts).sum(axis=0), m + np.log(w.sum(axis=0))

    o1, o2 = np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]])
    o, _ = bad_combine(np.stack([o1, o2]), np.array([[math.log(3.0)], [0.0]]))
    assert np.abs(o[0] - [0.75, 0.25]).max() > 1e-3


def test_planted_smoothing_mistake_is_caught(monkeypatch):
    """Subtracting each block's own mean instead of the sequence mean turns
    every block of the hand example into zero rows (sim 0, all columns forced):
    the hand-example pin fails."""
    def block_mean_smoothing(kg, blk=2):  # planted: per-block instead of per-sequence mean
        out = kg.copy()
        for j in range(0, kg.shape[0], blk):
            out[j:j + blk] -= kg[j:j + blk].mean(axis=0)
        return out

    monkeypatch.setattr(obm, "smooth_keys", block_mean_smoothing)
    with pytest.raises(AssertionError):
        test_smooth_k_hand_example()
