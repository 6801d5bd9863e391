"""The 128-row (q-block pair) attention path: lut_pair_union builds, per pair
of adjacent q blocks, the ascending union of their LUT rows with membership
flags (checked exactly against a plain host merge), and sparse_fmha_fwd_pairs
must give the oracle's attention over each q block's OWN LUT row: O within
atol 4e-2 / rtol 1e-2, LSE within 1e-3 nats, empty rows exactly (0, -inf)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_close_lse, assert_close_o, cached_prefill, prefill_on_gpu

pytestmark = pytest.mark.gpu


def host_union(lut, cnt, nk):
    """The pair-union rows by a plain host merge (bit 29: row 2p, bit 30: row 2p + 1)."""
    *lead, nq, _ = lut.shape
    npq = (nq + 1) // 2
    out = np.full(tuple(lead) + (npq, nk), -1, dtype=np.int64)
    ocnt = np.zeros(tuple(lead) + (npq,), dtype=np.int64)
    for idx in np.ndindex(*lead):
        for p in range(npq):
            a = set(int(j) for j in lut[idx][2 * p][:cnt[idx][2 * p]])
            b = set(int(j) for j in lut[idx][2 * p + 1][:cnt[idx][2 * p + 1]]) \
                if 2 * p + 1 < nq else set()
            u = sorted(a | b)
            out[idx][p][:len(u)] = [j | ((j in a) << 29) | ((j in b) << 30) for j in u]
            ocnt[idx][p] = len(u)
    return out, ocnt


def run_pairs(fbm, cfg, lut, cnt, units=None, dense=False, key_offset=0):
    x, (q, k, v) = prefill_on_gpu(cfg)
    nk = (k.shape[2] + 63) // 64
    if dense:
        pl = pc = None
    else:
        lut_d, cnt_d = torch.from_numpy(lut).cuda(), torch.from_numpy(cnt).cuda()
        pl, pc = fbm.lut_pair_union(lut_d, cnt_d, nk)
        want_l, want_c = host_union(lut, cnt, nk)
        assert (pc.cpu().numpy() == want_c).all()
        assert (pl.cpu().numpy().astype(np.int64) == want_l).all()
    out, lse = fbm.sparse_fmha_fwd_pairs(q, k, v, pl, pc, scale=cfg.scale, causal=cfg.causal,
                                         key_offset=key_offset, return_lse=True)
    assert fbm.get_error() == 0
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, cnt, cfg.scale, cfg.causal,
                             units=units, dtype=cfg.dtype, key_offset=key_offset)
    for (b, h, i), (o_ref, lse_ref) in res.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        assert_close_o(o_np[b, h, rows], o_ref, f"O{(b, h, i)}")
        assert_close_lse(l_np[b, h, rows], lse_ref, f"LSE{(b, h, i)}")
        if not dense and cnt[b, h, i] == 0:
            assert (o_np[b, h, rows] == 0).all() and np.isneginf(l_np[b, h, rows]).all()
    return out, lse


def hand_lut(cfg, seed=0):
    """Per pair of q blocks: disjoint rows, equal rows, one empty, both empty,
    nested rows, random rows."""
    nq = cfg.nq
    nk = nq
    rng = np.random.default_rng(seed)
    lut = np.full((cfg.b, cfg.hq, nq, nk), -1, dtype=np.int32)
    cnt = np.zeros((cfg.b, cfg.hq, nq), dtype=np.int32)
    for b in range(cfg.b):
        for h in range(cfg.hq):
            for i in range(nq):
                hi = i + 1 if cfg.causal else nk
                kind = (b * 5 + h * 3 + i // 2) % 6
                if kind == 0:
                    row = [j for j in range(hi) if j % 2 == i % 2]
                elif kind == 1:
                    row = list(range(0, hi, 3))
                elif kind == 2:
                    row = [] if i % 2 else sorted({0, hi - 1})
                elif kind == 3:
                    row = []
                elif kind == 4:
                    row = list(range(hi)) if i % 2 else list(range(0, hi, 2))
                else:
                    row = sorted(rng.choice(hi, size=max(1, hi // 3), replace=False).tolist())
                lut[b, h, i, :len(row)] = row
                cnt[b, h, i] = len(row)
    return lut, cnt


@pytest.mark.parametrize("hk", [4, 1])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_pairs_hand_luts_gqa(fbm_gpu, hk, dtype, d):
    cfg = synth.C1.replace(b=2, hq=4, hk=hk, s=640, d=d, dtype=dtype)
    lut, cnt = hand_lut(cfg)
    run_pairs(fbm_gpu, cfg, lut, cnt)


@pytest.mark.parametrize("causal", [False, True])
def test_pairs_ragged_odd_block_count(fbm_gpu, causal):
    # s = 1000: 16 q blocks, the last one 40 rows; s = 900: 15 q blocks, so
    # the last pair has a single q block
    for s in (1000, 900):
        cfg = synth.C1.replace(b=1, hq=2, hk=1, s=s, d=128, dtype="bf16", causal=causal)
        lut, cnt = hand_lut(cfg, seed=s)
        run_pairs(fbm_gpu, cfg, lut, cnt)


@pytest.mark.parametrize("causal", [False, True])
def test_pairs_dense_mode(fbm_gpu, causal):
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=704, d=128, dtype="f16", causal=causal)
    nq = cfg.nq
    lut = np.full((1, 2, nq, nq), -1, dtype=np.int32)
    cnt = np.zeros((1, 2, nq), dtype=np.int32)
    for i in range(nq):
        n = i + 1 if causal else nq
        lut[:, :, i, :n] = np.arange(n)
        cnt[:, :, i] = n
    o_dense, l_dense = run_pairs(fbm_gpu, cfg, lut, cnt, dense=True)
    o_full, l_full = run_pairs(fbm_gpu, cfg, lut, cnt)
    if not causal:  # the same visit order: bit-identical
        assert torch.equal(o_dense, o_full) and torch.equal(l_dense, l_full)


@pytest.mark.parametrize("off", [-96, 200])
def test_pairs_causal_key_offset(fbm_gpu, off):
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=640, d=128, dtype="bf16", causal=True)
    nq = cfg.nq
    lut = np.full((1, 2, nq, nq), -1, dtype=np.int32)
    cnt = np.zeros((1, 2, nq), dtype=np.int32)
    for i in range(nq):
        last = i * 64 + 63 + off
        n = 0 if last < 0 else min(nq, last // 64 + 1)
        lut[:, :, i, :n] = np.arange(n)
        cnt[:, :, i] = n
    run_pairs(fbm_gpu, cfg, lut, cnt, key_offset=off)
    run_pairs(fbm_gpu, cfg, lut, cnt, key_offset=off, dense=True)


def _oracle_lut(cfg, mode, param, heads=None):
    x = cached_prefill(cfg)
    ph = synth.per_head(cfg, param)
    r = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                ph if mode == "cdf" else None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype, heads=heads)
    return r["lut"], r["count"]


def test_pairs_c1_and_c2(fbm_gpu):
    lut, cnt = _oracle_lut(synth.C1, "topk", 0.5)
    run_pairs(fbm_gpu, synth.C1, lut, cnt)
    lut, cnt = _oracle_lut(synth.C2, "cdf", 0.9)
    run_pairs(fbm_gpu, synth.C2, lut, cnt)


@pytest.mark.parametrize("topk", [0.4, 1.0])
def test_pairs_c3_sampled(fbm_gpu, topk):
    cfg = synth.C3
    heads = [(0, 0), (1, 24)]
    lut, cnt = _oracle_lut(cfg, "topk", topk, heads=heads)
    units = [u for u in synth.sample_qblocks(cfg, 8) if (u[0], u[1]) in heads]
    run_pairs(fbm_gpu, cfg, lut, cnt, units=units)


def test_pairs_c4_causal_gqa_sampled(fbm_gpu):
    cfg = synth.C4
    heads = [(0, 0), (0, 29)]
    lut, cnt = _oracle_lut(cfg, "topk", 0.2, heads=heads)
    units = [u for u in synth.sample_qblocks(cfg, 6) if (u[0], u[1]) in heads]
    run_pairs(fbm_gpu, cfg, lut, cnt, units=units)


def test_pair_union_flags_range_errors(fbm_gpu):
    lut = torch.tensor([[[0, 5, 99, -1], [2, 5, -3, -1]]], dtype=torch.int32).cuda()
    cnt = torch.tensor([[3, 3]], dtype=torch.int32).cuda()
    pl, pc = fbm_gpu.lut_pair_union(lut, cnt, 8)
    assert fbm_gpu.get_error() == fbm_gpu.FBM_DEVERR_LUT_RANGE
    assert pc.cpu().tolist() == [[3]]
    assert pl.cpu().tolist()[0][0][:3] == [0 | 1 << 29, 2 | 1 << 30, 5 | 3 << 29]
