"""Context-parallel sparse attention, its ranks run one after another on one
GPU (no rank waits on another): every rank shards the LUT to its kv-block
range (lut_shard, bit-exact against the oracle's shard rule), computes its
fp32 partial over its own K/V rows (sparse_fmha_fwd in partial mode), and
attn_combine merges the stacked partials.  Each rank's partial and the
combined result are compared with the oracle on the same seeded inputs: O
within atol 4e-2 / rtol 1e-2, LSE within 1e-3 nats, empty partials exactly
(0, -inf)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_close_lse, assert_close_o, cached_prefill, prefill_on_gpu

pytestmark = pytest.mark.gpu


def oracle_lut(cfg, mode, param):
    x = cached_prefill(cfg)
    ph = synth.per_head(cfg, param)
    r = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                ph if mode == "cdf" else None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype)
    return r["lut"], r["count"]


def run_cp(fbm, cfg, world, lut, cnt, units):
    causal = cfg.causal
    from fmha_block_map_gb300 import cp

    x, (q, k, v) = prefill_on_gpu(cfg)
    lut_d, cnt_d = torch.from_numpy(lut).cuda(), torch.from_numpy(cnt).cuda()
    b, hq, s, _ = q.shape
    dv = v.shape[3]
    bounds = cp.kv_shard_bounds(cfg.nq, world)
    assert bounds == oracle.split_bounds(cfg.nq, world)
    o_all = torch.empty((world, b, hq, s, dv), dtype=torch.float32, device="cuda")
    l_all = torch.empty((world, b, hq, s), dtype=torch.float32, device="cuda")
    for r, (lo, hi) in enumerate(bounds):
        # the shard of every LUT row, bit-exact
        sub_lut, sub_cnt = fbm.lut_shard(lut_d, cnt_d, lo, hi)
        sub_lut, sub_cnt = sub_lut.cpu().numpy(), sub_cnt.cpu().numpy()
        for idx in np.ndindex(*cnt.shape):
            want = oracle.shard_lut_row(lut[idx][:cnt[idx]], lo, hi)
            assert sub_cnt[idx] == len(want), (r, idx)
            assert sub_lut[idx][:len(want)].tolist() == want, (r, idx)
            assert (sub_lut[idx][len(want):] == -1).all(), (r, idx)
        r0, r1 = cp.shard_rows(s, lo, hi)
        ks, vs = k[:, :, r0:r1].contiguous(), v[:, :, r0:r1].contiguous()
        cp.rank_partial(q, ks, vs, lut_d, cnt_d, lo, hi, scale=cfg.scale, causal=causal,
                        o_slot=o_all[r], lse_slot=l_all[r])
    out, lse = fbm.attn_combine(o_all, l_all, out_dtype=q.dtype)
    assert fbm.get_error() == 0
    o_parts, l_parts = o_all.double().cpu().numpy(), l_all.cpu().numpy().astype(np.float64)
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    ratio = cfg.hq // cfg.hk
    ref = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, cnt, cfg.scale, causal, units=units,
                             dtype=cfg.dtype)
    empty_parts = 0
    for (bi, h, i), (o_ref, lse_ref) in ref.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        qh = synth.bits_to_f64(x["q"][bi, h], cfg.dtype)
        kg = synth.bits_to_f64(x["k"][bi, h // ratio], cfg.dtype)
        vg = synth.bits_to_f64(x["v"][bi, h // ratio], cfg.dtype)
        po, pl = oracle.context_parallel_unit(qh, kg, vg, lut[bi, h, i, :cnt[bi, h, i]], i,
                                              world, 64, 64, cfg.scale, causal=causal)
        for r in range(world):
            assert_close_o(o_parts[r, bi, h, rows], po[r], f"partial O r{r} {(bi, h, i)}")
            assert_close_lse(l_parts[r, bi, h, rows], pl[r], f"partial LSE r{r} {(bi, h, i)}")
            if np.isneginf(pl[r]).all():
                empty_parts += 1
                assert (o_parts[r, bi, h, rows] == 0).all()
        assert_close_o(o_np[bi, h, rows], o_ref, f"O {(bi, h, i)}")
        assert_close_lse(l_np[bi, h, rows], lse_ref, f"LSE {(bi, h, i)}")
    print(f"{cfg.name} world={world}: {len(ref)} q blocks, {empty_parts} empty partials")
    return empty_parts


@pytest.mark.parametrize("world", [2, 3])
def test_cp_c2_cdf(fbm_gpu, world):
    cfg = synth.C2
    lut, cnt = oracle_lut(cfg, "cdf", 0.9)
    units = [(0, h, i) for h in (0, 5) for i in (0, 17, 63)]
    run_cp(fbm_gpu, cfg, world, lut, cnt, units)


def test_cp_ragged_gqa_d64(fbm_gpu):
    # s = 1000: 16 kv blocks over 3 ranks (6, 5, 5), the last block 40 rows
    cfg = synth.C2.replace(b=2, hq=4, hk=2, s=1000, d=64, cs_range=None, dtype="f16")
    lut, cnt = oracle_lut(cfg, "topk", 0.5)
    units = [(b, h, i) for b in range(2) for h in range(4) for i in (0, 7, 15)]
    run_cp(fbm_gpu, cfg, 3, lut, cnt, units)


def test_cp_hand_lut_with_empty_shards(fbm_gpu):
    cfg = synth.C1.replace(hq=2, hk=2)       # s = 512: 8 kv blocks
    nq = cfg.nq
    lut = np.full((1, 2, nq, nq), -1, dtype=np.int32)
    cnt = np.zeros((1, 2, nq), dtype=np.int32)
    rows = {0: [], 1: [0], 2: [0, 1, 2], 3: [5, 7], 4: list(range(8)), 5: [3], 6: [1, 6], 7: [7]}
    for h in range(2):
        for i, row in rows.items():
            lut[0, h, i, :len(row)] = row
            cnt[0, h, i] = len(row)
    units = [(0, h, i) for h in range(2) for i in range(nq)]
    assert run_cp(fbm_gpu, cfg, 4, lut, cnt, units) > 0


@pytest.mark.parametrize("world", [2, 4])
def test_cp_causal_gqa_sink(fbm_gpu, world):
    """Causal context parallelism: each rank's partial runs with the causal key
    offset -lo * 64 of its kv range; the combine equals causal attention over
    the block map's causal LUT (GQA, sink, ragged s = 1000)."""
    cfg = synth.C4.replace(s=1000, hq=4, hk=2)
    lut, cnt = oracle_lut(cfg, "topk", 0.3)
    units = [(0, h, i) for h in range(4) for i in (0, 3, 8, 15)]
    run_cp(fbm_gpu, cfg, world, lut, cnt, units)


# ---- causal key offset and the speculative two-pass recipe


@pytest.mark.parametrize("s_q,s_k,off,dense", [(192, 448, 256, True), (200, 200, -96, True),
                                               (256, 640, 384, False), (128, 128, 40, False)])
def test_causal_key_offset(fbm_gpu, s_q, s_k, off, dense):
    """sparse_fmha_fwd with causal and a key offset (key u visible to query t
    when u <= t + off) against the oracle, dense mode and a hand LUT; rows
    with no visible key are empty (0, -inf)."""
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=max(s_q, s_k), d=128, dtype="bf16")
    x, (q, k, v) = prefill_on_gpu(cfg)
    q, xq = q[:, :, :s_q].contiguous(), x["q"][:, :, :s_q]
    k, v, xk, xv = (k[:, :, :s_k].contiguous(), v[:, :, :s_k].contiguous(), x["k"][:, :, :s_k],
                    x["v"][:, :, :s_k])
    nq, nk = (s_q + 63) // 64, (s_k + 63) // 64
    rng = np.random.default_rng(s_q + off)
    lut = np.full((1, 2, nq, nk), -1, dtype=np.int32)
    cnt = np.zeros((1, 2, nq), dtype=np.int32)
    for h in range(2):
        for i in range(nq):
            if dense:
                last = i * 64 + 63 + off
                row = list(range(0 if last < 0 else min(nk, last // 64 + 1)))
            else:
                row = sorted(rng.choice(nk, size=max(1, nk // 2), replace=False).tolist())
            lut[0, h, i, :len(row)] = row
            cnt[0, h, i] = len(row)
    args = (None, None) if dense else (torch.from_numpy(lut).cuda(), torch.from_numpy(cnt).cuda())
    out, lse = fbm_gpu.sparse_fmha_fwd(q, k, v, *args, scale=cfg.scale, causal=True, key_offset=off,
                                       return_lse=True)
    assert fbm_gpu.get_error() == 0
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    res = oracle.sparse_fmha(xq, xk, xv, lut, cnt, cfg.scale, True, dtype="bf16", key_offset=off)
    empty = 0
    for (b, h, i), (o_ref, l_ref) in res.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        assert_close_o(o_np[b, h, rows], o_ref, f"O {(b, h, i)}")
        assert_close_lse(l_np[b, h, rows], l_ref, f"LSE {(b, h, i)}")
        empty += int(np.isneginf(l_ref).sum())
    if off < 0:
        assert empty > 0    # the first rows see no key


@pytest.mark.parametrize("missed", ["all", "sparse", "none"])
def test_speculative_two_pass(fbm_gpu, missed):
    """Stage 5 of the Incremental_FlashAttention updating_log on the GPU: a
    dense causal pass over the speculative window (the last two blocks of the
    sequence, which hold the queries' own positions), a sparse pass over the
    missed historical blocks, and the combine (cp.speculative_two_pass),
    against the oracle's two-pass unit; with every historical block missed the
    result is causal attention over the whole sequence."""
    from fmha_block_map_gb300 import cp

    n_blocks, s_q = 8, 64
    cfg = synth.C4.replace(s=n_blocks * 64, hq=4, hk=2)
    x, (q_all, k, v) = prefill_on_gpu(cfg)
    s = cfg.s
    q = q_all[:, :, s - s_q:].contiguous()          # the queries: the last 64 positions
    w0 = s - 2 * 64
    k_spec, v_spec = k[:, :, w0:].contiguous(), v[:, :, w0:].contiguous()
    hist = list(range(w0 // 64))
    rows = {"all": hist, "sparse": hist[::2], "none": []}[missed]
    lut = np.full((1, 4, 1, n_blocks), -1, dtype=np.int32)
    cnt = np.full((1, 4, 1), len(rows), dtype=np.int32)
    lut[..., :len(rows)] = rows
    out, lse = cp.speculative_two_pass(q, k_spec, v_spec, k, v, torch.from_numpy(lut).cuda(),
                                       torch.from_numpy(cnt).cuda(), scale=cfg.scale)
    assert fbm_gpu.get_error() == 0
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    for h in range(4):
        qh = synth.bits_to_f64(x["q"][0, h, s - s_q:], "bf16")
        kg = synth.bits_to_f64(x["k"][0, h // 2], "bf16")
        vg = synth.bits_to_f64(x["v"][0, h // 2], "bf16")
        o_ref, l_ref, _, _ = oracle.speculative_two_pass_unit(qh, kg[w0:], vg[w0:], kg, vg, rows,
                                                              0, 64, 64, cfg.scale)
        assert_close_o(o_np[0, h], o_ref, f"O h{h}")
        assert_close_lse(l_np[0, h], l_ref, f"LSE h{h}")
        if missed == "all":   # equals causal attention over the whole sequence
            o_full, l_full = oracle.attention_unit(qh, kg, vg, range(n_blocks), 0, 64, 64,
                                                   cfg.scale, True, key_offset=s - s_q)
            assert np.abs(o_ref - o_full).max() < 1e-12
