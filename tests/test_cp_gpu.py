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
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, False, False,
                                dtype=cfg.dtype)
    return r["lut"], r["count"]


def run_cp(fbm, cfg, world, lut, cnt, units):
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
        cp.rank_partial(q, ks, vs, lut_d, cnt_d, lo, hi, scale=cfg.scale, o_slot=o_all[r],
                        lse_slot=l_all[r])
    out, lse = fbm.attn_combine(o_all, l_all, out_dtype=q.dtype)
    assert fbm.get_error() == 0
    o_parts, l_parts = o_all.double().cpu().numpy(), l_all.cpu().numpy().astype(np.float64)
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    ratio = cfg.hq // cfg.hk
    ref = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, cnt, cfg.scale, False, units=units,
                             dtype=cfg.dtype)
    empty_parts = 0
    for (bi, h, i), (o_ref, lse_ref) in ref.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        qh = synth.bits_to_f64(x["q"][bi, h], cfg.dtype)
        kg = synth.bits_to_f64(x["k"][bi, h // ratio], cfg.dtype)
        vg = synth.bits_to_f64(x["v"][bi, h // ratio], cfg.dtype)
        po, pl = oracle.context_parallel_unit(qh, kg, vg, lut[bi, h, i, :cnt[bi, h, i]], i,
                                              world, 64, 64, cfg.scale)
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
