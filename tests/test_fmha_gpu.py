"""GPU sparse FMHA (sparse_fmha_fwd, attn_combine) against the fp64 oracle on
the same seeded inputs and the oracle's own LUTs: O within atol 4e-2 / rtol
1e-2, LSE within 1e-3 nats, empty rows exactly (0, -inf)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import (assert_close_lse, assert_close_o, cached_prefill, compare_lut_rows,
                   prefill_on_gpu, to_dev)

pytestmark = pytest.mark.gpu


def oracle_lut(cfg, mode="topk", param=None, heads=None, keep_aux=False):
    x = cached_prefill(cfg)
    param = cfg.topk if param is None else param
    ph = synth.per_head(cfg, param)
    r = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                ph if mode == "cdf" else None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype, heads=heads,
                                keep_aux=keep_aux)
    if keep_aux:
        return r["lut"], r["count"], r["aux"]
    return r["lut"], r["count"]


def check(fbm, cfg, lut, cnt, units=None, num_splits=1, dense=False):
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut_d = None if dense else torch.from_numpy(lut).cuda()
    cnt_d = None if dense else torch.from_numpy(cnt).cuda()
    if num_splits == 1:
        out, lse = fbm.sparse_fmha_fwd(q, k, v, lut_d, cnt_d, scale=cfg.scale, causal=cfg.causal,
                                       return_lse=True)
    else:
        op, lp = fbm.sparse_fmha_fwd(q, k, v, lut_d, cnt_d, scale=cfg.scale, causal=cfg.causal,
                                     num_splits=num_splits)
        out, lse = fbm.attn_combine(op, lp, out_dtype=q.dtype)
    assert fbm.get_error() == 0
    o_np = out.double().cpu().numpy()
    l_np = lse.cpu().numpy().astype(np.float64)
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, cnt, cfg.scale, cfg.causal, units=units,
                             dtype=cfg.dtype)
    worst_o = worst_l = 0.0
    for (b, h, i), (o_ref, lse_ref) in res.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        worst_o = max(worst_o, assert_close_o(o_np[b, h, rows], o_ref, f"O{(b, h, i)}"))
        worst_l = max(worst_l, assert_close_lse(l_np[b, h, rows], lse_ref, f"LSE{(b, h, i)}"))
        if (cnt[b, h, i] == 0) if not dense else False:
            assert (o_np[b, h, rows] == 0).all() and np.isneginf(l_np[b, h, rows]).all()
    print(f"{cfg.name}: {len(res)} q blocks, max |dO| {worst_o:.2e}, max |dLSE| {worst_l:.2e}")
    return out, lse


def hand_lut(cfg, seed=0):
    """Empty, single, discontinuous, full and random rows."""
    nq = cfg.nq
    nk = nq
    rng = np.random.default_rng(seed)
    lut = np.full((cfg.b, cfg.hq, nq, nk), -1, dtype=np.int32)
    cnt = np.zeros((cfg.b, cfg.hq, nq), dtype=np.int32)
    for b in range(cfg.b):
        for h in range(cfg.hq):
            for i in range(nq):
                hi = i + 1 if cfg.causal else nk
                kind = (b * 7 + h * 3 + i) % 5
                if kind == 0:
                    row = []
                elif kind == 1:
                    row = [int(rng.integers(0, hi))]
                elif kind == 2:
                    row = sorted({0, hi - 1, (hi - 1) // 2})
                elif kind == 3:
                    row = list(range(hi))
                else:
                    row = sorted(rng.choice(hi, size=max(1, hi // 3), replace=False).tolist())
                lut[b, h, i, :len(row)] = row
                cnt[b, h, i] = len(row)
    return lut, cnt


def test_c1_oracle_lut(fbm_gpu):
    lut, cnt = oracle_lut(synth.C1)
    check(fbm_gpu, synth.C1, lut, cnt)


@pytest.mark.parametrize("hk", [4, 2, 1])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_hand_luts_gqa(fbm_gpu, hk, dtype, d):
    cfg = synth.C1.replace(b=2, hq=4, hk=hk, s=640, d=d, dtype=dtype)
    lut, cnt = hand_lut(cfg)
    check(fbm_gpu, cfg, lut, cnt)


@pytest.mark.parametrize("causal", [False, True])
def test_hand_luts_causal_and_ragged(fbm_gpu, causal):
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=1000, d=128, dtype="bf16", causal=causal)
    lut, cnt = hand_lut(cfg, seed=3)
    check(fbm_gpu, cfg, lut, cnt)


@pytest.mark.parametrize("causal", [False, True])
def test_dense_mode_matches_full_lut(fbm_gpu, causal):
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=768, d=128, dtype="f16", causal=causal)
    nq = cfg.nq
    lut = np.full((1, 2, nq, nq), -1, dtype=np.int32)
    cnt = np.zeros((1, 2, nq), dtype=np.int32)
    for i in range(nq):
        n = i + 1 if causal else nq
        lut[:, :, i, :n] = np.arange(n)
        cnt[:, :, i] = n
    o_dense, l_dense = check(fbm_gpu, cfg, lut, cnt, dense=True)
    o_full, l_full = check(fbm_gpu, cfg, lut, cnt)
    # same kernel, same visit order: bit-identical
    assert torch.equal(o_dense, o_full) and torch.equal(l_dense, l_full)


@pytest.mark.parametrize("S,d", [(2, 128), (3, 128), (5, 128), (3, 64)])
def test_split_kv_partials_and_combine(fbm_gpu, S, d):
    cfg = synth.C1.replace(b=1, hq=4, hk=2, s=640, d=d, dtype="bf16")
    lut, cnt = hand_lut(cfg, seed=S)
    x, (q, k, v) = prefill_on_gpu(cfg)
    op, lp = fbm_gpu.sparse_fmha_fwd(q, k, v, torch.from_numpy(lut).cuda(),
                                     torch.from_numpy(cnt).cuda(), scale=cfg.scale, num_splits=S)
    op, lp = op.double().cpu().numpy(), lp.double().cpu().numpy()
    qf, kf, vf = (synth.bits_to_f64(x[t], "bf16") for t in ("q", "k", "v"))
    for h in range(cfg.hq):
        for i in range(cfg.nq):
            row = lut[0, h, i, :cnt[0, h, i]]
            parts = oracle.split_partials_unit(qf[0, h], kf[0, h // 2], vf[0, h // 2], row, i, S,
                                               64, 64, cfg.scale, False)
            for s in range(S):
                assert_close_o(op[s, 0, h, i * 64:(i + 1) * 64], parts[0][s], f"Opart{s}")
                assert_close_lse(lp[s, 0, h, i * 64:(i + 1) * 64], parts[1][s], f"LSEpart{s}")
    check(fbm_gpu, cfg, lut, cnt, num_splits=S)


@pytest.mark.parametrize("S", [2, 4])
def test_split_kv_dense_causal_ragged(fbm_gpu, S):
    # dense list (every causally visible block) cut into chunks; s = 1000
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=1000, d=128, dtype="f16", causal=True)
    nq = cfg.nq
    lut = np.tile(np.arange(nq, dtype=np.int32), (1, 2, nq, 1))
    cnt = np.tile(np.arange(1, nq + 1, dtype=np.int32), (1, 2, 1))
    check(fbm_gpu, cfg, lut, cnt, num_splits=S, dense=True)


def test_c2_cdf_attention(fbm_gpu):
    lut, cnt = oracle_lut(synth.C2, "cdf", 0.9)
    check(fbm_gpu, synth.C2, lut, cnt)


@pytest.mark.parametrize("topk", synth.C3_TOPKS)
def test_c3_sampled(fbm_gpu, topk):
    # every point of the headline topk sweep: 8 sampled q blocks (the first
    # and last always) of every 8th head, at full size
    cfg = synth.C3
    heads = [(b, h) for b in range(cfg.b) for h in range(0, cfg.hq, 8)]
    lut, cnt = oracle_lut(cfg, "topk", topk, heads=heads)
    units = [u for u in synth.sample_qblocks(cfg, 8) if u[1] % 8 == 0]
    check(fbm_gpu, cfg, lut, cnt, units=units)


def test_headline_step_gpu_lut_into_gpu_fmha(fbm_gpu):
    """The step the bench times, chained on the GPU: sparge_block_map's LUT
    fed straight to sparse_fmha_fwd at b2 h32 s16384 d128 fp16, topk 0.4.
    The GPU LUT of sampled heads must equal the oracle's up to counted
    near-ties; the oracle's attention then runs on the GPU's LUT (so a
    near-tie row is checked against the blocks the GPU actually chose)."""
    cfg = synth.C3
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut, cnt, _ = fbm_gpu.sparge_block_map(q, k, topk=0.4, simthreshd1=cfg.simthreshd1,
                                           scale=cfg.scale)
    out, lse = fbm_gpu.sparse_fmha_fwd(q, k, v, lut, cnt, scale=cfg.scale, return_lse=True)
    assert fbm_gpu.get_error() == 0
    g_lut, g_cnt = lut.cpu().numpy(), cnt.cpu().numpy()
    heads = [(0, 0), (0, 13), (1, 22), (1, 31)]
    o_lut, o_cnt, aux = oracle_lut(cfg, "topk", 0.4, heads=heads, keep_aux=True)
    near = 0
    for b, h in heads:
        near += compare_lut_rows(g_lut[b, h], g_cnt[b, h], o_lut[b, h], o_cnt[b, h], aux[(b, h)],
                                 "topk", 0.4, False, False)[1]
    units = [u for u in synth.sample_qblocks(cfg, 8) if (u[0], u[1]) in heads]
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], g_lut, g_cnt, cfg.scale, False, units=units,
                             dtype=cfg.dtype)
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    for (b, h, i), (o_ref, lse_ref) in res.items():
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        assert_close_o(o_np[b, h, rows], o_ref, f"O{(b, h, i)}")
        assert_close_lse(l_np[b, h, rows], lse_ref, f"LSE{(b, h, i)}")
    print(f"headline step: {len(res)} q blocks checked, {near} near-tie LUT rows")


def test_c4_sampled_with_lse(fbm_gpu):
    cfg = synth.C4
    lut, cnt = oracle_lut(cfg)
    units = [u for u in synth.sample_qblocks(cfg, 6) if u[1] % 5 == 0]
    check(fbm_gpu, cfg, lut, cnt, units=units)


def test_relaunch_is_bitwise_deterministic(fbm_gpu):
    cfg = synth.C1.replace(b=1, hq=4, hk=2, s=1024, d=128, dtype="bf16")
    lut, cnt = hand_lut(cfg, seed=9)
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut_d, cnt_d = torch.from_numpy(lut).cuda(), torch.from_numpy(cnt).cuda()
    ref = None
    for _ in range(50):
        o, l = fbm_gpu.sparse_fmha_fwd(q, k, v, lut_d, cnt_d, scale=cfg.scale, return_lse=True)
        if ref is None:
            ref = (o.clone(), l.clone())
        assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])


def test_out_of_range_entry_is_skipped_and_flagged(fbm_gpu):
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=512, d=128, dtype="f16")
    nq = cfg.nq
    lut = np.full((1, 2, nq, nq), -1, dtype=np.int32)
    cnt = np.full((1, 2, nq), 2, dtype=np.int32)
    lut[..., 0] = 1
    lut[..., 1] = nq + 5  # out of range: skipped, error bit set
    x, (q, k, v) = prefill_on_gpu(cfg)
    out, lse = fbm_gpu.sparse_fmha_fwd(q, k, v, torch.from_numpy(lut).cuda(),
                                       torch.from_numpy(cnt).cuda(), scale=cfg.scale,
                                       return_lse=True)
    assert fbm_gpu.get_error() == fbm_gpu.FBM_DEVERR_LUT_RANGE
    assert fbm_gpu.get_error() == 0  # read clears
    good = lut.copy()
    good[..., 1] = -1
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], good, np.ones_like(cnt), cfg.scale, False,
                             dtype="f16")
    o_np = out.double().cpu().numpy()
    for (b, h, i), (o_ref, _) in res.items():
        assert_close_o(o_np[b, h, i * 64:(i + 1) * 64], o_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_count_out_of_range_is_clamped_and_flagged(fbm_gpu, d):
    """A count above min(nk, stride) is clamped to it and a negative count
    gives an empty row, each with FBM_DEVERR_LUT_RANGE; the result equals the
    oracle over the clamped rows."""
    cfg = synth.C1.replace(b=1, hq=4, hk=2, s=512, d=d, dtype="f16")
    nq = cfg.nq
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut = np.tile(np.arange(nq, dtype=np.int32), (1, 4, nq, 1))
    cnt = np.full((1, 4, nq), nq, dtype=np.int32)
    cnt[0, 1] = nq + 5
    cnt[0, 2] = -3
    out, lse = fbm_gpu.sparse_fmha_fwd(q, k, v, torch.from_numpy(lut).cuda(),
                                       torch.from_numpy(cnt).cuda(), scale=cfg.scale,
                                       return_lse=True)
    assert fbm_gpu.get_error() == fbm_gpu.FBM_DEVERR_LUT_RANGE
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    good = cnt.copy()
    good[0, 1] = nq
    good[0, 2] = 0
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, good, cfg.scale, False, dtype="f16")
    for (b, h, i), (o_ref, l_ref) in res.items():
        assert_close_o(o_np[b, h, i * 64:(i + 1) * 64], o_ref)
        assert_close_lse(l_np[b, h, i * 64:(i + 1) * 64], l_ref)
    assert (o_np[0, 2] == 0).all() and np.isneginf(l_np[0, 2]).all()
    assert fbm_gpu.get_error() == 0


def test_lut_validate_finds_order_range_and_count_errors(fbm_gpu):
    """lut_validate checks the sparse block table contract without changing
    the LUT: duplicates and descending entries set FBM_DEVERR_LUT_ORDER,
    entries outside [0, nk) and counts outside [0, min(nk, stride)] set
    FBM_DEVERR_LUT_RANGE; the block map's own LUT at the headline shape is
    valid."""
    nk = 12
    R, O = fbm_gpu.FBM_DEVERR_LUT_RANGE, fbm_gpu.FBM_DEVERR_LUT_ORDER
    cases = [  # (row, count, expected bits)
        ([0, 3, 7, 11], 4, 0), ([], 0, 0), (list(range(nk)), nk, 0),
        ([1, 1, 3], 3, O), ([5, 2], 2, O), ([0, 4, 4, 9], 4, O),
        ([0, nk], 2, R), ([-1, 2], 2, R), (list(range(nk)), nk + 1, R), ([0, 1], -2, R),
        ([3, 2, nk + 4], 3, R | O),
        # a long row whose only fault (index 32 not above index 31) straddles
        # the 32-entry chunk boundary
        (list(range(32)) + [31, 40], 34, O),
    ]
    for row, count, want in cases:
        stride = max(nk, len(row), 40)
        lut = torch.full((2, stride), -1, dtype=torch.int32)
        lut[1, :len(row)] = torch.tensor(row, dtype=torch.int32)
        lut[0, :3] = torch.tensor([0, 1, 2], dtype=torch.int32)
        cnt = torch.tensor([3, count], dtype=torch.int32)
        lut_d, cnt_d = lut.cuda(), cnt.cuda()
        nk_case = 41 if len(row) > nk + 2 else nk
        bits = fbm_gpu.lut_validate(lut_d, cnt_d, nk_case)
        assert bits == want, (row, count, bits)
        assert torch.equal(lut_d.cpu(), lut) and torch.equal(cnt_d.cpu(), cnt)
    cfg = synth.C3
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut, cnt, _ = fbm_gpu.sparge_block_map(q, k, topk=0.4, scale=cfg.scale)
    assert fbm_gpu.lut_validate(lut, cnt, cfg.nq) == 0


def test_every_shape_runs_on_the_tcgen05_kernel(fbm_gpu):
    """Every supported shape runs the tcgen05 kernel (d = 64 and 128)."""
    for dt in (torch.float16, torch.bfloat16):
        assert fbm_gpu.fmha_kernel_kind(dt, 128, 128, 1, 16384, 16384) == 1
        assert fbm_gpu.fmha_kernel_kind(dt, 128, 128, 1, 1000, 1000) == 1
    assert fbm_gpu.fmha_kernel_kind(torch.float16, 64, 64, 1, 512, 512) == 1
    assert fbm_gpu.fmha_kernel_kind(torch.float16, 128, 128, 4, 512, 512) == 1


# ---- per-Q-tile PV skip (pv_threshold) on the tcgen05 kernel

def _pv_case(fbm, cfg, tau, lut, cnt):
    x, (q, k, v) = prefill_on_gpu(cfg)
    out, lse = fbm.sparse_fmha_fwd(q, k, v, torch.from_numpy(lut).cuda(),
                                   torch.from_numpy(cnt).cuda(), scale=cfg.scale,
                                   causal=cfg.causal, return_lse=True, pv_threshold=tau)
    assert fbm.get_error() == 0
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    ratio = cfg.hq // cfg.hk
    skipped = changed = 0
    for b in range(cfg.b):
        for h in range(cfg.hq):
            qh = synth.bits_to_f64(x["q"][b, h], cfg.dtype)
            kg = synth.bits_to_f64(x["k"][b, h // ratio], cfg.dtype)
            vg = synth.bits_to_f64(x["v"][b, h // ratio], cfg.dtype)
            for i in range(cfg.nq):
                row = lut[b, h, i, :cnt[b, h, i]]
                mg = []
                o_ref, l_ref, sk = oracle.attention_unit_pv_skip(qh, kg, vg, row, i, 64, 64,
                                                                 cfg.scale, cfg.causal, tau,
                                                                 margins=mg)
                fin = [abs(z) for z in mg if math.isfinite(z)]
                # every skip decision is far from its boundary in fp64 (checked)
                assert not fin or min(fin) > 1e-3, f"decision margin {min(fin)} at {(b, h, i)}"
                rows = slice(i * 64, i * 64 + o_ref.shape[0])
                assert_close_o(o_np[b, h, rows], o_ref, f"O {(b, h, i)} tau={tau}")
                assert_close_lse(l_np[b, h, rows], l_ref, f"LSE {(b, h, i)}")
                full = oracle.attention_unit(qh, kg, vg, row, i, 64, 64, cfg.scale, cfg.causal)[0]
                skipped += len(sk)
                changed += int(np.abs(full - o_ref).max() > 4e-2)
    print(f"{cfg.name} tau={tau}: {skipped} blocks skipped, {changed} q blocks visibly changed")
    return skipped, changed


@pytest.mark.parametrize("tau,d", [(0.5, 128), (2.0, 128), (6.0, 128), (0.5, 64), (2.0, 64)])
def test_pv_skip_full_rows_ragged(fbm_gpu, tau, d):
    cfg = synth.C1.replace(hq=2, hk=1, s=1000, d=d, dtype="f16")
    nq = cfg.nq
    lut = np.tile(np.arange(nq, dtype=np.int32), (1, 2, nq, 1))
    cnt = np.full((1, 2, nq), nq, dtype=np.int32)
    skipped, changed = _pv_case(fbm_gpu, cfg, tau, lut, cnt)
    assert skipped > 0
    if tau == 0.5:
        assert changed > 0      # the skip visibly changes O: a wrong decision would show


def test_pv_skip_causal_bf16_block_map_lut(fbm_gpu):
    cfg = synth.C1.replace(hq=4, hk=2, s=1000, d=128, dtype="bf16", causal=True, cs=3.0)
    x = cached_prefill(cfg)
    ph = synth.per_head(cfg, 0.5)
    r = oracle.sparge_block_map(x["q"], x["k"], ph, None, synth.per_head(cfg, cfg.simthreshd1),
                                cfg.scale, True, False, dtype="bf16")
    skipped, _ = _pv_case(fbm_gpu, cfg, 2.0, r["lut"], r["count"])
    assert skipped > 0


def test_pv_skip_infinite_threshold_is_bit_identical(fbm_gpu):
    cfg = synth.C1.replace(hq=2, hk=1, s=640, d=128, dtype="f16")
    lut, cnt = hand_lut(cfg, seed=3)
    x, (q, k, v) = prefill_on_gpu(cfg)
    args = (q, k, v, torch.from_numpy(lut).cuda(), torch.from_numpy(cnt).cuda())
    a = fbm_gpu.sparse_fmha_fwd(*args, scale=cfg.scale, return_lse=True)
    b = fbm_gpu.sparse_fmha_fwd(*args, scale=cfg.scale, return_lse=True, pv_threshold=math.inf)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_longest_sequence_sampled(fbm_gpu):
    # s = 65536 (LUT rows of up to 1024 kv blocks), causal GQA with a sink:
    # whole rows and 3-way split partials on sampled q blocks, first and last
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=65536, d=128, dtype="bf16", causal=True,
                           attention_sink=True, topk=0.1)
    lut, cnt = oracle_lut(cfg)
    units = [(0, h, i) for h in range(2) for i in (0, 1, 511, 1022, 1023)]
    check(fbm_gpu, cfg, lut, cnt, units=units)
    check(fbm_gpu, cfg, lut, cnt, units=units, num_splits=3)
