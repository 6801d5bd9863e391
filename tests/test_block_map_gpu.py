"""GPU block map (sparge_block_map) against the fp64 oracle on the same seeded
inputs: LUT bit-exact except counted near-ties, ascending rows, -1 padding,
deterministic relaunches."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import SIM_MARGIN, cached_prefill, compare_lut_rows, to_dev

pytestmark = pytest.mark.gpu


def run_case(fbm, cfg, mode, param, heads=None, check_sim_margin=True, smooth_k=False,
             theta=None):
    """param (topk or cdfthreshd) and theta (simthreshd1, default the
    config's) are one value for every head or one value per query head."""
    x = cached_prefill(cfg)
    q, k = to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)
    ph = (synth.per_head(cfg, param) if np.isscalar(param)
          else np.asarray(param, dtype=np.float32))
    th = (synth.per_head(cfg, cfg.simthreshd1 if theta is None else theta)
          if theta is None or np.isscalar(theta) else np.asarray(theta, dtype=np.float32))
    kw = {"topk": ph.tolist()} if mode == "topk" else {"cdfthreshd": ph.tolist()}
    lut, cnt, bmap = fbm.sparge_block_map(q, k, simthreshd1=th.tolist(), scale=cfg.scale,
                                          causal=cfg.causal, attention_sink=cfg.attention_sink,
                                          return_block_map=True, smooth_k=smooth_k, **kw)
    assert fbm.get_error() == 0
    lut, cnt, bmap = lut.cpu().numpy(), cnt.cpu().numpy(), bmap.cpu().numpy()
    ora = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                  ph if mode == "cdf" else None, th, cfg.scale, cfg.causal,
                                  cfg.attention_sink, keep_aux=True, dtype=cfg.dtype, heads=heads,
                                  smooth_k=smooth_k)
    todo = heads or [(b, h) for b in range(cfg.b) for h in range(cfg.hq)]
    exact = near = 0
    for b, h in todo:
        aux = ora["aux"][(b, h)]
        if check_sim_margin:
            for v in (aux["simq"], aux["simk"]):
                assert np.all(np.abs(v - th[h]) > SIM_MARGIN), "sim too close to theta"
        e, n = compare_lut_rows(lut[b, h], cnt[b, h], ora["lut"][b, h], ora["count"][b, h], aux,
                                mode, float(ph[h]), cfg.causal, cfg.attention_sink)
        exact += e
        near += n
        for i in range(lut.shape[2]):
            row = np.zeros(lut.shape[3], dtype=bool)
            row[lut[b, h, i, :cnt[b, h, i]]] = True
            assert (row == bmap[b, h, i].astype(bool)).all()
    print(f"{cfg.name} {mode}={param}: {exact} rows exact, {near} near-tie rows")
    return lut, cnt, exact, near


def test_c1_tiny(fbm_gpu):
    run_case(fbm_gpu, synth.C1, "topk", 0.5)


def test_c1_antithetic_forces_dense_rows_and_columns(fbm_gpu):
    cfg = synth.C1.replace(antithetic_diffuse=True)
    lut, cnt, _, _ = run_case(fbm_gpu, cfg, "topk", 0.5)
    assert (cnt == cfg.nq).any()          # dissimilar q blocks keep every column


def test_c1_theta_half_splits_populations(fbm_gpu):
    cfg = synth.C1.replace(simthreshd1=0.5)
    run_case(fbm_gpu, cfg, "topk", 0.5)


@pytest.mark.parametrize("topk", [0.1, 1e-6, 1.0])
def test_c1_topk_extremes(fbm_gpu, topk):
    lut, cnt, _, _ = run_case(fbm_gpu, synth.C1, "topk", topk)
    if topk == 1.0:
        assert (cnt == synth.C1.nq).all()


def test_c1_causal_sink_gqa(fbm_gpu):
    cfg = synth.C1.replace(hq=4, hk=2, causal=True, attention_sink=True, topk=0.3)
    lut, cnt, _, _ = run_case(fbm_gpu, cfg, "topk", 0.3)
    assert (lut[..., 0] == 0).all()


def test_ragged_sequence(fbm_gpu):
    cfg = synth.C2.replace(b=2, hq=2, hk=1, s=1000, cs_range=None, dtype="f16")
    run_case(fbm_gpu, cfg, "topk", 0.25)
    run_case(fbm_gpu, cfg.replace(causal=True, attention_sink=True), "cdf", 0.8)


def test_c2_cdf(fbm_gpu):
    run_case(fbm_gpu, synth.C2, "cdf", 0.9)


@pytest.mark.parametrize("tau", [0.5, 1.0])
def test_c2_cdf_extremes(fbm_gpu, tau):
    cfg = synth.C2.replace(hq=2, hk=2)
    run_case(fbm_gpu, cfg, "cdf", tau)


def test_c3_full_lut_topk04(fbm_gpu):
    run_case(fbm_gpu, synth.C3, "topk", 0.4)


@pytest.mark.parametrize("topk", [0.1, 0.2, 0.6, 1.0])
def test_c3_sampled_heads(fbm_gpu, topk):
    heads = [(0, 0), (0, 17), (1, 5), (1, 31)]
    run_case(fbm_gpu, synth.C3, "topk", topk, heads=heads)


def test_c4_causal_gqa_sink(fbm_gpu):
    lut, cnt, _, _ = run_case(fbm_gpu, synth.C4, "topk", 0.2)
    assert (lut[..., 0] == 0).all()


# Per-head hyperparameters ("Sparge Attention (Composable Kernel)" README,
# 'Status vs Upstream') on the causal GQA shape of config C4 (32 query heads on
# 8 KV heads, sink), shortened to s = 4096: every head has its own topk or
# cdfthreshd and one of three thresholds (0.001: nothing forced; 0.5: splits
# the diffuse and the compact blocks; 0.99: every block dissimilar, dense
# rows), and every group of four query heads reads a different KV head, so a
# wrong per-head index or KV-head mapping changes the LUT.
C4_SHORT = synth.C4.replace(s=4096)
THETAS = np.array([0.001, 0.5, 0.99, 0.5] * 8, dtype=np.float32)


def test_per_head_topk_and_theta_gqa(fbm_gpu):
    topk = np.linspace(0.05, 0.95, C4_SHORT.hq).astype(np.float32)[::-1].copy()
    lut, cnt, _, _ = run_case(fbm_gpu, C4_SHORT, "topk", topk, theta=THETAS)
    assert (lut[..., 0] == 0).all()
    dense = [h for h in range(C4_SHORT.hq) if THETAS[h] > 0.9]
    nq = C4_SHORT.nq
    for h in dense:  # every block dissimilar: every causally eligible column
        assert (cnt[0, h] == np.arange(1, nq + 1)).all()


def test_per_head_cdf_and_theta_gqa(fbm_gpu):
    cdf = np.linspace(0.5, 0.99, C4_SHORT.hq).astype(np.float32)
    run_case(fbm_gpu, C4_SHORT.replace(topk=None, cdfthreshd=0.9), "cdf", cdf,
             theta=np.roll(THETAS, 1))


def test_block_map_is_deterministic(fbm_gpu):
    cfg = synth.C2.replace(hq=4, hk=2)
    x = synth.prefill(cfg)
    q, k = to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)
    ref = None
    for _ in range(20):
        lut, cnt, _ = fbm_gpu.sparge_block_map(q, k, cdfthreshd=0.9, scale=cfg.scale)
        cur = (lut.cpu(), cnt.cpu())
        if ref is None:
            ref = cur
        assert torch.equal(cur[0], ref[0]) and torch.equal(cur[1], ref[1])


# K smoothing (pre-pool k -= km): keys carry a channel bias common to the whole
# head (key_offset), which makes every unsmoothed K block look similar; the
# thresholds sit where smoothing changes the similar / non-similar split.

def test_smooth_k_c1_key_offset(fbm_gpu):
    cfg = synth.C1.replace(key_offset=2.0, simthreshd1=0.5)
    lut, cnt, _, _ = run_case(fbm_gpu, cfg, "topk", 0.5, smooth_k=True)
    raw_lut, raw_cnt, _, _ = run_case(fbm_gpu, cfg, "topk", 0.5, smooth_k=False)
    assert not np.array_equal(cnt, raw_cnt)  # smoothing changed the map on this input


def test_smooth_k_causal_gqa_sink(fbm_gpu):
    cfg = synth.C1.replace(hq=4, hk=2, causal=True, attention_sink=True, key_offset=2.0,
                           simthreshd1=0.5)
    lut, cnt, _, _ = run_case(fbm_gpu, cfg, "topk", 0.3, smooth_k=True)
    assert (lut[..., 0] == 0).all()


def test_smooth_k_ragged_sequence(fbm_gpu):
    # s = 1000: the last K block has 40 rows and weighs 40 / 1000 in the mean
    cfg = synth.C2.replace(b=2, hq=2, hk=1, s=1000, cs_range=None, dtype="f16",
                           key_offset=1.5, simthreshd1=0.4)
    run_case(fbm_gpu, cfg, "topk", 0.25, smooth_k=True)
    run_case(fbm_gpu, cfg.replace(causal=True, attention_sink=True), "cdf", 0.8, smooth_k=True)


def test_smooth_k_c2_cdf(fbm_gpu):
    cfg = synth.C2.replace(key_offset=2.0, simthreshd1=0.3)
    run_case(fbm_gpu, cfg, "cdf", 0.9, smooth_k=True)


def test_smooth_k_c3_sampled_heads(fbm_gpu):
    heads = [(0, 3), (1, 30)]
    run_case(fbm_gpu, synth.C3, "topk", 0.4, heads=heads, smooth_k=True)



def _tied_case(fbm, cfg, period, mode, param):
    """K blocks j set to copies of block j mod `period` (every block when
    period = 1), so the pooled scores of a row take only `period` distinct
    values, each many times over: the selection threshold falls inside a group
    of exactly equal scores and the lower kv blocks must be taken first.  The
    GPU scores of identical blocks are bitwise equal, so every row must match
    the oracle exactly."""
    x = dict(cached_prefill(cfg))
    k = x["k"].copy()
    nb = cfg.nq
    for j in range(period, nb):
        src = j % period
        k[:, :, j * 64:(j + 1) * 64, :] = k[:, :, src * 64:(src + 1) * 64, :]
    q_d, k_d = to_dev(x["q"], cfg.dtype), to_dev(k, cfg.dtype)
    ph = synth.per_head(cfg, param)
    th = synth.per_head(cfg, cfg.simthreshd1)
    kw = {"topk": ph.tolist()} if mode == "topk" else {"cdfthreshd": ph.tolist()}
    lut, cnt, _ = fbm.sparge_block_map(q_d, k_d, simthreshd1=th.tolist(), scale=cfg.scale,
                                       causal=cfg.causal, attention_sink=cfg.attention_sink, **kw)
    assert fbm.get_error() == 0
    lut, cnt = lut.cpu().numpy(), cnt.cpu().numpy()
    ora = oracle.sparge_block_map(x["q"], k, ph if mode == "topk" else None,
                                  ph if mode == "cdf" else None, th, cfg.scale, cfg.causal,
                                  cfg.attention_sink, dtype=cfg.dtype)
    assert (cnt == ora["count"]).all()
    assert (lut == ora["lut"]).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("period", [5, 1])
def test_exact_ties_take_lower_blocks_first(fbm_gpu, causal, period):
    # nq = 64: about 13 copies of each score (the in-bin ranking with ties),
    # or a single value (a zero score range: the bitwise search)
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=4096, d=128, dtype="f16", causal=causal)
    _tied_case(fbm_gpu, cfg, period, "topk", 0.3)


def test_exact_ties_in_a_crowded_bin(fbm_gpu):
    # nq = 256: about 51 equal scores per value, more than a warp can rank
    # pairwise, so the crossing bin goes through the bitwise search
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=16384, d=128, dtype="bf16")
    _tied_case(fbm_gpu, cfg, 5, "topk", 0.45)


def test_exact_ties_cdf(fbm_gpu):
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=4096, d=64, dtype="f16")
    _tied_case(fbm_gpu, cfg, 7, "cdf", 0.6)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode,param", [("topk", 0.1), ("cdf", 0.9)])
def test_longest_sequence(fbm_gpu, causal, mode, param):
    # s = 65536: nk = 1024, the most the block map takes.  The selection runs
    # its 32-scores-per-lane kernels (causal rows their 8 / 16 / 24 / 32
    # bodies) and the scores kernel eight 128-block tiles per row of tiles
    cfg = synth.C1.replace(b=1, hq=2, hk=1, s=65536, d=128, dtype="bf16", causal=causal,
                           attention_sink=causal)
    run_case(fbm_gpu, cfg, mode, param)


@pytest.mark.parametrize("causal", [False, True])
def test_cdf_with_512_kv_blocks(fbm_gpu, causal):
    # nk = 512: the 16-scores-per-lane cdf kernel
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=32768, d=64, dtype="f16", causal=causal)
    run_case(fbm_gpu, cfg, "cdf", 0.8)


def _c4_small(seed):
    """A causal GQA + sink case with 256 kv blocks (the chained launches of the
    score and selection kernels, and the causal selection bodies)."""
    return synth.C4.replace(s=16384, hq=8, hk=2, seed=seed)


def test_back_to_back_calls_share_a_workspace(fbm_gpu):
    """Two block maps on one stream, one workspace, no sync between them: each
    LUT equals the one its inputs give alone (each kernel of the second call
    starts only after the kernels of the first it could disturb)."""
    fbm = fbm_gpu
    outs, solo = [], []
    cfgs = [_c4_small(11), _c4_small(12)]
    ins = []
    for cfg in cfgs:
        x = synth.prefill(cfg)
        ins.append((to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)))
    cfg = cfgs[0]
    ws = torch.empty(fbm.block_map_workspace_bytes(cfg.b, cfg.hq, cfg.hk, cfg.s, cfg.d),
                     dtype=torch.uint8, device="cuda")
    kw = dict(topk=cfg.topk, simthreshd1=cfg.simthreshd1, scale=cfg.scale, causal=True,
              attention_sink=True)
    for q, k in ins:
        solo.append(tuple(t.clone() for t in fbm.sparge_block_map(q, k, workspace=ws, **kw)[:2]))
        torch.cuda.synchronize()
    for q, k in ins:
        outs.append(fbm.sparge_block_map(q, k, workspace=ws, **kw)[:2])
    torch.cuda.synchronize()
    assert fbm.get_error() == 0
    for (lut, cnt), (slut, scnt) in zip(outs, solo):
        assert torch.equal(lut, slut) and torch.equal(cnt, scnt)
    assert not torch.equal(outs[0][0], outs[1][0])  # the two inputs select differently


def test_graph_capture_matches_eager(fbm_gpu):
    """The block map captured in a CUDA graph (its chained launches become graph
    dependencies) and replayed gives the eager LUT."""
    fbm = fbm_gpu
    cfg = _c4_small(13)
    x = synth.prefill(cfg)
    q, k = to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)
    kw = dict(topk=cfg.topk, simthreshd1=cfg.simthreshd1, scale=cfg.scale, causal=True,
              attention_sink=True)
    ref_lut, ref_cnt = (t.clone() for t in fbm.sparge_block_map(q, k, **kw)[:2])
    lut = torch.full_like(ref_lut, 7)
    cnt = torch.full_like(ref_cnt, 7)
    ws = torch.empty(fbm.block_map_workspace_bytes(cfg.b, cfg.hq, cfg.hk, cfg.s, cfg.d),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        fbm.sparge_block_map(q, k, lut=lut, lut_count=cnt, workspace=ws, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert fbm.get_error() == 0
    assert torch.equal(lut, ref_lut) and torch.equal(cnt, ref_cnt)
