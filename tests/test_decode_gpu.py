"""GPU sparse decode (sparse_decode_fwd + attn_combine) against the fp64 oracle:
paged gathers of top-k token rows, V = latent plane, split-KV partials."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_close_lse, assert_close_o
from oracle.attention import decode_rows

pytestmark = pytest.mark.gpu


def gpu_cache(cfg, device="cuda"):
    n_rows = cfg.n_pages * cfg.page
    cache = torch.empty((n_rows, cfg.d), dtype=torch.bfloat16, device=device)
    step = 1 << 18
    for r0 in range(0, n_rows, step):
        r1 = min(n_rows, r0 + step)
        cache[r0:r1] = synth.cache_rows_torch(cfg, r0, r1, device)
    return cache.view(cfg.n_pages, cfg.page, cfg.d)


def run(fbm, cfg, S, inp=None, cache=None, queries=None, idx_override=None):
    inp = inp or synth.decode(cfg)
    cache = cache if cache is not None else gpu_cache(cfg)
    idx = inp["idx"] if idx_override is None else idx_override
    q_bits = inp["q"]
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pt = torch.from_numpy(inp["page_table"]).cuda()
    ix = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    op, lp = fbm.sparse_decode_fwd(q, cache, pt, ix, dv=cfg.dv, scale=cfg.sm_scale, num_splits=S)
    out, lse = fbm.attn_combine(op, lp, out_dtype=torch.bfloat16)
    assert fbm.get_error() == 0
    op, lp = op.double().cpu().numpy(), lp.double().cpu().numpy()
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    qf = synth.bits_to_f64(q_bits, "bf16")
    rows = decode_rows(inp["page_table"], np.maximum(idx, 0), cfg.page)
    for c in (queries if queries is not None else range(cfg.n_queries)):
        keep = idx[c] >= 0
        kv = synth.bits_to_f64(synth.cache_rows(cfg, rows[c][keep]), "bf16")
        # partials follow the chunks of the full list (sentinels included)
        bounds = oracle.split_bounds(idx.shape[1], S)
        for s, (lo, hi) in enumerate(bounds):
            sel = keep[lo:hi]
            kv_s = synth.bits_to_f64(synth.cache_rows(cfg, rows[c][lo:hi][sel]), "bf16")
            po, pl = oracle.decode_attention(qf[c], kv_s, cfg.dv, cfg.sm_scale)
            assert_close_o(op[s, c], po, f"Opart q{c} s{s}")
            assert_close_lse(lp[s, c], pl, f"LSEpart q{c} s{s}")
        ro, rl = oracle.decode_attention(qf[c], kv, cfg.dv, cfg.sm_scale)
        assert_close_o(out[c], ro, f"O q{c}")
        assert_close_lse(lse[c], rl, f"LSE q{c}")


SMALL = synth.C5.replace(n_queries=8, pages_per_query=32, topk=300)


@pytest.mark.parametrize("S", [1, 2, 3, 8])
def test_small_decode(fbm_gpu, S):
    run(fbm_gpu, SMALL, S)


def test_sentinels_are_skipped(fbm_gpu):
    inp = synth.decode(SMALL)
    idx = inp["idx"].copy()
    idx[:, ::7] = -1
    idx[0, :] = -1  # a query with nothing to attend: O = 0, LSE = -inf
    run(fbm_gpu, SMALL, 3, inp=inp, idx_override=idx)


def test_full_decode_sampled(fbm_gpu):
    cfg = synth.C5
    inp = synth.decode(cfg)
    cache = gpu_cache(cfg)
    for S in (2, 4, 8):
        run(fbm_gpu, cfg, S, inp=inp, cache=cache, queries=[0, 13, 37, 63])


@pytest.mark.parametrize("S", [17, 20, 32])
def test_short_chunks(fbm_gpu, S):
    # 300 tokens in 17 / 20 / 32 chunks: 17-18, 15 and 9-10 tokens each, so a
    # chunk has two 16-token tiles, one full tile or one partial tile (the
    # second warp group of the CTA then has one short tile or none)
    run(fbm_gpu, SMALL, S)


def test_f16_cache(fbm_gpu):
    # the same decode with an f16 query and cache: the bf16 values of the
    # generator are exactly representable in f16, so the oracle values are the same
    cfg = SMALL
    inp = synth.decode(cfg)
    cache = gpu_cache(cfg).to(torch.float16)
    qf = synth.bits_to_f64(inp["q"], "bf16")
    assert np.abs(qf).max() < 60000 and np.abs(cache.float().cpu().numpy()).max() < 60000
    q = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).cuda().to(torch.float16)
    assert torch.equal(q.to(torch.float64).cpu(), torch.from_numpy(qf))
    op, lp = fbm_gpu.sparse_decode_fwd(q, cache, torch.from_numpy(inp["page_table"]).cuda(),
                                       torch.from_numpy(inp["idx"]).cuda(), dv=cfg.dv,
                                       scale=cfg.sm_scale, num_splits=3)
    out, lse = fbm_gpu.attn_combine(op, lp, out_dtype=torch.float16)
    assert fbm_gpu.get_error() == 0
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    rows = decode_rows(inp["page_table"], inp["idx"], cfg.page)
    for c in range(cfg.n_queries):
        kv = synth.bits_to_f64(synth.cache_rows(cfg, rows[c]), "bf16")
        ro, rl = oracle.decode_attention(qf[c], kv, cfg.dv, cfg.sm_scale)
        assert_close_o(out[c], ro, f"O q{c}")
        assert_close_lse(lse[c], rl, f"LSE q{c}")


def test_graph_capture_matches_eager(fbm_gpu):
    """Decode + combine (chained launches) captured in a CUDA graph and replayed
    give the eager partials and output, bit for bit."""
    fbm = fbm_gpu
    cfg = synth.C5.replace(n_queries=8, pages_per_query=16, topk=300)
    inp = synth.decode(cfg)
    cache = gpu_cache(cfg)
    q = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).cuda()
    pt = torch.from_numpy(inp["page_table"]).cuda()
    ix = torch.from_numpy(inp["idx"]).cuda()
    S = 3
    kw = dict(dv=cfg.dv, scale=cfg.sm_scale, num_splits=S)
    op0, lp0 = fbm.sparse_decode_fwd(q, cache, pt, ix, **kw)
    out0, lse0 = fbm.attn_combine(op0, lp0, out_dtype=torch.bfloat16)
    op = torch.full_like(op0, 7.0)
    lp = torch.full_like(lp0, 7.0)
    out = torch.zeros_like(out0)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        fbm.sparse_decode_fwd(q, cache, pt, ix, o_partial=op, lse_partial=lp, **kw)
        _, lse = fbm.attn_combine(op, lp, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert fbm.get_error() == 0
    assert torch.equal(op, op0) and torch.equal(lp, lp0)
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
