"""fp8 (e4m3) Q/K on the GPU against the oracle's fp8 reading on the same seeded
inputs: the block quantisation bit-exact (codes and scales), and the attention
over the quantised scores (sparse_fmha_fwd_fp8) within the attention
tolerances (O atol 4e-2 / rtol 1e-2, LSE 1e-3 nats) of the oracle's fp8
attention.  The distance of the fp8 result from exact attention is a property
of the format on these inputs and is printed, not tested."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_close_lse, assert_close_o, cached_prefill, prefill_on_gpu

pytestmark = pytest.mark.gpu

_TAB = oracle.e4m3_values()


def decode(codes: np.ndarray) -> np.ndarray:
    """e4m3 code bytes -> values (the oracle's table; 0x7f / 0xff are NaN)."""
    c = codes.astype(np.int64)
    mag = c & 0x7F
    assert (mag < 127).all(), "NaN code"
    return np.where(c & 0x80, -1.0, 1.0) * _TAB[mag]


def check_quant(fbm, x_bits, dtype, x_dev):
    codes, scales = fbm.quantize_e4m3_blocks(x_dev)
    assert fbm.get_error() == 0
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    b, h, s, d = x_bits.shape
    for bi in range(b):
        for hi in range(h):
            xf = synth.bits_to_f64(x_bits[bi, hi], dtype)
            vals, qs = oracle.quantize_blocks_e4m3(xf, 64)
            assert np.array_equal(scales[bi, hi].astype(np.float64), qs), (bi, hi)
            assert np.array_equal(decode(codes[bi, hi]), vals), (bi, hi)
    return codes, scales


def test_quantisation_bit_exact_ragged_with_zero_block(fbm_gpu):
    cfg = synth.C1.replace(hq=2, hk=2, s=1000, d=128, dtype="f16")
    x = cached_prefill(cfg)
    q = x["q"].copy()
    q[0, 1, 64:128] = 0                      # an all-zero block: scale 1, zero codes
    qd = torch.from_numpy(q.view(np.int16)).view(torch.float16).cuda()
    codes, scales = check_quant(fbm_gpu, q, "f16", qd)
    assert scales[0, 1, 1] == 1.0 and (codes[0, 1, 64:128] & 0x7F == 0).all()


def run_fp8(fbm, cfg, mode, param, units):
    x, (q, k, v) = prefill_on_gpu(cfg)
    check_quant(fbm, x["q"], cfg.dtype, q)
    check_quant(fbm, x["k"], cfg.dtype, k)
    ph = synth.per_head(cfg, param)
    r = oracle.sparge_block_map(x["q"], x["k"], ph if mode == "topk" else None,
                                ph if mode == "cdf" else None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, cfg.causal,
                                cfg.attention_sink, dtype=cfg.dtype,
                                heads=sorted({(b, h) for b, h, _ in units}))
    lut, cnt = r["lut"], r["count"]
    q8, qs = fbm.quantize_e4m3_blocks(q)
    k8, ks = fbm.quantize_e4m3_blocks(k)
    out, lse = fbm.sparse_fmha_fwd_fp8(q8, qs, k8, ks, v, torch.from_numpy(lut).cuda(),
                                       torch.from_numpy(cnt).cuda(), scale=cfg.scale,
                                       causal=cfg.causal, return_lse=True)
    assert fbm.get_error() == 0
    o_np, l_np = out.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)
    ratio = cfg.hq // cfg.hk
    d_exact = 0.0
    for b, h, i in units:
        qh = synth.bits_to_f64(x["q"][b, h], cfg.dtype)
        kg = synth.bits_to_f64(x["k"][b, h // ratio], cfg.dtype)
        vg = synth.bits_to_f64(x["v"][b, h // ratio], cfg.dtype)
        row = lut[b, h, i, :cnt[b, h, i]]
        o_ref, l_ref = oracle.attention_unit_fp8(qh, kg, vg, row, i, 64, 64, cfg.scale, cfg.causal)
        rows = slice(i * 64, i * 64 + o_ref.shape[0])
        assert_close_o(o_np[b, h, rows], o_ref, f"O {(b, h, i)}")
        assert_close_lse(l_np[b, h, rows], l_ref, f"LSE {(b, h, i)}")
        l_ex = oracle.attention_unit(qh, kg, vg, row, i, 64, 64, cfg.scale, cfg.causal)[1]
        fin = np.isfinite(l_ex)
        if fin.any():
            d_exact = max(d_exact, float(np.abs(l_np[b, h, rows][fin] - l_ex[fin]).max()))
    print(f"{cfg.name}: {len(units)} q blocks; fp8 LSE vs exact attention: max {d_exact:.3f} nats")


def test_fp8_attention_ragged_gqa_bf16(fbm_gpu):
    cfg = synth.C2.replace(b=1, hq=4, hk=2, s=1000, cs_range=None)
    units = [(0, h, i) for h in range(4) for i in range(cfg.nq)]
    run_fp8(fbm_gpu, cfg, "topk", 0.5, units)


def test_fp8_attention_causal_sink_f16(fbm_gpu):
    cfg = synth.C1.replace(hq=2, hk=1, s=1000, d=128, dtype="f16", causal=True,
                           attention_sink=True)
    units = [(0, h, i) for h in range(2) for i in range(cfg.nq)]
    run_fp8(fbm_gpu, cfg, "topk", 0.3, units)


def test_fp8_attention_headline_sampled(fbm_gpu):
    cfg = synth.C3
    units = [(0, 3, 0), (0, 3, 255), (1, 20, 100), (1, 20, 255)]
    run_fp8(fbm_gpu, cfg, "topk", 0.4, units)


@pytest.mark.parametrize("smooth_k", [False, True])
def test_fused_block_map_codes_bit_exact(fbm_gpu, smooth_k):
    # the e4m3 codes and scales written by the block map's pooling pass equal
    # the oracle's quantisation of the raw rows (ragged s = 1000, an all-zero Q
    # block, bf16 GQA), and the LUT is the one the plain block map writes
    cfg = synth.C2.replace(b=1, hq=4, hk=2, s=1000, cs_range=None)
    x = cached_prefill(cfg)
    qb = x["q"].copy()
    qb[0, 2, 128:192] = 0
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, k = dev(qb), dev(x["k"])
    kw = dict(topk=0.5, scale=cfg.scale, causal=True, attention_sink=True, smooth_k=smooth_k)
    lut, cnt, _, q8, qs, k8, ks = fbm_gpu.sparge_block_map_e4m3(q, k, **kw)
    lut0, cnt0, _ = fbm_gpu.sparge_block_map(q, k, **kw)
    assert fbm_gpu.get_error() == 0
    assert torch.equal(lut, lut0) and torch.equal(cnt, cnt0)
    for bits, codes, scales in ((qb, q8, qs), (x["k"], k8, ks)):
        codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
        for h in range(bits.shape[1]):
            vals, sc = oracle.quantize_blocks_e4m3(synth.bits_to_f64(bits[0, h], "bf16"), 64)
            assert np.array_equal(scales[0, h].astype(np.float64), sc), h
            assert np.array_equal(decode(codes[0, h]), vals), h
    assert qs[0, 2, 2].item() == 1.0


def test_fused_block_map_codes_headline_heads(fbm_gpu):
    # headline shape: the fused codes equal the separate quantiser's, and two
    # heads of them the oracle's
    cfg = synth.C3
    x, (q, k, v) = prefill_on_gpu(cfg)
    lut, cnt, _, q8, qs, k8, ks = fbm_gpu.sparge_block_map_e4m3(q, k, topk=0.4, scale=cfg.scale)
    q8b, qsb = fbm_gpu.quantize_e4m3_blocks(q)
    k8b, ksb = fbm_gpu.quantize_e4m3_blocks(k)
    assert fbm_gpu.get_error() == 0
    assert torch.equal(q8, q8b) and torch.equal(qs, qsb)
    assert torch.equal(k8, k8b) and torch.equal(ks, ksb)
    for bi, h in ((0, 0), (1, 31)):
        vals, sc = oracle.quantize_blocks_e4m3(synth.bits_to_f64(x["q"][bi, h], cfg.dtype), 64)
        assert np.array_equal(qs[bi, h].cpu().numpy().astype(np.float64), sc)
        assert np.array_equal(decode(q8[bi, h].cpu().numpy()), vals)
