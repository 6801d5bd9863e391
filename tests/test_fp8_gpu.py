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
