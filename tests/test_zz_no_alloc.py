"""The scratch-free block map entry point (sparge_block_map_static).

Some callers cannot allocate device memory when they call the library (a
runtime that plans every buffer up front and hands an operation only its
inputs and outputs, or a hot path that must stay out of the allocator).  For
them the library keeps the block map's scratch in a static device array.  This
file checks, through the C ABI, that two calls in a row give exactly the LUT,
counts and block map of the workspace version (LUTs are integer results, so the
tolerance is bit-exact), including a second call on a different shape that
reuses the array left over from the first.  It is named so that pytest runs it
last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from _util import to_dev

pytestmark = pytest.mark.gpu


def _call_static(fbm, q, k, mode, param, theta, causal, sink, bmap):
    b, hq, s, d = q.shape
    hk = k.shape[1]
    nq = (s + 63) // 64
    lut = torch.full((b, hq, nq, nq), 7, dtype=torch.int32, device=q.device)
    cnt = torch.full((b, hq, nq), 7, dtype=torch.int32, device=q.device)
    arr = lambda v: (ctypes.c_float * hq)(*([v] * hq))
    topk = arr(param) if mode == "topk" else None
    cdf = arr(param) if mode == "cdf" else None
    st = fbm.lib().sparge_block_map_static(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        fbm.FBM_F16 if q.dtype == torch.float16 else fbm.FBM_BF16, b, hq, hk, s, d, 64, 64,
        topk, cdf, arr(theta), 1.0 / math.sqrt(d), int(causal), int(sink), 0,
        ctypes.c_void_p(lut.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
        ctypes.c_void_p(bmap.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fbm.FBM_OK, fbm.lib().fbm_last_error_message()
    return lut, cnt


@pytest.mark.parametrize("first,second", [("C2", "C1"), ("C1", "C2")])
def test_static_scratch_matches_workspace_version(fbm_gpu, first, second):
    cases = {
        "C2": (synth.C2.replace(hq=4, hk=2), "cdf", 0.9),
        "C1": (synth.C1.replace(hq=4, hk=2, causal=True, attention_sink=True), "topk", 0.3),
    }
    for name in (first, second):
        cfg, mode, param = cases[name]
        x = synth.prefill(cfg)
        q, k = to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)
        kw = {"topk": param} if mode == "topk" else {"cdfthreshd": param}
        ref_lut, ref_cnt, ref_map = fbm_gpu.sparge_block_map(
            q, k, simthreshd1=cfg.simthreshd1, scale=cfg.scale, causal=cfg.causal,
            attention_sink=cfg.attention_sink, return_block_map=True, **kw)
        bmap = torch.empty_like(ref_map)
        lut, cnt = _call_static(fbm_gpu, q, k, mode, param, cfg.simthreshd1, cfg.causal,
                                cfg.attention_sink, bmap)
        assert fbm_gpu.get_error() == 0
        assert torch.equal(lut, ref_lut)
        assert torch.equal(cnt, ref_cnt)
        assert torch.equal(bmap, ref_map)


def test_static_scratch_headline_shape_fits_and_matches(fbm_gpu):
    cfg = synth.C3
    x = synth.prefill(cfg.replace(b=1))
    q, k = to_dev(x["q"], "f16"), to_dev(x["k"], "f16")
    ref_lut, ref_cnt, _ = fbm_gpu.sparge_block_map(q, k, topk=0.4, scale=cfg.scale)
    for _ in range(2):
        lut, cnt, _ = fbm_gpu.sparge_block_map_static(q, k, topk=0.4, scale=cfg.scale)
        assert torch.equal(lut, ref_lut) and torch.equal(cnt, ref_cnt)


def test_static_scratch_with_k_smoothing_matches(fbm_gpu):
    cfg = synth.C2.replace(hq=4, hk=2, key_offset=2.0, simthreshd1=0.3)
    x = synth.prefill(cfg)
    q, k = to_dev(x["q"], cfg.dtype), to_dev(x["k"], cfg.dtype)
    a = fbm_gpu.sparge_block_map(q, k, cdfthreshd=0.9, simthreshd1=0.3, scale=cfg.scale,
                                 smooth_k=True)
    b = fbm_gpu.sparge_block_map_static(q, k, cdfthreshd=0.9, simthreshd1=0.3, scale=cfg.scale,
                                        smooth_k=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
