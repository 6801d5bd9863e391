"""Failure detection on the GPU without a fault: a bounded mbarrier wait on a
barrier that nothing arrives on gives up, reports FBM_DEVERR_TIMEOUT through
the device error word, and leaves the context usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import assert_close_o, prefill_on_gpu

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_stays_usable(fbm_gpu):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fbm_gpu.selftest_wait_timeout(50_000_000)  # 50 ms
    bits = fbm_gpu.get_error()
    dt = time.perf_counter() - t0
    assert bits == fbm_gpu.FBM_DEVERR_TIMEOUT
    assert dt >= 0.045
    assert fbm_gpu.get_error() == 0  # reading cleared it
    # the next real call runs normally and is correct
    cfg = synth.C1.replace(b=1, hq=2, hk=2, s=256, d=128, dtype="bf16")
    x, (q, k, v) = prefill_on_gpu(cfg)
    out, _ = fbm_gpu.sparse_fmha_fwd(q, k, v, None, None, scale=cfg.scale)
    assert fbm_gpu.get_error() == 0
    nq = cfg.nq
    lut = np.tile(np.arange(nq, dtype=np.int32), (1, 2, nq, 1))
    cnt = np.full((1, 2, nq), nq, dtype=np.int32)
    res = oracle.sparse_fmha(x["q"], x["k"], x["v"], lut, cnt, cfg.scale, False, dtype="bf16")
    o = out.double().cpu().numpy()
    for (b, h, i), (o_ref, _) in res.items():
        assert_close_o(o[b, h, i * 64:(i + 1) * 64], o_ref)


def test_selftest_rejects_bad_limits(fbm_gpu):
    with pytest.raises(fbm_gpu.FbmError):
        fbm_gpu.selftest_wait_timeout(0)
