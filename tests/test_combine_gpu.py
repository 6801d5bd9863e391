"""GPU attn_combine against the fp64 oracle combine (the lse_max merge of the
updating_log's Stage 1), with empty partials and all-empty rows."""
import numpy as np
import pytest
import torch

import oracle
from _util import assert_close_lse, assert_close_o

pytestmark = pytest.mark.gpu


def partials(S, rows, dv, seed):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((S, rows, dv)).astype(np.float32)
    lse = (rng.standard_normal((S, rows)) * 3).astype(np.float32)
    empty = rng.random((S, rows)) < 0.2
    lse[empty] = -np.inf
    o[empty] = 0.0
    lse[:, :3] = -np.inf  # all-empty rows
    o[:, :3] = 0.0
    return o, lse


@pytest.mark.parametrize("S", [1, 2, 3, 8, 64])
@pytest.mark.parametrize("dv", [64, 128, 512])
def test_combine_f32(fbm_gpu, S, dv):
    o, lse = partials(S, 1000, dv, S * 7 + dv)
    out, lse_out = fbm_gpu.attn_combine(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(),
                                        out_dtype=torch.float32)
    ro, rl = oracle.combine(o.astype(np.float64), lse.astype(np.float64))
    got = out.double().cpu().numpy()
    assert np.abs(got - ro).max() < 1e-5
    gl = lse_out.double().cpu().numpy()
    assert (np.isneginf(gl) == np.isneginf(rl)).all()
    fin = np.isfinite(rl)
    assert np.abs(gl[fin] - rl[fin]).max() < 1e-5
    assert (got[:3] == 0).all()


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_combine_half_outputs(fbm_gpu, dt):
    o, lse = partials(4, 777, 128, 11)
    out, lse_out = fbm_gpu.attn_combine(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(),
                                        out_dtype=dt)
    ro, rl = oracle.combine(o.astype(np.float64), lse.astype(np.float64))
    assert_close_o(out.double().cpu().numpy(), ro)
    assert_close_lse(lse_out.double().cpu().numpy(), rl)
