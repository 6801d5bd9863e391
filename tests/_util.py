"""Helpers shared by the GPU parity tests (not collected by pytest)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}

# tolerances: output atol 4e-2 / rtol 1e-2 (fp16 / bf16, the dense-FMHA tolerance of the
# Sparge Attention (Composable Kernel) validation), LSE 1e-3 nats (the bf16 LSE error the
# ROCm/aiter sparse MHA pull reports is 0.0009 nats),
# LUT bit-exact except near-ties with pooled-score gap < 1e-6 (counted)
O_ATOL, O_RTOL, LSE_TOL = 4e-2, 1e-2, 1e-3
SCORE_GAP = 1e-6
MASS_EPS = 1e-5
SIM_MARGIN = 1e-4


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).to(device)


@functools.lru_cache(maxsize=2)
def cached_prefill(cfg: synth.PrefillConfig) -> dict:
    return synth.prefill(cfg)


def prefill_on_gpu(cfg: synth.PrefillConfig):
    x = cached_prefill(cfg)
    return x, tuple(to_dev(x[t], cfg.dtype) for t in ("q", "k", "v"))


def assert_close_o(got: np.ndarray, want: np.ndarray, what: str = "O"):
    err = np.abs(got - want)
    bad = err > O_ATOL + O_RTOL * np.abs(want)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance, max abs err "
                           f"{err.max():.3e}")
    return float(err.max())


def assert_close_lse(got: np.ndarray, want: np.ndarray, what: str = "LSE"):
    ninf_w, ninf_g = np.isneginf(want), np.isneginf(got)
    assert (ninf_w == ninf_g).all(), f"{what}: -inf pattern differs"
    fin = ~ninf_w
    err = np.abs(got[fin] - want[fin]) if fin.any() else np.zeros(1)
    assert err.max() <= LSE_TOL, f"{what}: max err {err.max():.3e} nats"
    return float(err.max())


def compare_lut_rows(gpu_lut, gpu_cnt, ora_lut, ora_cnt, aux, mode: str, param: float,
                     causal: bool, sink: bool):
    """Compare one head's LUT rows [nq, nk].  Rows must match exactly, except
    where the difference is explained by a near-tie of the fp64 pooled scores
    (gap < SCORE_GAP at the selection boundary) or, in cdf mode, by a
    cumulative mass within MASS_EPS of the threshold.  Returns (n_exact,
    n_near_tie); raises AssertionError on any other difference."""
    nq, nk = ora_lut.shape
    score, sel = aux["score"], aux["selected"]
    finite = np.isfinite(score)
    exact = near = 0
    for i in range(nq):
        G = np.zeros(nk, dtype=bool)
        O = np.zeros(nk, dtype=bool)
        gc = int(gpu_cnt[i])
        assert 0 <= gc <= nk, f"row {i}: count {gc}"
        grow = gpu_lut[i, :gc]
        assert (np.diff(grow) > 0).all(), f"row {i}: not strictly ascending {grow}"
        assert (gpu_lut[i, gc:] == -1).all(), f"row {i}: padding not -1"
        G[grow] = True
        O[ora_lut[i, :ora_cnt[i]]] = True
        if (G == O).all():
            exact += 1
            continue
        D = G ^ O
        forced = O & ~sel[i]
        assert not (D & forced).any(), f"row {i}: forced entries differ"
        assert finite[i][D].all(), f"row {i}: a non-selectable entry differs"
        chosen = sel[i] & finite[i]
        bnd = score[i][chosen].min()
        if np.all(np.abs(score[i][D] - bnd) < SCORE_GAP):
            if mode == "topk":
                # K_i fixes how many blocks are selected: a near-tie swaps
                # entries but keeps the count, except when the sink column
                # (forced on whether or not it is also selected) is one of the
                # tied entries
                oc = int(ora_cnt[i])
                sink_tie = sink and finite[i][0] and abs(score[i][0] - bnd) < SCORE_GAP
                assert gc == oc or (sink_tie and abs(gc - oc) == 1), \
                    f"row {i}: topk count {gc} != oracle {oc}"
            near += 1
            continue
        if mode == "cdf":
            idx = np.nonzero(finite[i])[0]
            sc = score[i][idx]
            p = np.exp(sc - sc.max())
            p /= p.sum()
            order = idx[np.lexsort((idx, -p))]
            cum = np.cumsum(np.sort(p)[::-1])
            m_o = int(chosen.sum())
            gsel = G & finite[i] & ~(forced & ~chosen)
            m_g = int(gsel.sum())
            top = np.zeros(nk, dtype=bool)
            top[order[:m_g]] = True
            # every prefix length between the two counts ends within MASS_EPS of
            # the threshold: the fp32 and fp64 cumulative masses may stop anywhere
            # in that band
            lo_len, hi_len = min(m_o, m_g), max(m_o, m_g)
            band = [abs(cum[n - 1] - param) < MASS_EPS for n in range(max(lo_len, 1), hi_len + 1)]
            if (top == gsel).all() and all(band):
                near += 1
                continue
        raise AssertionError(f"row {i}: LUT differs beyond near-ties: gpu {sorted(np.nonzero(G)[0])}"
                             f" oracle {sorted(np.nonzero(O)[0])}")
    return exact, near
