"""Writes tests/golden/decode_sm_scale.json: the softmax scale of the sparse
decode workload, found by bisection so that the median effective token count
n_eff = 1 / sum_u p_u^2 over all (query, head) pairs is 15.

The ROCm/aiter sparse-attention pull request (6841, 'peaked' input
distribution) describes logits spread onto about 10-20 effective tokens; the
decode workload targets 15.  Test infrastructure: calls only ``oracle`` and the
input generator.

    python -m oracle.calibrate_decode
"""
from __future__ import annotations

import json
import os

import numpy as np

import synth
from oracle.attention import decode_rows

TARGET = 15.0


def raw_scores(cfg: synth.DecodeConfig) -> np.ndarray:
    """Unscaled q . k of every (query, head, listed token): [C, H, T]."""
    inp = synth.decode(cfg)
    q = synth.bits_to_f64(inp["q"], "bf16")
    rows = decode_rows(inp["page_table"], inp["idx"], cfg.page)
    out = np.empty((cfg.n_queries, cfg.hq, cfg.topk))
    for c in range(cfg.n_queries):
        kv = synth.bits_to_f64(synth.cache_rows(cfg, rows[c]), "bf16")
        out[c] = q[c] @ kv.T
    return out


def median_neff(raw: np.ndarray, scale: float) -> float:
    z = raw * scale
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    return float(np.median(1.0 / (p * p).sum(axis=-1)))


def calibrate(cfg: synth.DecodeConfig, target: float = TARGET) -> float:
    raw = raw_scores(cfg)
    lo, hi = 1e-4, 1.0  # n_eff falls as the scale grows
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if median_neff(raw, mid) > target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def main() -> None:
    cfg = synth.C5
    scale = calibrate(cfg)
    raw = raw_scores(cfg)
    rec = {"config": cfg.name, "seed": cfg.seed, "sm_scale": float(np.float32(scale)),
           "median_n_eff": median_neff(raw, float(np.float32(scale))), "target": TARGET,
           "written_by": "python -m oracle.calibrate_decode"}
    path = os.path.join(os.path.dirname(__file__), "..", "tests", "golden",
                        "decode_sm_scale.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
