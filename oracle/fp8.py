"""fp8 (e4m3) Q/K for the QK^T product: per-block quantisation and the attention
over the quantised scores (test infrastructure; see the package header).

Sources:
* "Sparge Attention (Composable Kernel)" README, 'Not yet ported': Q/K
  quantisation fused into the pool kernel, so that the attention kernel's
  first GEMM runs on narrow operands.  (The README names int8; the GB300
  tensor cores take fp8, so e4m3 with one scale per 64-token block is the
  format here.)
* ROCm/aiter pull 6841: the bf16fp8 recipe (fp8 Q/K, 16-bit V) and its
  measured LSE error against exact attention (about 0.03 nats).

e4m3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
infinities, the all-ones pattern is NaN, largest finite value 448, smallest
positive 2^-9.  Rounding is to nearest, ties to the even code, saturating at
+-448 (the PTX cvt.rn.satfinite behaviour).

Reading taken (the pages give no recipe): for each 64-row block X of Q or K
(per (batch, head)), amax = max |x| over the block, taken in fp32 (exact for
fp16 / bf16 inputs); qscale = fp32(amax / 448) and inv = fp32(448 / amax)
(both 1 for an all-zero block); code = e4m3(fp32(x * inv)); the block is
represented as qscale * code.  Scores: S_tu = scale * qscale_Q(i) *
qscale_K(j) * sum_d codeQ_td codeK_ud, the sum exact (fp64 here; every e4m3
product is exact in fp32 and the tensor core accumulates in fp32).  V, P and
the softmax are as in attention.py.
"""
from __future__ import annotations

from typing import Iterable, Tuple

import numpy as np

from .attention import _softmax_attend, row_keys

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """The non-negative finite e4m3 values in code order (codes 0 .. 126):
    subnormals m/8 * 2^-6 (m = 0 .. 7), then (1 + m/8) * 2^(e - 7) for
    e = 1 .. 15, m = 0 .. 7, without e = 15, m = 7 (NaN)."""
    vals = [m / 8.0 * 2.0 ** -6 for m in range(8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_TABLE = e4m3_values()


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value of each element, ties to the even code, saturating at
    +-448 (values, as float64)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_TABLE, a, side="left"), 0, len(_TABLE) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _TABLE[lo], _TABLE[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    out = np.where(pick_hi, _TABLE[hi], _TABLE[lo])
    return np.copysign(out, x)


def quantize_block_e4m3(x: np.ndarray) -> Tuple[np.ndarray, float]:
    """One block [n, d] -> (e4m3 values [n, d], qscale) following the reading
    in the module header; x ~= qscale * values."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.abs(x32).max()) if x32.size else np.float32(0)
    if amax == 0:
        return np.zeros(x32.shape), 1.0
    qscale = np.float32(amax / np.float32(E4M3_MAX))
    inv = np.float32(np.float32(E4M3_MAX) / amax)
    y = (x32 * inv).astype(np.float32)
    return round_e4m3(y), float(qscale)


def quantize_blocks_e4m3(x: np.ndarray, blk: int = 64) -> Tuple[np.ndarray, np.ndarray]:
    """Every blk-row block of x [s, d] -> (values [s, d], qscales [ceil(s/blk)])."""
    s = x.shape[0]
    nb = (s + blk - 1) // blk
    vals = np.zeros(x.shape, dtype=np.float64)
    scales = np.zeros(nb, dtype=np.float64)
    for j in range(nb):
        vals[j * blk:(j + 1) * blk], scales[j] = quantize_block_e4m3(x[j * blk:(j + 1) * blk])
    return vals, scales


def attention_unit_fp8(q: np.ndarray, k: np.ndarray, v: np.ndarray, lut_row: Iterable[int],
                       i: int, blkq: int, blkk: int, scale: float, causal: bool):
    """Attention of q block ``i`` over the listed kv blocks with fp8 Q and K
    (scores from the quantised blocks and their scales; V unchanged).
    Returns (O [rows, dv], LSE [rows])."""
    s_q, s_k = q.shape[0], k.shape[0]
    t = np.arange(i * blkq, min((i + 1) * blkq, s_q))
    cq, sq = quantize_block_e4m3(q[t])
    lut_row = [int(j) for j in lut_row]
    keys = row_keys(lut_row, blkk, s_k)
    parts = []
    for j in lut_row:
        kj = np.arange(j * blkk, min((j + 1) * blkk, s_k))
        ck, sk = quantize_block_e4m3(k[kj])
        parts.append(scale * sq * sk * (cq @ ck.T))
    scores = np.concatenate(parts, axis=1) if parts else np.zeros((len(t), 0))
    if causal:
        scores = np.where(keys[None, :] <= t[:, None], scores, -np.inf)
    return _softmax_attend(scores, v[keys])
