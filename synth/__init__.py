"""Seeded synthetic inputs for the block-sparse attention path.

This module only draws numbers and lays them out. It holds none of the
method's arithmetic (no pooling, no similarity, no scores, no selection, no
softmax), so both the fp64 oracle and the CUDA path may import it.

Recipes (each input is a pure function of its seed):

* Prefill workloads (``prefill``): per (batch, head, 64-token block) a centroid
  ``c ~ N(0, I_d) * cs``; every token of the block is ``c + eps`` with
  ``eps ~ N(0, sigma^2 I_d)``.  ``sigma = 0.3``; an exactly-25% subset of the
  blocks of each (batch, head, tensor), picked by a seeded permutation, is
  "diffuse" with ``sigma = 1.5``.  ``cs`` is 1.0, or drawn per head from
  ``U(cs_lo, cs_hi)``.  With ``drift > 0`` a random walk ``w_0 = 0,
  w_j = w_{j-1} + N(0, drift^2 I_d)`` over the block index is added to the
  centroids of Q, K and V.  Centroids are drawn in float64, the noise in
  float32; the float32 sum is cast to fp16 / bf16 by round-to-nearest-even.  Q, K and V use three
  independent child streams of one ``numpy.random.SeedSequence``.

  This follows the workloads that the Sparge Attention (Composable Kernel)
  README benchmarks (b=2 h=32 s=16384 d=128 fp16, 'Performance' section) and
  the small CPU-validation shape of its 'Usage' section (b=1 h=2 s=512).

* Sparse decode workload (``decode``): 64 single-token queries, 16 query heads
  sharing one KV head of width 576 (512 latent + 64 rotary), V = the first 512
  columns of the same cache row (the ROCm/aiter sparse-MLA decode pull request,
  where the latent plane serves as V).  The cache of 65536 pages x 64 rows is
  filled by a counter-based generator (``cache_rows``) so that any subset of
  rows can be regenerated bit-for-bit, on the CPU (numpy) or on a GPU
  (torch integer ops), without materialising 4.8 GB on the host.  Entries are
  an Irwin-Hall(4) approximation of N(0, 1) built from 16-bit uniforms:
  integer arithmetic, one float32 multiply and an RNE cast to bf16, which give
  identical bits on every device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BLK = 64

# ----------------------------------------------------------------------------
# fp16 / bf16 bit patterns (round to nearest even)
# ----------------------------------------------------------------------------


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> IEEE half bit pattern (uint16), round-to-nearest-even."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern (uint16), round-to-nearest-even.

    Inputs are finite (the generators never produce inf/nan)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen fp16 / bf16 bit patterns exactly to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f32_to_f16_bits(x)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# Prefill workloads
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    b: int
    hq: int
    hk: int
    s: int
    d: int
    dtype: str  # "f16" | "bf16"
    seed: int
    topk: Optional[float] = None
    cdfthreshd: Optional[float] = None
    simthreshd1: float = 0.001
    causal: bool = False
    attention_sink: bool = False
    return_lse: bool = False
    cs: float = 1.0
    cs_range: Optional[tuple] = None  # per-head centroid scale ~ U(lo, hi)
    sigma: float = 0.3
    sigma_diffuse: float = 1.5
    diffuse_frac: float = 0.25
    drift: float = 0.0
    antithetic_diffuse: bool = False  # diffuse blocks built from +/- row pairs
    key_offset: float = 0.0  # std of one offset vector shared by all keys of a (batch, head)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def nq(self) -> int:
        return (self.s + BLK - 1) // BLK

    def replace(self, **kw) -> "PrefillConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  C1: tiny fp16 non-causal; C2: bf16 cdf mode; C3: the
# headline shape (topk swept by the caller); C4: causal GQA + sink + LSE.
C1 = PrefillConfig("tiny_b1h2s512d64_f16", 1, 2, 2, 512, 64, "f16", 1001, topk=0.5)
C2 = PrefillConfig("cdf_b1h8s4096d128_bf16", 1, 8, 8, 4096, 128, "bf16", 1002,
                   cdfthreshd=0.9, cs_range=(0.5, 2.0))
C3 = PrefillConfig("headline_b2h32s16384d128_f16", 2, 32, 32, 16384, 128, "f16", 1003,
                   topk=0.4)
C4 = PrefillConfig("causal_gqa_b1hq32hk8s32768d128_bf16", 1, 32, 8, 32768, 128, "bf16",
                   1004, topk=0.2, causal=True, attention_sink=True, return_lse=True,
                   drift=0.1)
C3_TOPKS = (0.1, 0.2, 0.4, 0.6, 1.0)
PREFILL_CONFIGS = {"C1": C1, "C2": C2, "C3": C3, "C4": C4}


def _tensor_f32(rng: np.random.Generator, b: int, h: int, s: int, d: int,
                cfg: PrefillConfig, cs_per_head: np.ndarray) -> np.ndarray:
    """One [b, h, s, d] float32 tensor following the centroid-plus-noise recipe."""
    nb = (s + BLK - 1) // BLK
    out = np.empty((b, h, nb * BLK, d), dtype=np.float32)
    n_diffuse = int(round(cfg.diffuse_frac * nb))
    for bi in range(b):
        for hi in range(h):
            cent = rng.standard_normal((nb, d)) * cs_per_head[hi]
            if cfg.drift > 0.0:
                steps = rng.standard_normal((nb, d)) * cfg.drift
                steps[0] = 0.0
                cent = cent + np.cumsum(steps, axis=0)
            perm = rng.permutation(nb)
            sig = np.full((nb, 1, 1), cfg.sigma)
            sig[perm[:n_diffuse]] = cfg.sigma_diffuse
            noise = rng.standard_normal((nb, BLK, d), dtype=np.float32)
            if cfg.antithetic_diffuse:
                # diffuse blocks: rows come in (+x, -x) pairs around zero, so the
                # normalised rows of the block sum to exactly zero
                for blk in perm[:n_diffuse]:
                    half = noise[blk, : BLK // 2].copy()
                    noise[blk, 0::2] = half
                    noise[blk, 1::2] = -half
            tok = noise * sig.astype(np.float32)
            if cfg.antithetic_diffuse:
                keep = np.ones((nb, 1, 1), dtype=np.float32)
                keep[perm[:n_diffuse]] = 0.0
                tok = tok + (cent[:, None, :] * keep).astype(np.float32)
            else:
                tok = tok + cent[:, None, :].astype(np.float32)
            out[bi, hi] = tok.reshape(nb * BLK, d)
    return out[:, :, :s]


def prefill(cfg: PrefillConfig) -> dict:
    """Q, K, V bit patterns (uint16, [b,h,s,d] contiguous) for a prefill config."""
    ss = np.random.SeedSequence(cfg.seed)
    s_q, s_k, s_v, s_cs, s_off = ss.spawn(5)
    rng_cs = np.random.default_rng(s_cs)
    if cfg.cs_range is not None:
        cs_q = rng_cs.uniform(cfg.cs_range[0], cfg.cs_range[1], size=cfg.hq)
        # a KV head takes the scale of the first query head that reads it
        ratio = cfg.hq // cfg.hk
        cs_k = cs_q[::ratio].copy()
    else:
        cs_q = np.full(cfg.hq, cfg.cs)
        cs_k = np.full(cfg.hk, cfg.cs)
    q = _tensor_f32(np.random.default_rng(s_q), cfg.b, cfg.hq, cfg.s, cfg.d, cfg, cs_q)
    k = _tensor_f32(np.random.default_rng(s_k), cfg.b, cfg.hk, cfg.s, cfg.d, cfg, cs_k)
    v = _tensor_f32(np.random.default_rng(s_v), cfg.b, cfg.hk, cfg.s, cfg.d, cfg, cs_k)
    if cfg.key_offset > 0.0:
        # a channel bias common to every key of a head (the structure K
        # smoothing removes), drawn from its own stream so the rest is unchanged
        off = np.random.default_rng(s_off).standard_normal((cfg.b, cfg.hk, 1, cfg.d))
        k = k + (off * cfg.key_offset).astype(np.float32)
    return {
        "q": to_bits(q, cfg.dtype),
        "k": to_bits(k, cfg.dtype),
        "v": to_bits(v, cfg.dtype),
        "dtype": cfg.dtype,
    }


def per_head(cfg: PrefillConfig, value: Optional[float]) -> Optional[np.ndarray]:
    """A per-query-head float32 hyperparameter array (or None)."""
    if value is None:
        return None
    return np.full(cfg.hq, value, dtype=np.float32)


def sample_qblocks(cfg: PrefillConfig, per_bh: int, seed: int = 7) -> list:
    """A seeded sample of (b, h, q-block) units, always holding the first and
    last q-block of every (b, h)."""
    rng = np.random.default_rng(seed)
    units = []
    nq = cfg.nq
    for bi in range(cfg.b):
        for hi in range(cfg.hq):
            pick = {0, nq - 1}
            if nq > 2 and per_bh > 2:
                extra = rng.choice(np.arange(1, nq - 1), size=min(per_bh - 2, nq - 2),
                                   replace=False)
                pick.update(int(e) for e in extra)
            units.extend((bi, hi, i) for i in sorted(pick))
    return units


# ----------------------------------------------------------------------------
# Decode workload (counter-based cache)
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str = "mla_decode_c64h16d576dv512_bf16"
    n_queries: int = 64
    hq: int = 16
    d: int = 576
    dv: int = 512
    page: int = 64
    pages_per_query: int = 1024  # 65536 tokens per query
    topk: int = 2048
    seed: int = 1005
    dtype: str = "bf16"
    # softmax scale giving a median effective token count of 15 on this seed;
    # written by ``python -m oracle.calibrate_decode`` into
    # tests/golden/decode_sm_scale.json (a test checks the two agree)
    sm_scale: float = 0.12705914676189423

    @property
    def n_pages(self) -> int:
        return self.n_queries * self.pages_per_query

    @property
    def tokens_per_query(self) -> int:
        return self.pages_per_query * self.page

    def replace(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


C5 = DecodeConfig()

_M32 = 0xFFFFFFFF
# odd multipliers below 2**31 keep every product inside int64 on all backends
_HASH_MUL1 = 0x2C1B3C6D
_HASH_MUL2 = 0x297A2D39
_IH_MEAN = 2 * 65535
_IH_INV_STD = np.float32(1.0 / math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))


def _mix32(x, xp):
    """A 32-bit integer finaliser (xor-shift / multiply rounds) on int64 arrays
    holding values in [0, 2**32)."""
    x = x ^ (x >> 16)
    x = (x * _HASH_MUL1) & _M32
    x = x ^ (x >> 15)
    x = (x * _HASH_MUL2) & _M32
    x = x ^ (x >> 16)
    return x


def _irwin_hall_f32(counter, seed: int, xp):
    """N(0,1)-like float32 values from 64-bit counters (int64 arrays)."""
    key = (seed * 0x9E3779B1) & _M32
    lo = counter & _M32
    hi = (counter >> 32) & _M32
    h1 = _mix32(lo ^ key, xp)
    h1 = _mix32(h1 ^ hi, xp)
    h2 = _mix32(h1 ^ 0x5BD1E995, xp)
    u = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16) - _IH_MEAN
    return u, _IH_INV_STD


def cache_rows(cfg: DecodeConfig, rows: np.ndarray) -> np.ndarray:
    """bf16 bits [len(rows), d] of the given physical cache rows (numpy)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(cfg.d, dtype=np.int64)
    counter = rows[:, None] * cfg.d + cols[None, :]
    u, inv = _irwin_hall_f32(counter, cfg.seed * 2 + 1, np)
    x = u.astype(np.float32) * inv
    return f32_to_bf16_bits(x)


def cache_rows_torch(cfg: DecodeConfig, row_begin: int, row_end: int, device):
    """The same rows as ``cache_rows(cfg, arange(row_begin, row_end))``, built
    with torch integer ops on ``device``; returns a bf16 tensor [n, d]."""
    import torch

    rows = torch.arange(row_begin, row_end, dtype=torch.int64, device=device)
    cols = torch.arange(cfg.d, dtype=torch.int64, device=device)
    counter = rows[:, None] * cfg.d + cols[None, :]
    u, inv = _irwin_hall_f32(counter, cfg.seed * 2 + 1, torch)
    x = u.to(torch.float32) * float(inv)
    return x.to(torch.bfloat16)


def decode(cfg: DecodeConfig) -> dict:
    """Queries, page table and per-query index lists for the decode workload.

    The cache itself is not materialised here: see ``cache_rows``."""
    ss = np.random.SeedSequence(cfg.seed)
    s_q, s_pt, s_idx = ss.spawn(3)
    q = np.random.default_rng(s_q).standard_normal((cfg.n_queries, cfg.hq, cfg.d),
                                                   dtype=np.float32)
    perm = np.random.default_rng(s_pt).permutation(cfg.n_pages).astype(np.int32)
    page_table = perm.reshape(cfg.n_queries, cfg.pages_per_query)
    rng = np.random.default_rng(s_idx)
    idx = np.empty((cfg.n_queries, cfg.topk), dtype=np.int32)
    for c in range(cfg.n_queries):
        pos = rng.choice(cfg.tokens_per_query, size=cfg.topk, replace=False)
        idx[c] = np.sort(pos).astype(np.int32)
    return {"q": f32_to_bf16_bits(q), "page_table": page_table, "idx": idx,
            "dtype": "bf16"}
