"""Context-parallel sparse attention over kv-block ranges.

The LSE that ``sparse_fmha_fwd`` exports exists so that partial attentions
over disjoint key sets can be merged across ranks (ROCm/aiter pull 6841); the
merge is the Stage 1 combine of the Incremental_FlashAttention updating_log
(``attn_combine``).  Here the kv blocks of a sequence are cut into contiguous
ranges, one per rank (the first nk mod W ranks hold one block more).  Each
rank holds only the K/V rows of its range, shards every LUT row to it
(``lut_shard``, a kernel), computes its fp32 partial with ``sparse_fmha_fwd``
in partial mode, and the partials of all ranks, stacked in rank order, are
merged by ``attn_combine``.  The one exchange step is an all-gather of the
partials (``gather_partials``, any torch.distributed backend).

Non-causal only: a rank's keys start at lo * 64, and the causal mask of the
attention kernel assumes keys and queries share position 0.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch

from . import attn_combine, lut_shard, sparse_fmha_fwd

BLK = 64


def kv_shard_bounds(nk: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous kv-block ranges [lo, hi) of ``world`` ranks over nk blocks:
    the first nk mod world ranges hold ceil(nk / world) blocks, the rest
    floor(nk / world).  Every range must be non-empty (world <= nk)."""
    if world < 1 or nk < world:
        raise ValueError(f"need 1 <= world ({world}) <= nk ({nk})")
    base, extra = divmod(nk, world)
    out, lo = [], 0
    for r in range(world):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def shard_rows(s_k: int, lo: int, hi: int) -> Tuple[int, int]:
    """The K/V rows [r0, r1) that the rank holding kv blocks [lo, hi) keeps."""
    return lo * BLK, min(hi * BLK, s_k)


def rank_partial(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor,
                 lut: torch.Tensor, lut_count: torch.Tensor, lo: int, hi: int, *,
                 scale: Optional[float] = None, o_slot: Optional[torch.Tensor] = None,
                 lse_slot: Optional[torch.Tensor] = None, stream=None):
    """This rank's partial: q [b, hq, s_q, d] (all queries), k_shard /
    v_shard [b, hk, rows of the range, *], the full LUT.  Writes and returns
    (o_slot [b, hq, s_q, dv] fp32, lse_slot [b, hq, s_q] fp32)."""
    rows = k_shard.shape[2]
    if v_shard.shape[2] != rows or (rows + BLK - 1) // BLK != hi - lo:
        raise ValueError(f"k_shard / v_shard must hold the rows of kv blocks [{lo}, {hi})")
    sub_lut, sub_cnt = lut_shard(lut, lut_count, lo, hi, stream=stream)
    b, hq, s_q, _ = q.shape
    dv = v_shard.shape[3]
    if o_slot is None:
        o_slot = torch.empty((b, hq, s_q, dv), dtype=torch.float32, device=q.device)
    if lse_slot is None:
        lse_slot = torch.empty((b, hq, s_q), dtype=torch.float32, device=q.device)
    sparse_fmha_fwd(q, k_shard, v_shard, sub_lut, sub_cnt, scale=scale, o_partial=o_slot,
                    lse_partial=lse_slot, partial=True, stream=stream)
    return o_slot, lse_slot


def gather_partials(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """The exchange step: every rank's (o_part, lse_part) stacked in rank
    order, [world, ...], on every rank (torch.distributed all_gather)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    o_all = torch.empty((world,) + tuple(o_part.shape), dtype=o_part.dtype, device=o_part.device)
    l_all = torch.empty((world,) + tuple(lse_part.shape), dtype=lse_part.dtype,
                        device=lse_part.device)
    dist.all_gather(list(o_all.unbind(0)), o_part.contiguous(), group=group)
    dist.all_gather(list(l_all.unbind(0)), lse_part.contiguous(), group=group)
    return o_all, l_all


def context_parallel_attention(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor,
                               lut: torch.Tensor, lut_count: torch.Tensor, lo: int, hi: int, *,
                               scale: Optional[float] = None, out_dtype=torch.float32,
                               group=None, stream=None):
    """One rank's call: its partial, the all-gather, the combine.  Returns
    (out [b, hq, s_q, dv] in out_dtype, lse [b, hq, s_q]) on every rank."""
    o, l = rank_partial(q, k_shard, v_shard, lut, lut_count, lo, hi, scale=scale,
                        stream=stream)
    o_all, l_all = gather_partials(o, l, group)
    return attn_combine(o_all, l_all, out_dtype=out_dtype, stream=stream)
