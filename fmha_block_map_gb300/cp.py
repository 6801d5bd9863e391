"""Context-parallel sparse attention over kv-block ranges.

The LSE that ``sparse_fmha_fwd`` exports exists so that partial attentions
over disjoint key sets can be merged across ranks (ROCm/aiter pull 6841); the
merge is the Stage 1 combine of the Incremental_FlashAttention updating_log
(``attn_combine``).  Here the kv blocks of a sequence are cut into contiguous
ranges, one per rank (the first nk mod W ranks hold one block more).  Each
rank holds only the K/V rows of its range, shards every LUT row to it
(``lut_shard``, a kernel), computes its fp32 partial with ``sparse_fmha_fwd``
in partial mode, and the partials of all ranks, stacked in rank order, are
merged by ``attn_combine``.  Under causal attention a rank's keys start at
position lo * 64, so its partial runs with the causal key offset -lo * 64.

The exchange step: every rank owns a contiguous share of the output rows
(``row_owner_bounds``); an all-to-all sends each rank the other ranks'
partials of its own rows only (``scatter_partials_to_owners``), and each rank
combines just those (``context_parallel_attention``).  ``gather_partials``
(an all-gather of whole partials, every rank combining every row) is kept for
callers that want the full output on every rank.
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
                 scale: Optional[float] = None, causal: bool = False,
                 o_slot: Optional[torch.Tensor] = None,
                 lse_slot: Optional[torch.Tensor] = None, stream=None):
    """This rank's partial: q [b, hq, s_q, d] (all queries), k_shard /
    v_shard [b, hk, rows of the range, *], the full LUT.  Under causal (queries
    and the full key sequence start at position 0) the rank's local key u sits
    at position lo * 64 + u: key offset -lo * 64.  Writes and returns
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
    sparse_fmha_fwd(q, k_shard, v_shard, sub_lut, sub_cnt, scale=scale, causal=causal,
                    key_offset=-lo * BLK, o_partial=o_slot, lse_partial=lse_slot, partial=True,
                    stream=stream)
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


def row_owner_bounds(rows: int, world: int) -> List[Tuple[int, int]]:
    """The contiguous output rows [r0, r1) each rank owns after the exchange:
    the first rows mod world ranks own one row more."""
    if world < 1:
        raise ValueError("world must be >= 1")
    base, extra = divmod(rows, world)
    out, r0 = [], 0
    for r in range(world):
        r1 = r0 + base + (1 if r < extra else 0)
        out.append((r0, r1))
        r0 = r1
    return out


def scatter_partials_to_owners(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """The exchange step as a reduce-scatter: o_part [rows, dv] / lse_part
    [rows] (this rank's partial, rows flattened) are cut by row owner; an
    all-to-all hands each owner every rank's slice of its rows.  Returns
    (o_all [world, own rows, dv], lse_all [world, own rows]) in rank order,
    ready for attn_combine, and this rank's (r0, r1)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    rows, dv = o_part.shape
    bounds = row_owner_bounds(rows, world)
    sizes = [r1 - r0 for r0, r1 in bounds]
    r0, r1 = bounds[rank]
    own = r1 - r0
    o_all = torch.empty((world, own, dv), dtype=o_part.dtype, device=o_part.device)
    l_all = torch.empty((world, own), dtype=lse_part.dtype, device=lse_part.device)
    # send slice `peer` of my rows to rank `peer`; receive my rows from every rank
    dist.all_to_all_single(o_all.view(world * own, dv), o_part.contiguous(),
                           output_split_sizes=[own] * world, input_split_sizes=sizes, group=group)
    dist.all_to_all_single(l_all.view(world * own), lse_part.contiguous(),
                           output_split_sizes=[own] * world, input_split_sizes=sizes, group=group)
    return o_all, l_all, (r0, r1)


def context_parallel_attention(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor,
                               lut: torch.Tensor, lut_count: torch.Tensor, lo: int, hi: int, *,
                               scale: Optional[float] = None, causal: bool = False,
                               out_dtype=torch.float32, group=None, stream=None):
    """One rank's call: its partial, the reduce-scatter to row owners, the
    combine of the rows it owns.  Returns (out [own rows, dv] in out_dtype,
    lse [own rows], (r0, r1)): this rank's rows r0 .. r1 of the flattened
    [b * hq * s_q] output."""
    o, l = rank_partial(q, k_shard, v_shard, lut, lut_count, lo, hi, scale=scale, causal=causal,
                        stream=stream)
    dv = o.shape[-1]
    o_all, l_all, own = scatter_partials_to_owners(o.view(-1, dv), l.view(-1), group)
    out, lse = attn_combine(o_all, l_all, out_dtype=out_dtype, stream=stream)
    return out, lse, own


def speculative_two_pass(q: torch.Tensor, k_spec: torch.Tensor, v_spec: torch.Tensor,
                         k: torch.Tensor, v: torch.Tensor, missed_lut: torch.Tensor,
                         missed_count: torch.Tensor, *, scale: Optional[float] = None,
                         causal_spec: bool = True, out_dtype=None, stream=None):
    """The two-pass recipe of "Incremental_FlashAttention updating_log.md"
    Stage 5: a dense pass over the caller-gathered speculative keys k_spec /
    v_spec [b, hk, s_spec, *] (causal with the queries at their end: key
    offset s_spec - s_q), a sparse pass over the missed kv blocks of the full
    k / v listed in missed_lut / missed_count (fully historical blocks: no
    mask), and the LSE combine of the two.  Returns (out [b, hq, s_q, dv] in
    out_dtype (default q's), lse [b, hq, s_q])."""
    b, hq, s_q, _ = q.shape
    dv = v.shape[3]
    o_all = torch.empty((2, b, hq, s_q, dv), dtype=torch.float32, device=q.device)
    l_all = torch.empty((2, b, hq, s_q), dtype=torch.float32, device=q.device)
    sparse_fmha_fwd(q, k_spec, v_spec, None, None, scale=scale, causal=causal_spec,
                    key_offset=k_spec.shape[2] - s_q, o_partial=o_all[0], lse_partial=l_all[0],
                    partial=True, stream=stream)
    sparse_fmha_fwd(q, k, v, missed_lut, missed_count, scale=scale, o_partial=o_all[1],
                    lse_partial=l_all[1], partial=True, stream=stream)
    return attn_combine(o_all, l_all, out_dtype=q.dtype if out_dtype is None else out_dtype,
                        stream=stream)
