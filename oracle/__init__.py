"""fp64 CPU oracle for LUT-driven block-sparse attention (test infrastructure).

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import it. The library
in ``fmha_block_map_gb300`` never calls it, and it never calls the library: the
two share no code. The one shared module is ``synth``, which only draws
inputs.

All arithmetic is float64 on inputs widened exactly from their fp16 / bf16 bit
patterns. Library primitives (numpy matmul, exp, argsort) are allowed as single
steps. There is no blocking, fusion or reordering beyond what the definitions
below state.

Sources (web pages; cited by title and section):

* "Sparge Attention (Composable Kernel)" README, ROCm/composable_kernel
  example/ck_tile/50_sparse_attn: the block-map pipeline "mean-pool -> cosine
  sim -> pooled QK -> top-k LUT", per-head topk / simthreshd1 / cdfthreshd,
  and the 'Not yet ported' list (causal mask in the pooled score, attention
  sink = kv-block column 0 forced on, sort-based top-k).
* "Incremental_FlashAttention updating_log.md", Stage 1 (the combine identity
  FA(A u B) = Combine(FA(A), FA(B)) with the lse_max trick, order invariance,
  the empty partial with LSE = -inf) and Stage 3 (an empty block list writes
  O = 0 and LSE = -inf).
* ROCm/aiter pull 6841 (sorted-sparse MHA with LSE): LSE is the natural-log
  logsumexp of the scores that were actually computed; an empty LUT row gives
  LSE = -inf.
* ROCm/aiter pull 4919 (sparse MLA decode): top-k token index lists resolved
  through a page table, a 576-wide K row (512 latent + 64 rotary) whose latent
  plane is V, split-KV partials merged by an LSE reduce.

Block map, as computed here (the pages only name the steps; where they leave a
step open, the plainest reading is taken):

0. optional K smoothing (README 'Not yet ported': pre-pool k -= km): every key
   row minus the mean key row of its (batch, KV head) sequence; steps 1-7 then
   use the smoothed keys (queries unchanged);
1. pool: qbar_i, kbar_j = mean of the rows of each 64-token block (a partial
   last block averages the rows it has);
2. self-similarity of a block X of n rows: the mean cosine over all ordered
   row pairs, self-pairs included, = ||sum_t x_t/||x_t|| ||^2 / n^2 (a zero row
   contributes a zero unit vector); a block is "similar" when sim > theta_h;
3. eligibility: non-causal -> all; causal -> j*BLKK <= (i+1)*BLKQ - 1;
4. pooled score S_ij = scale * qbar_i . kbar_j, = -inf where kv block j is not
   similar or (i, j) is not eligible; P_i = softmax_j(S_i);
5. selection among finite entries ordered by (P desc, j asc):
   topk mode takes K_i = min(ceil(fl32(topk_h * n_elig_i)), #finite) entries,
   cdf mode takes the shortest prefix whose cumulative P reaches cdfthreshd_h
   (crossing entry included; all finite entries when rounding keeps it short);
6. forced on (where eligible): every non-similar kv column; every column of a
   non-similar q row; column 0 when attention_sink;
7. LUT_i = ascending {j : selected or forced, and eligible}; count_i = |LUT_i|;
   the LUT row is padded with -1.

Parity status: every function is pinned by tests/test_oracle_pins.py against
closed forms, brute force on tiny inputs and textbook attention. What cannot be
pinned is agreement with the CK / SpargeAttn block map itself (no input/output
pair for it exists on the pages): the readings of steps 2-6 are readings.
"""
from .block_map import (  # noqa: F401
    pool_blocks,
    self_similarity,
    eligible_mask,
    topk_count,
    select_row,
    block_map_head,
    smooth_keys,
    sparge_block_map,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_values,
    round_e4m3,
    quantize_block_e4m3,
    quantize_blocks_e4m3,
    attention_unit_fp8,
)
from .attention import (  # noqa: F401
    row_keys,
    attention_unit,
    sparse_fmha,
    split_bounds,
    split_partials_unit,
    combine,
    attention_unit_pv_skip,
    shard_lut_row,
    context_parallel_unit,
    speculative_two_pass_unit,
    decode_rows,
    decode_attention,
    decode_partials,
)
