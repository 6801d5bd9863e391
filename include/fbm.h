/*
 * fbm.h - C ABI of libfbm: LUT-driven block-sparse attention forward on one
 * GB300 GPU (sm_103a).
 *
 * The method (web pages, cited by title and section):
 *  - "Sparge Attention (Composable Kernel)" README, intro and 'Status vs
 *    Upstream': a block-map pipeline (per-block mean-pool -> cosine
 *    similarity -> pooled QK -> top-k / cdfthreshd block selection -> LUT)
 *    followed by a sparse FMHA stage that visits only the selected K/V tiles;
 *    per-head topk / simthreshd1 / cdfthreshd; 'Not yet ported': causal mask in
 *    the pooled score, attention sink (kv-block column 0 forced on).
 *  - "Incremental_FlashAttention updating_log.md", Stage 1 (combine identity,
 *    lse_max trick, empty partial = identity) and Stage 3 (an empty block list
 *    writes O = 0 and LSE = -inf).
 *  - ROCm/aiter pull 6841: LSE export of the computed scores, -inf for an
 *    empty LUT row; the GQA mapping query head j -> KV head j / (hq / hk).
 *  - ROCm/aiter pull 4919: sparse MLA decode over per-query token index lists
 *    through a page table, split-KV partials and an LSE reduce; a caller
 *    provided output buffer.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument marked "device" is caller-owned device memory; the
 *    library allocates nothing per call and keeps no pointer after returning.
 *    "host" arrays are read before the call returns.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*, NULL =
 *    the legacy default stream) and runs asynchronously; outputs are valid
 *    once the stream reaches that point.  The score and selection kernels of
 *    the block map, the decode and the combine are programmatic dependent
 *    launches: each may start while the kernel before it on the stream
 *    finishes, but waits for it (griddepcontrol.wait) before reading any
 *    input or writing any output, so stream order holds for all memory.
 *  - Argument checks run on the host before any launch.  A failed check
 *    returns FBM_ERR_INVALID_ARG or FBM_ERR_UNSUPPORTED and launches nothing;
 *    fbm_last_error_message() then describes it (per thread).
 *  - A launch failure returns FBM_ERR_CUDA.
 *  - Conditions detected on the device (a LUT entry out of range, a bounded
 *    wait that expired) set bits of a device error word; fbm_get_error()
 *    synchronises the stream and reads (and clears) it.
 *  - Tensors are contiguous, row-major, with the shapes given below; base
 *    pointers must be 16-byte aligned.
 *  - Head layout is BHSD: Q/O [b, hq, s_q, d], K/V [b, hk, s_k, d].
 */
#ifndef FBM_H_
#define FBM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FBM_OK = 0,
  FBM_ERR_INVALID_ARG = 1, /* a null pointer, a bad size or an inconsistent argument */
  FBM_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels implement */
  FBM_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
  FBM_ERR_DEVICE = 4       /* fbm_get_error found device error bits set */
} fbm_status;

typedef enum { FBM_F16 = 0, FBM_BF16 = 1, FBM_F32 = 2 } fbm_dtype;

/* Bits of the device error word. */
#define FBM_DEVERR_LUT_RANGE 0x1u /* a LUT / index entry outside [0, n) or a count > n */
#define FBM_DEVERR_TIMEOUT 0x2u   /* a bounded wait on an mbarrier expired */
#define FBM_DEVERR_LUT_ORDER 0x4u /* a LUT entry not above the one before it (duplicate or descending) */

/* Largest number of query heads a call may pass per-head parameters for. */
#define FBM_MAX_HEADS 256

/* Library version, as major * 10000 + minor * 100 + patch. */
int fbm_version(void);

/* Description of the last failed argument check of the calling thread. */
const char *fbm_last_error_message(void);

/* Synchronises `stream`, then reads and clears the device error word into
 * *detail (FBM_DEVERR_* bits; may be NULL).  Returns FBM_ERR_DEVICE when any
 * bit was set, FBM_ERR_CUDA when the synchronisation failed, else FBM_OK. */
fbm_status fbm_get_error(void *stream, uint32_t *detail);

/*
 * Workspace (bytes) that sparge_block_map needs for the given shape: the
 * pooled mean of every Q and K block (fp32, kept as three bf16 terms in
 * 128-block tiles: 6 d bytes per block, rounded up to whole tiles), the
 * self-similarity (fp32) of every block, and the mean key row (fp32) of every
 * (batch, KV head) for K smoothing.
 */
size_t fbm_block_map_workspace_bytes(int b, int hq, int hk, int s, int d, int blkq,
                                     int blkk);

/* The same for the implemented block size (blkq = blkk = 64). */
size_t fbm_workspace_bytes(int b, int hq, int hk, int s, int d);

/*
 * sparge_block_map - block-map prediction ("Sparge Attention (Composable
 * Kernel)" README: mean-pool -> cosine sim -> pooled QK -> top-k LUT).
 *
 * For every (batch, query head h, q block i), with KV head g = h / (hq / hk):
 *   0. smooth_k != 0 (K smoothing; the README lists it, pre-pool k -= km, as
 *      'Not yet ported'): every key row of (batch, g) minus the mean key row
 *      km of its s rows; steps 1-7 use the smoothed keys, queries unchanged.
 *      The pooled scores of a q row move by one constant, so only the K
 *      self-similarities (step 2) can change the result;
 *   1. qbar_i, kbar_j = means of the rows of each block (a partial last block
 *      averages the rows it has);
 *   2. sim(X) = || sum_t x_t / ||x_t|| ||^2 / n^2 of every block; a block is
 *      similar when sim > simthreshd1[h] (K blocks of head g are compared with
 *      the threshold of query head h);
 *   3. eligible(i, j) = causal ? j * blkk <= (i + 1) * blkq - 1 : true;
 *   4. S_ij = scale * qbar_i . kbar_j, -inf where kv block j is not similar or
 *      (i, j) is not eligible; P_i = softmax_j S_i;
 *   5. entries ordered by P descending, lower j first on ties; topk mode keeps
 *      ceil(topk[h] * n_eligible_i) of them (product in fp32), cdf mode the
 *      shortest prefix whose mass reaches cdfthreshd[h] (crossing entry
 *      included; everything finite when the mass never reaches it);
 *   6. forced on where eligible: non-similar kv columns, every column of a
 *      non-similar q row, column 0 when attention_sink;
 *   7. lut[b][h][i][0 .. count) = the kept kv blocks in ascending order,
 *      lut[b][h][i][count .. nk) = -1, lut_count[b][h][i] = count.
 *
 * q: device [b, hq, s, d], k: device [b, hk, s, d], dtype FBM_F16 / FBM_BF16.
 * d in {64, 128}; blkq = blkk = 64; nk = ceil(s / 64) <= 1024; hq % hk == 0;
 * hq <= FBM_MAX_HEADS.
 * topk, cdfthreshd, simthreshd1: host float[hq]; exactly one of topk /
 *   cdfthreshd is non-NULL; topk and cdfthreshd values in (0, 1].
 * lut: device int32 [b, hq, nq, nk]; lut_count: device int32 [b, hq, nq].
 *   During the call the lut buffer also holds the fp32 pooled scores of step 4
 *   (the same size); it holds the LUT once the stream reaches the end of the
 *   call, and is unspecified if the call fails.
 * block_map: device uint8 [b, hq, nq, nk] (1 = kept) or NULL.
 * workspace: device, >= fbm_block_map_workspace_bytes(...) bytes, 16-byte
 *   aligned; its contents are scratch between calls.
 */
fbm_status sparge_block_map(const void *q, const void *k, int dtype, int b, int hq, int hk,
                            int s, int d, int blkq, int blkk, const float *topk,
                            const float *cdfthreshd, const float *simthreshd1, float scale,
                            int causal, int attention_sink, int smooth_k, int32_t *lut,
                            int32_t *lut_count, uint8_t *block_map, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * sparge_block_map_static - sparge_block_map for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot give the library a workspace, such as a runtime that plans
 * every device buffer before it starts and passes each operation only its
 * inputs and outputs, or a hot path that must never call cudaMalloc (which
 * can synchronise the device and take unbounded time).
 *
 * Same arguments, results and checks as sparge_block_map, without workspace
 * and workspace_bytes: the scratch lives in a static device array of
 * FBM_STATIC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  A shape whose scratch (fbm_block_map_workspace_bytes) is
 * larger returns FBM_ERR_UNSUPPORTED and launches nothing.  The first call on
 * a device looks the array's address up; under CUDA's lazy module loading
 * (the default) that lookup may be what loads the module and reserves the
 * array's device memory.  Make one warm-up call per device at start-up,
 * outside any stream capture and outside the hot path.
 * All calls share the array, so calls that overlap on the GPU race; nothing
 * in it needs to start at zero.  The library allocates nothing.
 */
#define FBM_STATIC_SCRATCH_BYTES (32u << 20)
fbm_status sparge_block_map_static(const void *q, const void *k, int dtype, int b, int hq, int hk,
                                   int s, int d, int blkq, int blkk, const float *topk,
                                   const float *cdfthreshd, const float *simthreshd1, float scale,
                                   int causal, int attention_sink, int smooth_k, int32_t *lut,
                                   int32_t *lut_count, uint8_t *block_map, void *stream);

/*
 * sparge_block_map_e4m3 - sparge_block_map that also writes the e4m3 codes of
 * Q and K from the same pass over them: the quantisation fused into the pool
 * kernel that the "Sparge Attention (Composable Kernel)" README lists under
 * 'Not yet ported' (it names int8; GB300's tensor cores take fp8).
 *
 * Same arguments, results and checks as sparge_block_map, plus:
 * q8: device uint8 [b, hq, s, 128], q_scale: device fp32 [b, hq, ceil(s / 64)];
 * k8: device uint8 [b, hk, s, 128], k_scale: device fp32 [b, hk, ceil(s / 64)].
 * The codes and scales are those of quantize_e4m3_blocks (bit for bit): per
 * 64-row block of the raw (unsmoothed) rows, amax = max |x| in fp32,
 * scale = amax / 448 and code = e4m3(x * (448 / amax)) (IEEE rounding, round
 * to nearest even, saturating; scale 1 for an all-zero block).  They feed
 * sparse_fmha_fwd_fp8.  d = 128 only (FBM_ERR_UNSUPPORTED otherwise); the code
 * buffers must be 16-byte aligned.  Caller-owned; the library allocates
 * nothing.
 */
fbm_status sparge_block_map_e4m3(const void *q, const void *k, int dtype, int b, int hq, int hk,
                                 int s, int d, int blkq, int blkk, const float *topk,
                                 const float *cdfthreshd, const float *simthreshd1, float scale,
                                 int causal, int attention_sink, int smooth_k, int32_t *lut,
                                 int32_t *lut_count, uint8_t *block_map, void *workspace,
                                 size_t workspace_bytes, uint8_t *q8, float *q_scale, uint8_t *k8,
                                 float *k_scale, void *stream);

/*
 * sparse_fmha_fwd - flash attention over the LUT-selected K/V tiles
 * ("Sparge Attention (Composable Kernel)" README: the sparse FMHA stage;
 * updating_log Stage 3 for the per-row-block loop over a block list).
 *
 * For each query row t of q block i (head h, KV head g = h / (hq / hk)), the
 * keys are the union of kv blocks lut[b][h][i][0 .. lut_count[b][h][i]); under
 * causal only the keys at index u <= t + key_offset (key_offset = 0 when
 * queries and keys start at the same position; s_k - s_q when the queries
 * are the last s_q positions of the keys' sequence, the causal dense pass of
 * the speculative two-pass recipe, "Incremental_FlashAttention
 * updating_log.md" Stage 5; -lo * 64 for a context-parallel rank whose keys
 * start at position lo * 64; ignored without causal, |key_offset| <= 2^30).
 * A row with no visible key is an empty row.  With s = scale * q_t . k_u,
 * O_t = sum_u e^(s_u - m) v_u / sum_u e^(s_u - m) and LSE_t = m + ln sum_u
 * e^(s_u - m) (natural log).  An empty key set gives O_t = 0, LSE_t = -inf.
 *
 * q: device [b, hq, s_q, d]; k: device [b, hk, s_k, d]; v: device [b, hk, s_k, dv];
 * dtype FBM_F16 / FBM_BF16; d = dv in {64, 128}; blkq = blkk = 64.
 * lut: device int32 [b, hq, nq, lut_stride] with nq = ceil(s_q / 64), entries in
 *   [0, ceil(s_k / 64)), strictly ascending; lut_count: device int32
 *   [b, hq, nq], in [0, min(nk, lut_stride)].  The kernel checks each entry's
 *   range (one outside is skipped and sets FBM_DEVERR_LUT_RANGE) and the count
 *   (one outside its range is clamped into it and sets FBM_DEVERR_LUT_RANGE).
 *   The order is the caller's contract and is not checked here (a duplicate
 *   entry would be counted twice): lut_validate checks it on request.
 *   lut == NULL (and lut_count == NULL) selects dense attention: every kv
 *   block (under causal, every block up to the one holding the q block's last
 *   visible key).
 * pv_threshold: +inf turns the PV skip off.  A finite value >= 0 (natural log
 *   units of the scaled scores) enables the per-Q-tile PV skip (README, 'Not
 *   yet ported': pv_threshold per-Q-tile skip): the listed kv blocks are
 *   visited in LUT order with an exact running max m per row, and a block
 *   whose scores lie below m - pv_threshold in every row of the q block
 *   (rows past s_q do not count) is left out of O's P.V sum while its
 *   probabilities stay in the denominator and in the LSE.  Whole rows only
 *   (num_splits == 1, out given); otherwise FBM_ERR_UNSUPPORTED.  NaN or a
 *   negative value: FBM_ERR_INVALID_ARG.
 * num_splits == 1: out = device [b, hq, s_q, dv] in dtype; lse = device fp32
 *   [b, hq, s_q] or NULL (return_lse off); o_partial / lse_partial unused.
 * num_splits == 1 with out == NULL (partial mode): the whole row's normalised
 *   O and its LSE go to o_partial = device fp32 [1, b, hq, s_q, dv] and
 *   lse_partial = device fp32 [1, b, hq, s_q] (empty row: 0 and -inf), one
 *   slot of a stack that attn_combine merges (context-parallel shards,
 *   see lut_shard; two passes over disjoint key sets).  Both pointers are
 *   required.
 * num_splits > 1 (split-KV): the LUT row of each q block is cut into
 *   num_splits contiguous chunks (the first n mod S chunks hold ceil(n/S)
 *   entries, the rest floor(n/S)); chunk s writes its normalised partial to
 *   o_partial = device fp32 [S, b, hq, s_q, dv] and its LSE to lse_partial =
 *   device fp32 [S, b, hq, s_q] (empty chunk: 0 and -inf); out / lse unused.
 *   attn_combine merges them.
 */
fbm_status sparse_fmha_fwd(const void *q, const void *k, const void *v, int dtype, int b,
                           int hq, int hk, int s_q, int s_k, int d, int dv, int blkq, int blkk,
                           const int32_t *lut, const int32_t *lut_count, int lut_stride,
                           int num_splits, float scale, int causal, int key_offset,
                           float pv_threshold, void *out, float *lse, float *o_partial,
                           float *lse_partial, void *stream);

/*
 * attn_combine - merge split-KV partials over disjoint key sets
 * (updating_log Stage 1, the lse_max trick): per row, m = max_s LSE_s,
 * w_s = e^(LSE_s - m), O = sum_s w_s O_s / sum_s w_s, LSE = m + ln sum_s w_s;
 * rows whose partials are all empty (LSE = -inf) give O = 0, LSE = -inf.
 *
 * o_part: device fp32 [num_splits, rows, dv]; lse_part: device fp32
 * [num_splits, rows]; out: device [rows, dv] in out_dtype (FBM_F16, FBM_BF16 or
 * FBM_F32); lse_out: device fp32 [rows] or NULL.  dv % 4 == 0, dv <= 1024,
 * 1 <= num_splits <= 64.
 */
fbm_status attn_combine(const float *o_part, const float *lse_part, int num_splits,
                        int64_t rows, int dv, int out_dtype, void *out, float *lse_out,
                        void *stream);

/*
 * quantize_e4m3_blocks - fp8 Q or K for sparse_fmha_fwd_fp8: one scale per
 * 64-row block ("Sparge Attention (Composable Kernel)" README, 'Not yet
 * ported': Q/K quantisation fused into the pool stage; ROCm/aiter pull 6841:
 * the bf16fp8 recipe).
 *
 * For every (head, 64-row block) of x: amax = max |x| (fp32), scales[block] =
 * amax / 448 and codes = e4m3(x * (448 / amax)) (fp32, round to nearest; e4m3
 * "fn": round to nearest even, saturating at +-448); an all-zero block gets
 * scale 1 and zero codes.  x ~= scale * code.
 *
 * x: device [bh, s, d] fp16 / bf16 (dtype); d == 128.  codes: device uint8
 * [bh, s, d]; scales: device fp32 [bh, ceil(s / 64)].  x and codes 16-byte
 * aligned; all buffers are the caller's.  A null pointer, a non-positive size,
 * another dtype or a misaligned buffer returns FBM_ERR_INVALID_ARG, d != 128
 * FBM_ERR_UNSUPPORTED, before any launch.  Asynchronous on `stream`.
 */
fbm_status quantize_e4m3_blocks(const void *x, int dtype, int64_t bh, int s, int d,
                                uint8_t *codes, float *scales, void *stream);

/*
 * sparse_fmha_fwd_fp8 - sparse_fmha_fwd with e4m3 Q and K: the scores of
 * q block i against kv block j are scale * q_scale[i] * k_scale[j] *
 * (Q codes . K codes^T) (tcgen05 kind::f8f6f4, fp32 accumulation); V, P, the
 * softmax, O and the LSE as in sparse_fmha_fwd (whole rows, num_splits = 1).
 *
 * q8 / q_scale: quantize_e4m3_blocks of Q [b * hq, s_q, 128]; k8 / k_scale:
 * of K [b * hk, s_k, 128].  v: device [b, hk, s_k, 128] in dtype; out: device
 * [b, hq, s_q, 128] in dtype; lse: device fp32 [b, hq, s_q] or NULL.  lut,
 * lut_count, lut_stride, causal as in sparse_fmha_fwd (lut == NULL: dense).
 * d = dv = 128.  All buffers are the caller's.  Argument errors return
 * FBM_ERR_INVALID_ARG (null pointers, sizes, dtype, hq % hk, scale,
 * alignment) or FBM_ERR_UNSUPPORTED (d, causal with s_q != s_k) before any
 * launch; device-detected LUT range errors and wait expiry set the error word
 * as in sparse_fmha_fwd.  Asynchronous on `stream`.
 */
fbm_status sparse_fmha_fwd_fp8(const uint8_t *q8, const float *q_scale, const uint8_t *k8,
                               const float *k_scale, const void *v, int dtype, int b, int hq,
                               int hk, int s_q, int s_k, int d, int dv, const int32_t *lut,
                               const int32_t *lut_count, int lut_stride, float scale, int causal,
                               void *out, float *lse, void *stream);

/*
 * lut_shard - the part of every LUT row inside one rank's kv-block range
 * [lo, hi), re-based to that rank's own K/V rows (context-parallel attention:
 * the LSE export exists so that partials over disjoint key sets can be merged
 * across ranks, ROCm/aiter pull 6841; the merge is updating_log Stage 1).
 *
 * For each row r < rows: the entries e of lut[r][0 .. min(lut_count[r],
 * lut_stride)) with lo <= e < hi, in their order, written as e - lo to
 * out_lut[r][0 .. out_count[r]); the rest of out_lut[r] (out_stride entries)
 * is -1.  A rank holding K/V rows [lo * 64, min(hi * 64, s_k)) then calls
 * sparse_fmha_fwd (partial mode) with out_lut / out_count and lut_stride =
 * out_stride, and attn_combine over the ranks' slots gives the attention of
 * the full LUT.
 *
 * lut: device int32 [rows, lut_stride]; lut_count: device int32 [rows];
 * out_lut: device int32 [rows, out_stride] with out_stride >= hi - lo;
 * out_count: device int32 [rows]; 0 <= lo < hi.  Invalid arguments return
 * FBM_ERR_INVALID_ARG before any launch.  A row that is not strictly ascending
 * can hold more in-range entries than out_stride: the excess is dropped and
 * FBM_DEVERR_LUT_RANGE is set.
 */
fbm_status lut_shard(const int32_t *lut, const int32_t *lut_count, int64_t rows, int lut_stride,
                     int lo, int hi, int32_t *out_lut, int32_t *out_count, int out_stride,
                     void *stream);

/*
 * lut_validate - check a LUT against the contract sparse_fmha_fwd relies on,
 * without changing it: per row a count and that many strictly ascending
 * kv-block indices (the sparse_block_table / sparse_num_blocks pair of
 * "Incremental_FlashAttention updating_log.md", 'Design decisions (locked)',
 * whose contract the caller guarantees and the kernels do not assert).
 *
 * For each row r < rows: lut_count[r] outside [0, min(nk, lut_stride)], or an
 * entry of lut[r][0 .. min(lut_count[r], ...)) outside [0, nk), sets
 * FBM_DEVERR_LUT_RANGE; an entry not above the entry before it (a duplicate or
 * a descending entry) sets FBM_DEVERR_LUT_ORDER.  Read the bits with
 * fbm_get_error.  The attention kernels check ranges and counts themselves
 * but not the order, which would cost the hot loop a dependent read per kv
 * block: call this where LUTs come from outside sparge_block_map, whose rows
 * are valid by construction.
 *
 * lut: device int32 [rows, lut_stride]; lut_count: device int32 [rows];
 * rows, lut_stride, nk > 0, else FBM_ERR_INVALID_ARG before any launch.
 * Asynchronous on `stream`.
 */
fbm_status lut_validate(const int32_t *lut, const int32_t *lut_count, int64_t rows,
                        int lut_stride, int nk, void *stream);

/*
 * lut_pair_union - the LUT rows of q blocks 2p and 2p + 1 merged into one
 * row, for sparse_fmha_fwd_pairs.  Not a step of the pages' method: it
 * re-lays the block table ("Sparge Attention (Composable Kernel)" README: the
 * per-q-block kv-block LUT) so that two q blocks can share 128-row tensor-core
 * tiles.
 *
 * For each (bh < bh, p < ceil(nq / 2)): the union of the entries of
 * lut[bh][2p][0 .. lut_count[bh][2p]) and lut[bh][2p + 1][...] (the second
 * row absent when 2p + 1 == nq), ascending and without duplicates, each
 * written as j | (j in row 2p) << 29 | (j in row 2p + 1) << 30 to
 * pair_lut[bh][p][0 .. pair_count[bh][p]), -1 padded.  Entries outside
 * [0, nk) are skipped and counts outside [0, min(nk, lut_stride)] clamped,
 * each setting FBM_DEVERR_LUT_RANGE.
 *
 * lut: device int32 [bh, nq, lut_stride]; lut_count: device int32 [bh, nq];
 * pair_lut: device int32 [bh, ceil(nq / 2), pair_stride], pair_stride >= nk;
 * pair_count: device int32 [bh, ceil(nq / 2)].  nk <= 1024.  Invalid
 * arguments return FBM_ERR_INVALID_ARG / FBM_ERR_UNSUPPORTED before any
 * launch.  Asynchronous on `stream`.
 */
fbm_status lut_pair_union(const int32_t *lut, const int32_t *lut_count, int64_t bh, int nq,
                          int lut_stride, int nk, int32_t *pair_lut, int32_t *pair_count,
                          int pair_stride, void *stream);

/*
 * sparse_fmha_fwd_pairs - sparse_fmha_fwd (whole rows, dtype output) on
 * 128-row tiles.  The result is that of sparse_fmha_fwd with the LUT the
 * pairs were built from: each query row attends over its own q block's LUT
 * row ("Sparge Attention (Composable Kernel)" README, the sparse FMHA stage),
 * with the same causal rule and key_offset, O and LSE conventions and empty
 * rows.  Rows 128 p .. 128 p + 127 (q blocks 2p and 2p + 1) share one tile
 * that visits the union of the two LUT rows (pair_lut from lut_pair_union;
 * each row masks the union members that are not its own), so every tensor-
 * core MMA spans 128 query rows: |A u B| 128-row tiles instead of |A| + |B|
 * 64-row ones.  pair_lut == NULL (with pair_count == NULL) is dense attention.
 *
 * q / k / v / out / lse / dtype / d / scale / causal / key_offset as in
 * sparse_fmha_fwd (d = dv in {64, 128}); pair_lut: device int32
 * [b, hq, ceil(nq / 2), pair_stride] and pair_count [b, hq, ceil(nq / 2)]
 * with entries as lut_pair_union writes them (a range error is skipped and
 * flagged as in sparse_fmha_fwd).  Argument errors return before any launch.
 * Asynchronous on `stream`.
 */
fbm_status sparse_fmha_fwd_pairs(const void *q, const void *k, const void *v, int dtype, int b,
                                 int hq, int hk, int s_q, int s_k, int d, int dv,
                                 const int32_t *pair_lut, const int32_t *pair_count,
                                 int pair_stride, float scale, int causal, int key_offset,
                                 void *out, float *lse, void *stream);

/*
 * sparse_decode_fwd - sparse decode over per-query token index lists through a
 * page table (ROCm/aiter pull 4919: sparse MLA decode with split-KV partials).
 *
 * Query c (one token, hq heads sharing one KV head) attends to the tokens
 * listed in indices[c][0 .. topk); token position p lives in cache row
 * page_table[c][p / page_size] * page_size + p % page_size; K = that row
 * (d values), V = its first dv values.  A negative index is a sentinel and is
 * skipped.  The list is cut into num_splits contiguous chunks (sizes as in
 * sparse_fmha_fwd); chunk s writes the normalised partial o_partial[s][c][h][:]
 * and its LSE lse_partial[s][c][h] (empty chunk: 0 and -inf).  attn_combine
 * over rows = n_q * hq merges them.
 *
 * q: device [n_q, hq, d] in dtype; kv_cache: device [n_pages, page_size, d];
 * dtype FBM_BF16 or FBM_F16; implemented shape: hq == 16, d == 576, dv == 512,
 * page_size == 64 (other shapes return FBM_ERR_UNSUPPORTED);
 * ceil(topk / num_splits) <= 16384;
 * page_table: device int32 [n_q, pages_per_query], entries in [0, n_pages);
 * indices: device int32 [n_q, topk], entries < pages_per_query * page_size;
 * o_partial: device fp32 [num_splits, n_q, hq, dv]; lse_partial: device fp32
 * [num_splits, n_q, hq]; 1 <= num_splits <= 64.
 */
fbm_status sparse_decode_fwd(const void *q, const void *kv_cache, int dtype, int n_q, int hq,
                             int d, int dv, int page_size, int64_t n_pages,
                             const int32_t *page_table, int pages_per_query,
                             const int32_t *indices, int topk, int num_splits, float scale,
                             float *o_partial, float *lse_partial, void *stream);

/* Diagnostic without a counterpart on the pages: launches one CTA that waits,
 * with the bounded mbarrier wait the tcgen05 kernels use, on a barrier that
 * nothing arrives on.  After limit_ns (0 < limit_ns <= 1e10) the wait gives up
 * and sets FBM_DEVERR_TIMEOUT in the device error word (read it with
 * fbm_get_error); the kernel then returns and the context stays usable.
 * Asynchronous on `stream`. */
fbm_status fbm_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* Which sparse-FMHA kernel sparse_fmha_fwd launches for these arguments:
 * 1 = the tcgen05 / TMA kernel (every supported shape: d = dv in {64, 128}),
 * 0 = none (the arguments would be rejected).  Host-only; launches nothing. */
int fbm_fmha_kernel_kind(int dtype, int d, int dv, int num_splits, int s_q, int s_k);

#ifdef __cplusplus
}
#endif

#endif /* FBM_H_ */
