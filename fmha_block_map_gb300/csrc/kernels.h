// Internal launch interfaces between the C ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fbm.h"

namespace fbm {

struct HeadParams {
  float theta[FBM_MAX_HEADS];  // simthreshd1 per query head
  float sel[FBM_MAX_HEADS];    // topk or cdfthreshd per query head
};

// Pooled block means in the block-map workspace: each fp32 mean x is kept as
// the three bf16 terms of x = x0 + x1 + x2 (x0 = bf16(x), x1 = bf16(x - x0),
// x2 = bf16(x - x0 - x1)), laid out for the tensor-core product of the pooled
// scores.  Per (batch, head): ceil(nb / 128) tiles of 128 blocks; per tile
// d / 64 chunks of 64 values; per chunk the planes x0, x1, x2, each 128 rows
// (blocks) of 128 bytes in the 128-byte-swizzled K-major layout (16-byte piece
// c of row r at r * 128 + ((c ^ (r mod 8)) * 16)).  Rows past nb are never
// written.
constexpr int kPlaneRows = 128;
constexpr size_t kPlaneBytes = 128 * 128;
__host__ __device__ inline size_t plane_chunk_bytes() { return 3 * kPlaneBytes; }
__host__ __device__ inline size_t plane_tile_bytes(int d) { return (size_t)(d / 64) * plane_chunk_bytes(); }
__host__ __device__ inline size_t plane_head_bytes(int nb, int d) {
  return (size_t)((nb + kPlaneRows - 1) / kPlaneRows) * plane_tile_bytes(d);
}

struct SelectArgs {
  const uint8_t *qpl, *kpl;  // pooled means as split planes (layout above)
  const float *qsim, *ksim;
  int b, hq, hk, nq, nk, blkq, blkk;
  float scale;
  int causal, sink, mode_cdf;
  int32_t *lut, *cnt;
  uint8_t *bmap;
  uint32_t *err;  // device error word
};
cudaError_t launch_pooled_scores_tc(const SelectArgs &a, int d, cudaStream_t st);

struct BlockMapLaunch {
  const void *q, *k;
  int bf16, b, hq, hk, s, d, nq, nk;
  float scale;
  int causal, sink, mode_cdf, smooth_k;
  HeadParams hp;
  uint8_t *qpl, *kpl;                 // workspace carve-out: split planes,
  float *qsim, *ksim, *kmu;           // self-similarities, mean key rows
  uint8_t *q8, *k8;                   // e4m3 codes of Q and K, or null (d = 128)
  float *q_scale, *k_scale;           // one scale per 64-row block
  int32_t *lut, *cnt;
  uint8_t *bmap;
  uint32_t *err;  // device error word
};
cudaError_t launch_block_map(const BlockMapLaunch &L, cudaStream_t st);

struct FmhaLaunch {
  const void *q, *k, *v;
  int bf16, b, hq, hk, s_q, s_k, d, nq, nk;
  const int32_t *lut, *cnt;  // lut == nullptr: dense
  int lut_stride, num_splits, causal;
  int key_offset;      // causal: key index u visible to query row t when u <= t + key_offset
  float scale;
  float pv_threshold;  // +inf: no PV skip
  const float *q_scale, *k_scale;  // fp8 Q / K (q, k hold e4m3 codes) or nullptr
  void *out;
  float *lse, *o_part, *lse_part;
  uint32_t *err;
};
cudaError_t launch_fmha_tc(const FmhaLaunch &L, cudaStream_t st);
bool fmha_tc_supported(int d, int dv, int num_splits, int s_q, int s_k);

struct CombineLaunch {
  const float *o_part, *lse_part;
  int num_splits;
  int64_t rows;
  int dv, out_dtype;
  void *out;
  float *lse_out;
};
cudaError_t launch_combine(const CombineLaunch &L, cudaStream_t st);

struct QuantLaunch {
  const void *x;     // [bh, s, 128] fp16 / bf16
  int bf16, s, nb;   // nb = ceil(s / 64)
  int64_t units;     // bh * nb
  uint8_t *codes;    // [bh, s, 128] e4m3
  float *scales;     // [bh, nb]
};
cudaError_t launch_quant_e4m3(const QuantLaunch &L, cudaStream_t st);

struct LutShardLaunch {
  const int32_t *lut, *cnt;
  int64_t rows;
  int lut_stride, lo, hi, out_stride;
  int32_t *out_lut, *out_cnt;
  uint32_t *err;
};
cudaError_t launch_lut_shard(const LutShardLaunch &L, cudaStream_t st);

struct LutValidateLaunch {
  const int32_t *lut, *cnt;
  int64_t rows;
  int lut_stride, nk;
  uint32_t *err;
};
cudaError_t launch_lut_validate(const LutValidateLaunch &L, cudaStream_t st);

struct PairUnionLaunch {
  const int32_t *lut, *cnt;  // [bh, nq, lut_stride], [bh, nq]
  int64_t bh;
  int nq, lut_stride, nk, out_stride;
  int32_t *out_lut, *out_cnt;  // [bh, ceil(nq / 2), out_stride], [bh, ceil(nq / 2)]
  uint32_t *err;
};
cudaError_t launch_lut_pair_union(const PairUnionLaunch &L, cudaStream_t st);
// the 128-row (q-block pair) attention kernel: whole rows, dtype output
cudaError_t launch_fmha_pair(const FmhaLaunch &L, cudaStream_t st);

struct DecodeLaunch {
  const void *q, *cache;
  int bf16, n_q, hq, d, dv, page;
  int64_t n_pages;
  const int32_t *page_table;
  int pages_per_query;
  const int32_t *idx;
  int topk, num_splits;
  float scale;
  float *o_part, *lse_part;
  uint32_t *err;
};
cudaError_t launch_decode(const DecodeLaunch &L, cudaStream_t st);

}  // namespace fbm
