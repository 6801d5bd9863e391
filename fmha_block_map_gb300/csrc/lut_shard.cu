// Context-parallel LUT shard: the part of every LUT row that falls in one
// rank's contiguous kv-block range [lo, hi), re-based to the rank's own K/V
// rows (entry e becomes e - lo).  With the key set of a row split this way,
// the ranks' partial attentions recombine to the full row through the LSE
// combine (Incremental_FlashAttention updating_log, Stage 1; the LSE export
// exists for ring / context-parallel merging, ROCm/aiter pull 6841).
//
// One warp per row: the row is read in 32-entry chunks, a ballot marks the
// entries in range, and each lane writes its entry at the running count plus
// the popcount of the lower lanes' marks.  The order of the row is kept, no
// atomics take part, and the rest of the output row is padded with -1.
#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

__global__ void __launch_bounds__(256) k_lut_shard(const LutShardLaunch L) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= L.rows) return;
  const int32_t *src = L.lut + row * L.lut_stride;
  int32_t *dst = L.out_lut + row * L.out_stride;
  const int n = min(max(L.cnt[row], 0), L.lut_stride);
  int kept = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int c = c0 + lane;
    const int e = c < n ? src[c] : -1;
    const bool in = c < n && e >= L.lo && e < L.hi;
    const unsigned m = __ballot_sync(0xffffffffu, in);
    const int slot = kept + __popc(m & ((1u << lane) - 1u));
    // an entry past out_stride cannot occur when the row is strictly ascending;
    // for any other row it is dropped and flagged
    if (in) {
      if (slot < L.out_stride) dst[slot] = e - L.lo;
      else atomicOr(L.err, FBM_DEVERR_LUT_RANGE);
    }
    kept += __popc(m);
  }
  kept = min(kept, L.out_stride);
  for (int c = kept + lane; c < L.out_stride; c += 32) dst[c] = -1;
  if (lane == 0) L.out_cnt[row] = kept;
}

}  // namespace

cudaError_t launch_lut_shard(const LutShardLaunch &L, cudaStream_t st) {
  const int64_t blocks = (L.rows + 7) / 8;
  k_lut_shard<<<(unsigned)blocks, 256, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace fbm

// ---------------------------------------------------------------------------
// LUT validation
// ---------------------------------------------------------------------------
//
// The attention kernels trust the order of a LUT row (strictly ascending kv
// blocks, the contract of the sparse block table) and check only each entry's
// range and the row's count.  k_lut_validate checks all of it without touching
// the LUT: one warp per row reads the row in 32-entry chunks, compares every
// entry with the one before it (a shuffle inside the chunk, the previous
// chunk's last entry across chunks) and ORs FBM_DEVERR_LUT_RANGE (a count
// outside [0, min(nk, lut_stride)], an entry outside [0, nk)) and
// FBM_DEVERR_LUT_ORDER (an entry not above the one before it) into the device
// error word.

namespace fbm {
namespace {

__global__ void __launch_bounds__(256) k_lut_validate(const LutValidateLaunch L) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= L.rows) return;
  const int32_t *src = L.lut + row * L.lut_stride;
  const int raw = L.cnt[row];
  const int lim = min(L.nk, L.lut_stride);
  uint32_t bits = (raw < 0 || raw > lim) ? FBM_DEVERR_LUT_RANGE : 0u;
  const int n = min(max(raw, 0), lim);
  int last = INT32_MIN;  // the previous chunk's last entry
  for (int c0 = 0; c0 < n; c0 += 32) {
    const int c = c0 + lane;
    const int e = c < n ? __ldg(src + c) : INT32_MAX;
    int before = __shfl_up_sync(0xffffffffu, e, 1);
    if (lane == 0) before = last;
    if (c < n) {
      if (e < 0 || e >= L.nk) bits |= FBM_DEVERR_LUT_RANGE;
      if (c > 0 && e <= before) bits |= FBM_DEVERR_LUT_ORDER;
    }
    last = __shfl_sync(0xffffffffu, e, 31);
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits) atomicOr(L.err, bits);
}

}  // namespace

cudaError_t launch_lut_validate(const LutValidateLaunch &L, cudaStream_t st) {
  const int64_t blocks = (L.rows + 7) / 8;
  k_lut_validate<<<(unsigned)blocks, 256, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace fbm
