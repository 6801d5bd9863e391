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

// ---------------------------------------------------------------------------
// q-block pair union
// ---------------------------------------------------------------------------
//
// For the 128-row attention kernel: q blocks 2p and 2p + 1 of a (batch, head)
// share one 128-row tile, which visits the union of their LUT rows.  One warp
// per pair builds the union as a bitmask in shared memory (lane L owns the 32
// kv blocks 32 L .. 32 L + 31), so the output is ascending and duplicate-free
// whatever the input order, and emits every member j as
// j | (in row 2p) << 29 | (in row 2p + 1) << 30, -1 padded, with the count.
// Entries outside [0, nk) and counts outside [0, min(nk, lut_stride)] are
// skipped (clamped) and set FBM_DEVERR_LUT_RANGE.

namespace fbm {
namespace {

__global__ void __launch_bounds__(256) k_lut_pair_union(const PairUnionLaunch L) {
  __shared__ uint32_t masks[8][2][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int npq = (L.nq + 1) / 2;
  const int64_t unit = (int64_t)blockIdx.x * 8 + w;  // (bh, pair)
  if (unit >= L.bh * npq) return;
  const int64_t bh = unit / npq;
  const int p = (int)(unit - bh * npq);
  uint32_t *mA = masks[w][0], *mB = masks[w][1];
  mA[lane] = 0u;
  mB[lane] = 0u;
  __syncwarp();
  uint32_t bits = 0;
  const int lim = min(L.nk, L.lut_stride);
  for (int half = 0; half < 2; ++half) {
    const int i = 2 * p + half;
    if (i >= L.nq) break;
    const int64_t row = bh * L.nq + i;
    const int raw = L.cnt[row];
    if (raw < 0 || raw > lim) bits |= FBM_DEVERR_LUT_RANGE;
    const int n = min(max(raw, 0), lim);
    const int32_t *src = L.lut + row * L.lut_stride;
    uint32_t *m = half ? mB : mA;
    for (int t = lane; t < n; t += 32) {
      const int j = __ldg(src + t);
      if (j < 0 || j >= L.nk) {
        bits |= FBM_DEVERR_LUT_RANGE;
        continue;
      }
      atomicOr(m + (j >> 5), 1u << (j & 31));
    }
  }
  __syncwarp();
  const uint32_t a = mA[lane], b = mB[lane], u = a | b;
  const int mine = __popc(u);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int up = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += up;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int32_t *dst = L.out_lut + unit * L.out_stride;
  int pos = incl - mine;
  for (uint32_t rest = u; rest; rest &= rest - 1u) {
    const int bit = __ffs(rest) - 1;
    const int j = 32 * lane + bit;
    dst[pos++] = j | (int)(((a >> bit) & 1u) << 29) | (int)(((b >> bit) & 1u) << 30);
  }
  for (int t = total + lane; t < L.out_stride; t += 32) dst[t] = -1;
  if (lane == 0) L.out_cnt[unit] = total;
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (lane == 0 && bits) atomicOr(L.err, bits);
}

}  // namespace

cudaError_t launch_lut_pair_union(const PairUnionLaunch &L, cudaStream_t st) {
  const int64_t units = L.bh * ((L.nq + 1) / 2);
  k_lut_pair_union<<<(unsigned)((units + 7) / 8), 256, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace fbm
