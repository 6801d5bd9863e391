// Block-map prediction kernels ("Sparge Attention (Composable Kernel)" README:
// mean-pool -> cosine sim -> pooled QK -> top-k / cdfthreshd LUT).
//
//  k_pool_sim     one warp per 64-token block of Q or K: each lane streams 32
//                 bytes of a row per step (128-bit loads, 16 in flight per
//                 lane), row norms by a 3-level shuffle, fp32 row sums (the
//                 pooled mean, two interleaved partial sums per element) and the
//                 sum of unit rows (self-similarity = ||sum u||^2 / n^2).
//                 HBM-bound: it reads Q and K once and writes, per block, the
//                 mean as three bf16 split planes (the operands of the pooled
//                 scores' tensor-core product, in their shared-memory layout)
//                 and one float.
//  k_key_mean     K smoothing only: one CTA per (batch, KV head) forms the mean
//                 key row from the block means of the first pooling pass (fixed
//                 summation order, so the result is deterministic); a second
//                 pooling pass over K then subtracts it from every key row
//                 before the norms and sums.
//  pooled scores  scale * qbar . kbar on tcgen05 from the split planes
//                 (pooled_scores_tc.cu), written as fp32 into the caller's LUT
//                 buffer, which has exactly the size of the score matrix.
//  k_select       one warp per q block: loads its score row, then the pooled
//                 softmax, a radix (bitwise) threshold search for top-k / cdf,
//                 and ballot-scan emission of the ascending LUT row over the
//                 scores it has read.  No atomics take part in slot assignment.
//                 Apart from the product (which keeps every SM's FMA pipe busy)
//                 the selection is a chain of warp reductions; a kernel of its
//                 own runs it at full occupancy.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {

// ---------------------------------------------------------------------------
// k_pool_sim
// ---------------------------------------------------------------------------

struct PoolSide {
  const uint16_t *x;  // [bh, s, D] bit patterns
  uint8_t *planes;    // pooled means as split planes (kernels.h)
  float *sim;         // [bh * nb]
  int s;              // rows per (batch, head)
  int nb;             // blocks per (batch, head)
  int nunits;         // bh * nb
  const float *mu;    // [bh, D] row subtracted before pooling (SMOOTH only)
};

// x = x0 + x1 + x2 in bf16, each difference exact in fp32: the three terms
// carry the 24 significand bits of a normal fp32 value (the three-term bf16
// scheme of Henry, Tang and Heinecke, "Leveraging the bfloat16 Artificial
// Intelligence Datatype For Higher-Precision Computations", ARITH 2019)
FBM_DEVICE void split3(float x, uint32_t &h0, uint32_t &h1, uint32_t &h2) {
  const __nv_bfloat16 b0 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(b0);
  const __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b1);
  h0 = __bfloat16_as_ushort(b0);
  h1 = __bfloat16_as_ushort(b1);
  h2 = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

FBM_DEVICE float plane_value(const uint8_t *p) {
  return __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(p) << 16);
}

// Persistent: one CTA per SM, 8 consumer warps and one producer warp.  The
// rows of a 64-token block are contiguous in memory, so one bulk copy brings
// a whole block into a stage of a shared-memory ring (kPoolStageBytes of
// stages, kept full by the producer); consumer warp w reduces the CTA's
// blocks k = w, w + 8, ... from shared memory.
constexpr int kPoolConsumers = 8;
constexpr int kPoolThreads = 32 * (kPoolConsumers + 1);
constexpr int kPoolRingBytes = 192 * 1024;
constexpr uint64_t kPoolWaitNs = 2000000000ull;

template <int D>
struct PoolRing {
  static constexpr int kBlockBytes = kBlk * D * 2;  // one 64-row block of 16-bit values
  static constexpr int kStages = kPoolRingBytes / kBlockBytes;
  static constexpr int kBarOff = kPoolRingBytes;   // full[kStages], empty[kStages]
  static constexpr int kFlagOff = kBarOff + 16 * kStages;
  static constexpr int kSmem = kFlagOff + 16 + 128;  // + alignment slack
};

template <class E, int D, bool SMOOTH>
__global__ void __launch_bounds__(kPoolThreads, 1) k_pool_sim(PoolSide qs, PoolSide ks, uint32_t *err) {
  using R = PoolRing<D>;
  // a lane owns 16 elements of a row: 8 at sub * 8 and 8 at D / 2 + sub * 8,
  // so the 8 lanes of a quarter warp read 128 contiguous bytes of shared
  // memory; a row spans LPR lanes and one warp-wide step covers RPI rows
  constexpr int LPR = D / 16;
  constexpr int RPI = 32 / LPR;
  constexpr int STEPS = kBlk / RPI;
  constexpr int UNR = 4;  // shared-memory loads in flight per lane and step group
  extern __shared__ uint8_t pool_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(pool_smem_raw) + 127) &
                                              ~uintptr_t(127));
  const uint32_t sbase = smem_u32(smem);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + R::kFlagOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = qs.nunits + ks.nunits;
  auto full = [&](int st) { return sbase + R::kBarOff + 8 * st; };
  auto empty = [&](int st) { return sbase + R::kBarOff + 8 * (R::kStages + st); };
  if (threadIdx.x == 0) {
    for (int st = 0; st < R::kStages; ++st) {
      tc::mbar_init(full(st), 1);
      tc::mbar_init(empty(st), 1);
    }
    tc::fence_mbar_init();
    *abort_flag = 0;
  }
  __syncthreads();

  if (warp == kPoolConsumers) {
    // producer: one elected thread issues the bulk copies in order
    if (lane == 0) {
      int k = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x, ++k) {
        const int st = k % R::kStages;
        if (k >= R::kStages &&
            !tc::mbar_wait(empty(st), ((k / R::kStages) - 1) & 1, abort_flag, kPoolWaitNs)) {
          set_error(err, FBM_DEVERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const PoolSide &side = u < qs.nunits ? qs : ks;
        const int unit = u < qs.nunits ? u : u - qs.nunits;
        const int bh = unit / side.nb, j = unit - bh * side.nb;
        const int n = min(kBlk, side.s - j * kBlk);
        const uint32_t bytes = (uint32_t)n * D * 2;
        tc::mbar_arrive_tx(full(st), bytes);
        tc::bulk_load(sbase + st * R::kBlockBytes, side.x + ((size_t)bh * side.s + (size_t)j * kBlk) * D,
                      bytes, full(st));
      }
      // every copy this CTA issued has landed before it exits (bounded)
      for (int kk = max(0, k - R::kStages); kk < k; ++kk)
        tc::mbar_wait_for(full(kk % R::kStages), (kk / R::kStages) & 1, kPoolWaitNs);
    }
    return;
  }

  // consumers
  const int sub = lane % LPR;
  const int rgrp = lane / LPR;
  int k = warp;
  for (int u = blockIdx.x + warp * gridDim.x; u < total; u += kPoolConsumers * gridDim.x,
           k += kPoolConsumers) {
    const int st = k % R::kStages;
    if (!tc::mbar_wait(full(st), (k / R::kStages) & 1, abort_flag, kPoolWaitNs)) {
      set_error(err, FBM_DEVERR_TIMEOUT);
      *abort_flag = 1;
      break;
    }
    const PoolSide &side = u < qs.nunits ? qs : ks;
    const int unit = u < qs.nunits ? u : u - qs.nunits;
    const int bh = unit / side.nb;
    const int j = unit - bh * side.nb;
    const int n = min(kBlk, side.s - j * kBlk);
    const uint8_t *blk = smem + st * R::kBlockBytes;
    float mu[16];
    if constexpr (SMOOTH) {
      const float4 *m0 = reinterpret_cast<const float4 *>(side.mu + (size_t)bh * D + sub * 8);
      const float4 *m1 = reinterpret_cast<const float4 *>(side.mu + (size_t)bh * D + D / 2 + sub * 8);
      const float4 a0 = m0[0], a1 = m0[1], b0 = m1[0], b1 = m1[1];
      const float mv[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                            b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 16; ++e) mu[e] = mv[e];
    }

    // two interleaved partial sums per element keep the fp32 sums short
    float msum[2][16], usum[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) msum[0][e] = msum[1][e] = usum[e] = 0.f;
#pragma unroll
    for (int s0 = 0; s0 < STEPS; s0 += UNR) {
      uint4 raw[UNR][2];
#pragma unroll
      for (int uu = 0; uu < UNR; ++uu) {
        const int r = (s0 + uu) * RPI + rgrp;
        if (r < n) {  // rows past a partial block's end hold stale data
          const uint8_t *row = blk + r * (2 * D);
          raw[uu][0] = *reinterpret_cast<const uint4 *>(row + sub * 16);
          raw[uu][1] = *reinterpret_cast<const uint4 *>(row + D + sub * 16);
        } else {
          raw[uu][0] = raw[uu][1] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int uu = 0; uu < UNR; ++uu) {
        float x[16];
        const uint32_t w[8] = {raw[uu][0].x, raw[uu][0].y, raw[uu][0].z, raw[uu][0].w,
                               raw[uu][1].x, raw[uu][1].y, raw[uu][1].z, raw[uu][1].w};
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const float2 f = E::to_f2(w[p]);
          x[2 * p] = f.x;
          x[2 * p + 1] = f.y;
        }
        if constexpr (SMOOTH) {
          // rows past the end stay zero: they add nothing to either sum
          const int r = (s0 + uu) * RPI + rgrp;
          if (r < n) {
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] -= mu[e];
          }
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          usum[e] = fmaf(x[e], inv, usum[e]);
          msum[uu & 1][e] += x[e];
        }
      }
    }
    // the stage is free once every lane has read it
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty(st));

    float tot[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) tot[e] = msum[0][e] + msum[1][e];
#pragma unroll
    for (int o = 16; o >= LPR; o >>= 1) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        tot[e] += __shfl_xor_sync(0xffffffffu, tot[e], o);
        usum[e] += __shfl_xor_sync(0xffffffffu, usum[e], o);
      }
    }
    float su = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) su = fmaf(usum[e], usum[e], su);
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
    {
      // the mean, split into three bf16 planes.  Every lane holds the sums of
      // its sub's 16 values (pieces sub and D / 16 + sub of the block's row);
      // row group rgrp splits 16 / RPI of them, so the RPI lanes of a sub
      // fill 16-byte pieces of each plane together
      const float fn = (float)n;
      const int t = j / kPlaneRows, rr = j % kPlaneRows;
      uint8_t *tile = side.planes + (size_t)bh * plane_head_bytes(side.nb, D) +
                      (size_t)t * plane_tile_bytes(D);
      constexpr int VPL = 16 / RPI;  // values per lane: 4 (d = 128) or 2 (d = 64)
      const int e0 = rgrp * VPL;     // first of this lane's values within the 16
      const int gp = (e0 < 8 ? 0 : D / 16) + sub;
      const int c = gp >> 3, c8 = gp & 7;  // 64-value chunk, piece within it
      float val[VPL];
#pragma unroll
      for (int e = 0; e < VPL; ++e) val[e] = 0.f;
#pragma unroll
      for (int q = 0; q < 16; q += VPL)  // constant indices into tot[]
        if (q == e0) {
#pragma unroll
          for (int e = 0; e < VPL; ++e) val[e] = tot[q + e];
        }
      uint32_t w[3][VPL / 2];
#pragma unroll
      for (int e = 0; e < VPL / 2; ++e) {
        uint32_t a0, a1, a2, b0, b1, b2;
        split3(val[2 * e] / fn, a0, a1, a2);
        split3(val[2 * e + 1] / fn, b0, b1, b2);
        w[0][e] = a0 | (b0 << 16);
        w[1][e] = a1 | (b1 << 16);
        w[2][e] = a2 | (b2 << 16);
      }
      uint8_t *dst = tile + c * plane_chunk_bytes() + rr * 128 + ((c8 ^ (rr & 7)) << 4) + (e0 & 7) * 2;
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        if constexpr (VPL == 4)
          *reinterpret_cast<uint2 *>(dst + p * kPlaneBytes) = make_uint2(w[p][0], w[p][1]);
        else
          *reinterpret_cast<uint32_t *>(dst + p * kPlaneBytes) = w[p][0];
      }
      if (lane == 0) side.sim[unit] = su / (fn * fn);
    }
  }
}

// ---------------------------------------------------------------------------
// k_key_mean
// ---------------------------------------------------------------------------

// mean key row of every (batch, KV head): sum_j n_j * kbar_j / s over the K
// blocks, n_j the rows of block j, kbar_j = x0 + x1 + x2 read back from the
// split planes.  256 threads = (256 / D) groups of D; group g sums the blocks
// j = g mod (256 / D), then thread g = 0 adds the groups in order.
template <int D>
__global__ void __launch_bounds__(256) k_key_mean(const uint8_t *__restrict__ kpl,
                                                  float *__restrict__ mu, int s, int nk) {
  constexpr int G = 256 / D;
  __shared__ float part[G][D];
  const int e = threadIdx.x % D, g = threadIdx.x / D;
  const uint8_t *head = kpl + (size_t)blockIdx.x * plane_head_bytes(nk, D);
  const int c = e >> 6, c8 = (e & 63) >> 3, w = e & 7;
  float acc = 0.f;
#pragma unroll 4
  for (int j = g; j < nk; j += G) {
    const int t = j / kPlaneRows, rr = j % kPlaneRows;
    const uint8_t *p = head + (size_t)t * plane_tile_bytes(D) + c * plane_chunk_bytes() +
                       rr * 128 + ((c8 ^ (rr & 7)) << 4) + w * 2;
    const float x = (plane_value(p) + plane_value(p + kPlaneBytes)) + plane_value(p + 2 * kPlaneBytes);
    acc = fmaf((float)min(kBlk, s - j * kBlk), x, acc);
  }
  part[g][e] = acc;
  __syncthreads();
  if (g == 0) {
    float tot = part[0][e];
#pragma unroll
    for (int i = 1; i < G; ++i) tot += part[i][e];
    mu[(size_t)blockIdx.x * D + e] = tot / (float)s;
  }
}

// ---------------------------------------------------------------------------
// k_select
// ---------------------------------------------------------------------------

FBM_DEVICE uint32_t order_key(float f) {
  // order-preserving map of a finite float onto uint32 (finite values > 0x7FFFFF)
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The kcount-th largest key of a warp's row (NT keys per lane; key 0 = not
// selectable; 1 <= kcount <= number of selectable keys), by radix selection:
//  1. a coarse digit: each selectable score s maps to bin
//     min(255, floor((s - lo) * 256 / (hi - lo))) over the row's range
//     [lo, hi], a monotone map, so every key of a higher bin is larger than
//     every key of a lower one;
//  2. a 256-bin histogram of the digits (shared-memory counters of the warp)
//     and a warp scan from the top bin down find the bin holding the
//     kcount-th largest key and how many keys lie above it;
//  3. that bin's keys are ranked exactly: when the bin is taken whole the
//     answer is its smallest key; else, with at most 32 keys in the bin, each
//     lane ranks one of them against the others; else (many scores within one
//     bin) a bitwise search over the 32 key bits among the bin's keys.
// Any monotone digit gives the exact result; this one spreads the pooled
// scores of a row evenly over the bins, where the leading bits of the
// order-preserving key (sign and exponent) would crowd them into a few.
template <int NT>
FBM_DEVICE uint32_t fin_mask(const uint32_t (&key)[NT]) {
  uint32_t msk = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) msk |= (key[t] != 0u ? 1u : 0u) << t;
  return msk;
}

template <int NT>
FBM_DEVICE uint32_t bitwise_kth(const uint32_t (&key)[NT], uint32_t cand, int kcount) {
  // largest T with #(candidate key >= T) >= kcount
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) cnt += ((cand >> t) & 1u) && key[t] >= c ? 1 : 0;
    const int tot = __reduce_add_sync(0xffffffffu, cnt);
    if (tot >= kcount) T = c;
    if (tot == kcount) break;  // exactly kcount keys >= T: no tie left to resolve
  }
  // T may sit below the smallest qualifying key: move it up to that key
  uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (((cand >> t) & 1u) && key[t] >= T) mn = min(mn, key[t]);
  return __reduce_min_sync(0xffffffffu, mn);
}

template <int NT>
FBM_DEVICE uint32_t kth_largest_key(const uint32_t (&key)[NT], const float (&sc)[NT],
                                    uint32_t fin, int kcount, float hi, int *hist, int lane) {
  float lo_l = INFINITY;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if ((fin >> t) & 1u) lo_l = fminf(lo_l, sc[t]);
  float lo = lo_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
  const float range = hi - lo;
  const float inv = 256.0f / range;
  if (!(range > 0.f) || !(inv < INFINITY) || !(inv > 0.f))
    return bitwise_kth<NT>(key, fin, kcount);  // one value, or a range fp32 cannot split
  int dig[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) dig[t] = min(255, (int)((sc[t] - lo) * inv));
  // histogram: this warp's 256 counters
  reinterpret_cast<int4 *>(hist)[2 * lane] = make_int4(0, 0, 0, 0);
  reinterpret_cast<int4 *>(hist)[2 * lane + 1] = make_int4(0, 0, 0, 0);
  __syncwarp();
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if ((fin >> t) & 1u) atomicAdd(hist + dig[t], 1);
  __syncwarp();
  // lane L owns bins 255 - 8 L down to 248 - 8 L
  int c[8];
  {
    const int4 x = reinterpret_cast<const int4 *>(hist)[62 - 2 * lane];  // bins 248-8L .. 251-8L
    const int4 y = reinterpret_cast<const int4 *>(hist)[63 - 2 * lane];  // bins 252-8L .. 255-8L
    c[0] = y.w; c[1] = y.z; c[2] = y.y; c[3] = y.x;
    c[4] = x.w; c[5] = x.z; c[6] = x.y; c[7] = x.x;
  }
  int ssum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) ssum += c[i];
  int incl = ssum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int up = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += up;
  }
  int run = incl - ssum, found = -1, above = 0, binc = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (found < 0 && run + c[i] >= kcount) {
      found = 255 - 8 * lane - i;
      above = run;
      binc = c[i];
    }
    run += c[i];
  }
  // the first crossing from the top (lanes after it cross at once)
  const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
  const int src = __ffs(bal) - 1;
  const int dsel = __shfl_sync(0xffffffffu, found, src);
  const int need = kcount - __shfl_sync(0xffffffffu, above, src);
  const int nbin = __shfl_sync(0xffffffffu, binc, src);
  uint32_t cand = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) cand |= (((fin >> t) & 1u) && dig[t] == dsel ? 1u : 0u) << t;
  if (need == nbin) {
    // the bin is taken whole: its smallest key
    uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if ((cand >> t) & 1u) mn = min(mn, key[t]);
    return __reduce_min_sync(0xffffffffu, mn);
  }
  if (nbin > 32) return bitwise_kth<NT>(key, cand, need);
  // compact the bin's keys, one per lane, in the warp's counters (done with)
  __syncwarp();
  uint32_t *slot = reinterpret_cast<uint32_t *>(hist);
  const unsigned lt = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const bool cnd = (cand >> t) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, cnd);
    if (cnd) slot[base + __popc(b & lt)] = key[t];
    base += __popc(b);
  }
  __syncwarp();
  const uint32_t mine = lane < nbin ? slot[lane] : 0u;
  int gt = 0;
  for (int i = 0; i < nbin; ++i) gt += slot[i] > mine ? 1 : 0;
  // the need-th largest: the smallest key with fewer than `need` keys above it
  const uint32_t v = (lane < nbin && gt < need) ? mine : 0xFFFFFFFFu;
  return __reduce_min_sync(0xffffffffu, v);
}

// The selection of one q block (row), by one warp.  NT keys per lane cover
// columns 0 .. 32 NT - 1; every eligible column of the row must lie below
// 32 NT (the causal rows of a long sequence take a smaller NT than the
// kernel's, so that they do work for their eligible prefix only).
template <int NT>
FBM_DEVICE void select_row(const SelectArgs &a, const HeadParams &hp, int rowid, int n_elig,
                           int *hist, int lane) {
  const int i = rowid % a.nq;
  const int bh = rowid / a.nq;
  const int h = bh % a.hq, bi = bh / a.hq;
  const int g = h / (a.hq / a.hk);
  const float *qsim = a.qsim + (size_t)(bi * a.hq + h) * a.nq;
  const float *ksim = a.ksim + (size_t)(bi * a.hk + g) * a.nk;
  const float *srow = reinterpret_cast<const float *>(a.lut) + (size_t)rowid * a.nk;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int ncols = min(a.nk, 32 * NT);
  {
    const float theta = hp.theta[h];
    const bool q_similar = qsim[i] > theta;
    float sc[NT];
    uint32_t key[NT];
    bool elig[NT], ksim_ok[NT];
    float mloc = -INFINITY;
    int nfin = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j = lane + 32 * t;
      const bool valid = j < ncols;
      elig[t] = valid && j < n_elig;
      ksim_ok[t] = elig[t] && ksim[j] > theta;
      const bool fin = elig[t] && ksim_ok[t];
      // a plain load (this kernel rewrites the row); adding +0 turns a -0
      // score into +0, so the float compares of the threshold search and the
      // integer keys order signed zeros alike
      sc[t] = elig[t] ? __fadd_rn(srow[j], 0.0f) : 0.f;
      key[t] = fin ? order_key(sc[t]) : 0u;
      if (fin) mloc = fmaxf(mloc, sc[t]);
      nfin += fin ? 1 : 0;
    }
    nfin = __reduce_add_sync(0xffffffffu, nfin);
    bool sel[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) sel[t] = false;
    if (nfin > 0) {
      const float m = warp_max(mloc);
      if (!a.mode_cdf) {
        const float prod = __fmul_rn(hp.sel[h], (float)n_elig);
        const int kcount = min((int)ceilf(prod), nfin);
        const uint32_t T = kth_largest_key<NT>(key, sc, fin_mask(key), kcount, m, hist, lane);
        int cgt = 0;
#pragma unroll
        for (int t = 0; t < NT; ++t) cgt += key[t] > T ? 1 : 0;
        const int need = kcount - __reduce_add_sync(0xffffffffu, cgt);
        int run = 0;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const bool tie = key[t] == T && key[t] != 0u;
          const unsigned bal = __ballot_sync(0xffffffffu, tie);
          sel[t] = key[t] > T || (tie && run + __popc(bal & lt_mask) < need);
          run += __popc(bal);
        }
      } else {
        float p[NT];
        float ps = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          p[t] = key[t] ? expf(sc[t] - m) : 0.f;
          ps += p[t];
        }
        const float inv = 1.0f / warp_sum(ps);
#pragma unroll
        for (int t = 0; t < NT; ++t) p[t] *= inv;
        const float tau = hp.sel[h];
        float mass_all = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) mass_all += p[t];
        mass_all = warp_sum(mass_all);
        if (mass_all < tau) {
#pragma unroll
          for (int t = 0; t < NT; ++t) sel[t] = key[t] != 0u;
        } else {
          // largest T with mass(key >= T) >= tau
          uint32_t T = 0;
          for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            float ms = 0.f;
#pragma unroll
            for (int t = 0; t < NT; ++t) ms += key[t] >= cand ? p[t] : 0.f;
            if (warp_sum(ms) >= tau) T = cand;
          }
          float mgt = 0.f;
#pragma unroll
          for (int t = 0; t < NT; ++t) mgt += key[t] > T ? p[t] : 0.f;
          float carry = warp_sum(mgt);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const bool tie = key[t] == T && key[t] != 0u;
            float v = tie ? p[t] : 0.f;
            float incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float up = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += up;
            }
            sel[t] = key[t] > T || (tie && carry + (incl - v) < tau);
            carry += __shfl_sync(0xffffffffu, incl, 31);
          }
        }
      }
    }
    // forced columns / rows, sink, causal; ascending emission by ballot scan
    // (over the scores every lane has already read)
    __syncwarp();
    const size_t row = (size_t)rowid;
    int32_t *lut = a.lut + row * a.nk;
    int run = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j = lane + 32 * t;
      const bool forced = elig[t] && (!ksim_ok[t] || !q_similar || (a.sink && j == 0));
      const bool keep = elig[t] && (sel[t] || forced);
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (keep) lut[run + __popc(bal & lt_mask)] = j;
      if (a.bmap && j < ncols) a.bmap[row * a.nk + j] = keep ? 1 : 0;
      run += __popc(bal);
    }
    for (int p = run + lane; p < a.nk; p += 32) lut[p] = -1;
    if (a.bmap)
      for (int j = ncols + lane; j < a.nk; j += 32) a.bmap[row * a.nk + j] = 0;
    if (lane == 0) a.cnt[row] = run;
  }
}


// one warp per q block (row): 8 warps per CTA.  NT = ceil(nk / 32) keys per
// lane; a causal row whose eligible prefix is shorter runs the body of a
// smaller NT (the branch is uniform over the warp).
template <int NT>
__global__ void __launch_bounds__(256) k_select(SelectArgs a, const __grid_constant__ HeadParams hp) {
  __shared__ __align__(16) int hist_all[8][256];  // radix-select counters, one set per warp
  const int lane = threadIdx.x & 31;
  int *hist = hist_all[threadIdx.x >> 5];
  const int rowid = blockIdx.x * 8 + (threadIdx.x >> 5);  // (batch, head, q block)
  if (rowid >= a.b * a.hq * a.nq) return;
  const int i = rowid % a.nq;
  const int last_q = (i + 1) * a.blkq - 1;
  const int n_elig = a.causal ? min(a.nk, last_q / a.blkk + 1) : a.nk;
  constexpr int kQ = NT / 4;  // quarter steps (NT is a multiple of 4)
  if (NT >= 8 && n_elig <= 32 * kQ) select_row<kQ>(a, hp, rowid, n_elig, hist, lane);
  else if (NT >= 8 && n_elig <= 64 * kQ) select_row<2 * kQ>(a, hp, rowid, n_elig, hist, lane);
  else if (NT >= 8 && n_elig <= 96 * kQ) select_row<3 * kQ>(a, hp, rowid, n_elig, hist, lane);
  else select_row<NT>(a, hp, rowid, n_elig, hist, lane);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------

template <int NT>
static cudaError_t launch_select(const SelectArgs &a, const HeadParams &hp, cudaStream_t st) {
  const int rows = a.b * a.hq * a.nq;
  k_select<NT><<<(rows + 7) / 8, 256, 0, st>>>(a, hp);
  return cudaGetLastError();
}

static cudaError_t launch_select_nt(const SelectArgs &a, const HeadParams &hp, cudaStream_t st) {
  if (a.nk <= 256) return launch_select<8>(a, hp, st);
  if (a.nk <= 512) return launch_select<16>(a, hp, st);
  return launch_select<32>(a, hp, st);
}

int device_sm_count();  // fmha_tc.cu

constexpr int kMaxPoolDevices = 64;

template <class E, int D, bool SMOOTH>
static cudaError_t launch_pool_t(const PoolSide &qs, const PoolSide &ks, uint32_t *err,
                                 cudaStream_t st) {
  // the shared-memory attribute is per device: set it once on each
  static std::atomic<bool> attr_done[kMaxPoolDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxPoolDevices || !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_pool_sim<E, D, SMOOTH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PoolRing<D>::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxPoolDevices) attr_done[dev].store(true, std::memory_order_release);
  }
  const int total = qs.nunits + ks.nunits;
  if (total == 0) return cudaSuccess;
  const int grid = std::min(total, device_sm_count());
  k_pool_sim<E, D, SMOOTH><<<grid, kPoolThreads, PoolRing<D>::kSmem, st>>>(qs, ks, err);
  return cudaGetLastError();
}

template <bool SMOOTH>
static cudaError_t launch_pool(const BlockMapLaunch &L, const PoolSide &qs, const PoolSide &ks,
                               cudaStream_t st) {
  if (L.d == 128)
    return L.bf16 ? launch_pool_t<BF16, 128, SMOOTH>(qs, ks, L.err, st)
                  : launch_pool_t<F16, 128, SMOOTH>(qs, ks, L.err, st);
  return L.bf16 ? launch_pool_t<BF16, 64, SMOOTH>(qs, ks, L.err, st)
                : launch_pool_t<F16, 64, SMOOTH>(qs, ks, L.err, st);
}

cudaError_t launch_block_map(const BlockMapLaunch &L, cudaStream_t st) {
  PoolSide qs{static_cast<const uint16_t *>(L.q), L.qpl, L.qsim, L.s, L.nq, L.b * L.hq * L.nq,
              nullptr};
  PoolSide ks{static_cast<const uint16_t *>(L.k), L.kpl, L.ksim, L.s, L.nk, L.b * L.hk * L.nk,
              nullptr};
  cudaError_t e = launch_pool<false>(L, qs, ks, st);
  if (e != cudaSuccess) return e;
  if (L.smooth_k) {
    // K smoothing: mean key row from the block means just written, then pool
    // and measure K again on the centred rows (Q results are kept)
    if (L.d == 128) k_key_mean<128><<<L.b * L.hk, 256, 0, st>>>(L.kpl, L.kmu, L.s, L.nk);
    else k_key_mean<64><<<L.b * L.hk, 256, 0, st>>>(L.kpl, L.kmu, L.s, L.nk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    PoolSide none = qs;
    none.nunits = 0;
    ks.mu = L.kmu;
    e = launch_pool<true>(L, none, ks, st);
    if (e != cudaSuccess) return e;
  }
  SelectArgs a{};
  a.qpl = L.qpl; a.qsim = L.qsim; a.kpl = L.kpl; a.ksim = L.ksim;
  a.b = L.b; a.hq = L.hq; a.hk = L.hk; a.nq = L.nq; a.nk = L.nk;
  a.blkq = kBlk; a.blkk = kBlk;
  a.scale = L.scale; a.causal = L.causal; a.sink = L.sink; a.mode_cdf = L.mode_cdf;
  a.lut = L.lut; a.cnt = L.cnt; a.bmap = L.bmap;
  a.err = L.err;
  e = launch_pooled_scores_tc(a, L.d, st);
  if (e != cudaSuccess) return e;
  return launch_select_nt(a, L.hp, st);
}

}  // namespace fbm
