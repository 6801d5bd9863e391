// Block-map prediction kernels ("Sparge Attention (Composable Kernel)" README:
// mean-pool -> cosine sim -> pooled QK -> top-k / cdfthreshd LUT).
//
//  k_pool_sim     persistent, one CTA per SM: a producer lane bulk-copies
//                 whole 64-token blocks of Q and K (contiguous rows) into a
//                 192 KB shared-memory ring with an evict-first L2 hint; eight
//                 consumer warps reduce them: row norms, fp32 row sums (the
//                 pooled mean, two interleaved packed f32x2 partial sums per
//                 element) and the sum of unit rows (self-similarity =
//                 ||sum u||^2 / n^2).  HBM-bound: it reads Q and K once and
//                 writes, per block, the mean as three bf16 split planes (the
//                 operands of the pooled scores' tensor-core product, in their
//                 shared-memory layout) and one float.
//  k_key_mean     K smoothing only: one CTA per (batch, KV head) forms the mean
//                 key row from the block means of the first pooling pass (fixed
//                 summation order, so the result is deterministic); a second
//                 pooling pass over K then subtracts it from every key row
//                 before the norms and sums.
//  pooled scores  scale * qbar . kbar on tcgen05 from the split planes
//                 (pooled_scores_tc.cu), written as fp32 into the caller's LUT
//                 buffer, which has exactly the size of the score matrix.
//  k_select       one warp per q block: loads its score row, then (cdf mode) the
//                 pooled softmax, a radix select of the threshold (a 256-bin
//                 histogram of a linear digit, exact ranking inside the
//                 crossing bin) and ballot-scan emission of the ascending LUT
//                 row over the scores it has read.  No atomics take part in
//                 slot assignment.  The paths real-valued rows rarely take run
//                 out of line, so that the unrolled row bodies stay in the
//                 instruction cache.
#include <algorithm>
#include <atomic>

#include <cuda_fp8.h>

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
  uint8_t *codes;     // [bh, s, D] e4m3 codes of the raw rows (QUANT only)
  float *scales;      // [bh * nb] one scale per block (QUANT only)
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

template <class E, int D, bool SMOOTH, bool QUANT>
__global__ void __launch_bounds__(kPoolThreads, 1) k_pool_sim(PoolSide qs, PoolSide ks, uint32_t *err) {
  static_assert(!QUANT || (D == 128 && !SMOOTH), "e4m3 codes: d = 128, raw rows");
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
  pdl_trigger();  // the score kernel may launch now and wait for this grid
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
      // Q and K are read once: keep them from evicting the split planes,
      // which the pooled-score kernel reads next
      const uint64_t policy = tc::l2_evict_first();
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
        tc::bulk_load_hint(sbase + st * R::kBlockBytes,
                           side.x + ((size_t)bh * side.s + (size_t)j * kBlk) * D, bytes, full(st),
                           policy);
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
    // element pairs (2 p, 2 p + 1) in one 64-bit register: packed f32x2
    // arithmetic, each half an ordinary IEEE fp32 operation
    uint64_t nmu[8];
    if constexpr (SMOOTH) {
      const float4 *m0 = reinterpret_cast<const float4 *>(side.mu + (size_t)bh * D + sub * 8);
      const float4 *m1 = reinterpret_cast<const float4 *>(side.mu + (size_t)bh * D + D / 2 + sub * 8);
      const float4 a0 = m0[0], a1 = m0[1], b0 = m1[0], b1 = m1[1];
      nmu[0] = tc::f2_pack(-a0.x, -a0.y); nmu[1] = tc::f2_pack(-a0.z, -a0.w);
      nmu[2] = tc::f2_pack(-a1.x, -a1.y); nmu[3] = tc::f2_pack(-a1.z, -a1.w);
      nmu[4] = tc::f2_pack(-b0.x, -b0.y); nmu[5] = tc::f2_pack(-b0.z, -b0.w);
      nmu[6] = tc::f2_pack(-b1.x, -b1.y); nmu[7] = tc::f2_pack(-b1.z, -b1.w);
    }

    // two interleaved partial sums per element keep the fp32 sums short
    uint64_t msum[2][8], usum[8];
    const uint64_t zero2 = tc::f2_pack(0.f, 0.f);
    float amax = 0.f;  // max |x| over the block (QUANT; absent rows read as 0)
#pragma unroll
    for (int p = 0; p < 8; ++p) msum[0][p] = msum[1][p] = usum[p] = zero2;
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
        uint64_t x[8];
        const uint32_t w[8] = {raw[uu][0].x, raw[uu][0].y, raw[uu][0].z, raw[uu][0].w,
                               raw[uu][1].x, raw[uu][1].y, raw[uu][1].z, raw[uu][1].w};
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const float2 f = E::to_f2(w[p]);
          x[p] = tc::f2_pack(f.x, f.y);
          if constexpr (QUANT) amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
        if constexpr (SMOOTH) {
          // rows past the end stay zero: they add nothing to either sum
          const int r = (s0 + uu) * RPI + rgrp;
          if (r < n) {
#pragma unroll
            for (int p = 0; p < 8; ++p) x[p] = tc::f2_add(x[p], nmu[p]);
          }
        }
        uint64_t ss2 = zero2;
#pragma unroll
        for (int p = 0; p < 8; ++p) ss2 = tc::f2_fma(x[p], x[p], ss2);
        const float2 ssp = tc::f2_unpack(ss2);
        float ss = ssp.x + ssp.y;
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
        const uint64_t inv2 = tc::f2_pack(inv, inv);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          usum[p] = tc::f2_fma(x[p], inv2, usum[p]);
          msum[uu & 1][p] = tc::f2_add(msum[uu & 1][p], x[p]);
        }
      }
    }
    if constexpr (QUANT) {
      // e4m3 codes of the block from the same shared-memory copy: one scale
      // per block (amax / 448, IEEE), codes = e4m3(x * (448 / amax)) rounded
      // to nearest even with saturation; an all-zero block has scale 1
      amax = warp_max(amax);
      const float qscale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
      if (lane == 0) side.scales[unit] = qscale;
      uint8_t *dst = side.codes + ((size_t)bh * side.s + (size_t)j * kBlk) * D;
      const int qsub = lane & 15, qsel = lane >> 4;  // 8 values of a row; even / odd row
#pragma unroll 4
      for (int r = qsel; r < n; r += 2) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(blk + r * (2 * D) + qsub * 16);
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t out[2];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 f = E::to_f2(ws[p]);
          const float2 y = make_float2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
          const uint32_t c2 = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);  // .x low
          if (p & 1) out[p >> 1] |= c2 << 16;
          else out[p >> 1] = c2;
        }
        *(reinterpret_cast<uint2 *>(dst + (size_t)r * D) + qsub) = make_uint2(out[0], out[1]);
      }
    }
    // the stage is free once every lane has read it
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty(st));

    float tot[16], us[16];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const float2 a = tc::f2_unpack(msum[0][p]), b = tc::f2_unpack(msum[1][p]);
      const float2 u2 = tc::f2_unpack(usum[p]);
      tot[2 * p] = a.x + b.x;
      tot[2 * p + 1] = a.y + b.y;
      us[2 * p] = u2.x;
      us[2 * p + 1] = u2.y;
    }
#pragma unroll
    for (int o = 16; o >= LPR; o >>= 1) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        tot[e] += __shfl_xor_sync(0xffffffffu, tot[e], o);
        us[e] += __shfl_xor_sync(0xffffffffu, us[e], o);
      }
    }
    float su = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) su = fmaf(us[e], us[e], su);
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
FBM_DEVICE float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A row of scores held by one warp: NT per lane, column j = lane + 32 t; bit
// t of a lane's word `fin` marks a selectable score (eligible and similar).
// Scores carry no -0 (the loader adds +0), so comparing the floats orders
// them exactly as their order-preserving keys do.
FBM_DEVICE bool is_fin(uint32_t fin, int t) { return (fin >> t) & 1u; }

// Largest T (a key) with #(selectable key >= T) >= kcount, by a bitwise
// search over the 32 key bits among the candidates `cand` (bit t of this
// lane's word).
template <int NT>
FBM_DEVICE uint32_t bitwise_kth(const float (&sc)[NT], uint32_t cand, int kcount) {
  uint32_t key[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) key[t] = ((cand >> t) & 1u) ? order_key(sc[t]) : 0u;
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) cnt += key[t] >= c ? 1 : 0;
    const int tot = __reduce_add_sync(0xffffffffu, cnt);
    if (tot >= kcount) T = c;
    if (tot == kcount) break;  // exactly kcount keys >= T: no tie left to resolve
  }
  // T may sit below the smallest qualifying key: move it up to that key
  uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (key[t] >= T && key[t] != 0u) mn = min(mn, key[t]);
  return __reduce_min_sync(0xffffffffu, mn);
}

// A row's scores by value, for the out-of-line rare paths (the hot path keeps
// them in registers).
template <int NT>
struct RowScores {
  float v[NT];
};
struct KthResult {
  float tv;
  bool exact;
};

// The kcount-th largest score among `cand` by the bitwise key search, and
// whether exactly kcount candidates lie at or above it.  Out of line: taken
// only for a row whose range fp32 cannot split or whose crossing bin holds
// more than 32 scores.
template <int NT>
__device__ __noinline__ KthResult kth_by_bits(const RowScores<NT> r, uint32_t cand, int kcount) {
  const uint32_t T = bitwise_kth<NT>(r.v, cand, kcount);
  const float tv = key_value(T);
  int ge = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) ge += ((cand >> t) & 1u) && r.v[t] >= tv ? 1 : 0;
  KthResult k;
  k.tv = tv;
  k.exact = __reduce_add_sync(0xffffffffu, ge) == kcount;
  return k;
}

// Selection bits of a row whose threshold score tv is tied: every score above
// tv, then the tied ones in ascending column order up to kcount.  Out of line
// (rare for real-valued scores).
template <int NT>
__device__ __noinline__ uint32_t select_ties(const RowScores<NT> r, uint32_t fin, float tv, int kcount,
                                             int lane) {
  const unsigned lt_mask = (1u << lane) - 1u;
  int cgt = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) cgt += is_fin(fin, t) && r.v[t] > tv ? 1 : 0;
  const int need = kcount - __reduce_add_sync(0xffffffffu, cgt);
  int run = 0;
  uint32_t sel = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const bool tie = is_fin(fin, t) && r.v[t] == tv;
    const unsigned bal = __ballot_sync(0xffffffffu, tie);
    const bool s = (is_fin(fin, t) && r.v[t] > tv) || (tie && run + __popc(bal & lt_mask) < need);
    sel |= (s ? 1u : 0u) << t;
    run += __popc(bal);
  }
  return sel;
}

// The kcount-th largest selectable score of a warp's row (1 <= kcount <=
// number of selectable scores), by radix selection:
//  1. a coarse digit: each selectable score s maps to bin
//     min(255, floor((s - lo) * 256 / (hi - lo))) over the row's range
//     [lo, hi], a monotone map, so every score of a higher bin is larger than
//     every score of a lower one;
//  2. a 256-bin histogram of the digits (shared-memory counters of the warp)
//     and a warp scan from the top bin down find the bin holding the
//     kcount-th largest score and how many scores lie above it;
//  3. that bin's scores are ranked exactly: when the bin is taken whole the
//     answer is its smallest score; else, with at most 32 scores in the bin,
//     each lane ranks one of them against the others; else (many scores
//     within one bin) a bitwise search over the 32 key bits of the bin.
// Any monotone digit gives the exact result; this one spreads the pooled
// scores of a row evenly over the bins, where the leading bits of the
// order-preserving key (sign and exponent) would crowd them into a few.
// `exact` is set when the scores >= the result number exactly kcount (no
// tie at the threshold needs breaking).
template <int NT>
FBM_DEVICE float kth_largest(const float (&sc)[NT], uint32_t finl, int kcount, float hi,
                             int *hist, int lane, bool &exact) {
  const unsigned lt = (1u << lane) - 1u;
  float lo_l = INFINITY;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (is_fin(finl, t)) lo_l = fminf(lo_l, sc[t]);
  float lo = lo_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
  const float range = hi - lo;
  const float inv = 256.0f / range;
  if (!(range > 0.f) || !(inv < INFINITY) || !(inv > 0.f)) {
    // one value, or a range fp32 cannot split
    RowScores<NT> r;
#pragma unroll
    for (int t = 0; t < NT; ++t) r.v[t] = sc[t];
    const KthResult k = kth_by_bits<NT>(r, finl, kcount);
    exact = k.exact;
    return k.tv;
  }
  int dig[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) dig[t] = min(255, (int)((sc[t] - lo) * inv));
  // histogram: this warp's 256 counters
  reinterpret_cast<int4 *>(hist)[2 * lane] = make_int4(0, 0, 0, 0);
  reinterpret_cast<int4 *>(hist)[2 * lane + 1] = make_int4(0, 0, 0, 0);
  __syncwarp();
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if ((finl >> t) & 1u) atomicAdd(hist + dig[t], 1);
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
  for (int k = 0; k < 8; ++k) ssum += c[k];
  int incl = ssum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int up = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += up;
  }
  int run = incl - ssum, found = -1, above = 0, binc = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (found < 0 && run + c[k] >= kcount) {
      found = 255 - 8 * lane - k;
      above = run;
      binc = c[k];
    }
    run += c[k];
  }
  // the first crossing from the top (lanes after it cross at once)
  const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
  const int src = __ffs(bal) - 1;
  const int dsel = __shfl_sync(0xffffffffu, found, src);
  const int need = kcount - __shfl_sync(0xffffffffu, above, src);
  const int nbin = __shfl_sync(0xffffffffu, binc, src);
  uint32_t cand = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) cand |= (((finl >> t) & 1u) && dig[t] == dsel ? 1u : 0u) << t;
  if (need == nbin) {
    // the bin is taken whole: its smallest score (every larger score is
    // taken too, and every score equal to it lies in the bin)
    float mn = INFINITY;
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if ((cand >> t) & 1u) mn = fminf(mn, sc[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    exact = true;
    return mn;
  }
  if (nbin > 32) {
    RowScores<NT> r;
#pragma unroll
    for (int t = 0; t < NT; ++t) r.v[t] = sc[t];
    const KthResult k = kth_by_bits<NT>(r, cand, need);
    exact = k.exact;
    return k.tv;
  }
  // compact the bin's scores, one per lane, in the warp's counters (done with)
  __syncwarp();
  float *slot = reinterpret_cast<float *>(hist);
  int base = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const bool cnd = (cand >> t) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, cnd);
    if (cnd) slot[base + __popc(b & lt)] = sc[t];
    base += __popc(b);
  }
  __syncwarp();
  const float mine = lane < nbin ? slot[lane] : -INFINITY;
  int gt = 0;
  for (int k = 0; k < nbin; ++k) gt += slot[k] > mine ? 1 : 0;
  // the need-th largest: the smallest score with fewer than `need` above it
  const float v = (lane < nbin && gt < need) ? mine : INFINITY;
  float tv = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tv = fminf(tv, __shfl_xor_sync(0xffffffffu, tv, o));
  exact = __popc(__ballot_sync(0xffffffffu, lane < nbin && mine >= tv)) == need;
  return tv;
}

// The selection of one q block (row), by one warp.  NT scores per lane cover
// columns 0 .. 32 NT - 1; every eligible column of the row must lie below
// 32 NT (the causal rows of a long sequence take a smaller NT than the
// kernel's, so that they do work for their eligible prefix only).
template <int NT, bool CDF>
FBM_DEVICE void select_row(const SelectArgs &a, const HeadParams &hp, int rowid, int n_elig,
                           int *hist, int lane) {
  const int i = rowid % a.nq;
  const int bh = rowid / a.nq;
  const int h = bh % a.hq, bi = bh / a.hq;
  const int g = h / (a.hq / a.hk);
  const float *ksim = a.ksim + (size_t)(bi * a.hk + g) * a.nk;
  const float *srow = reinterpret_cast<const float *>(a.lut) + (size_t)rowid * a.nk;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int ncols = min(a.nk, 32 * NT);
  const float theta = hp.theta[h];
  const bool q_similar = a.qsim[(size_t)(bi * a.hq + h) * a.nq + i] > theta;
  float sc[NT];
  uint32_t fin = 0;  // bit t: column lane + 32 t is selectable
  float mloc = -INFINITY;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int j = lane + 32 * t;
    const bool elig = j < n_elig;  // eligible columns form a prefix of the row
    // a plain load (this kernel rewrites the row); adding +0 turns a -0
    // score into +0, so float compares and integer keys order them alike
    sc[t] = elig ? __fadd_rn(srow[j], 0.0f) : 0.f;
    const bool f = elig && ksim[j] > theta;
    fin |= (f ? 1u : 0u) << t;
    if (f) mloc = fmaxf(mloc, sc[t]);
  }
  const int nfin = __reduce_add_sync(0xffffffffu, __popc(fin));
  uint32_t sel = 0;  // this lane's selected scores, bit t
  if (nfin > 0) {
    const float m = warp_max(mloc);
    if constexpr (!CDF) {
      const float prod = __fmul_rn(hp.sel[h], (float)n_elig);
      const int kcount = min((int)ceilf(prod), nfin);
      bool exact = false;
      const float tv = kth_largest<NT>(sc, fin, kcount, m, hist, lane, exact);
      if (exact) {
#pragma unroll
        for (int t = 0; t < NT; ++t) sel |= (is_fin(fin, t) && sc[t] >= tv ? 1u : 0u) << t;
      } else {
        // ties at the threshold: the lower kv blocks first
        RowScores<NT> r;
#pragma unroll
        for (int t = 0; t < NT; ++t) r.v[t] = sc[t];
        sel = select_ties<NT>(r, fin, tv, kcount, lane);
      }
    } else {
      uint32_t key[NT];
      float p[NT];
      float ps = 0.f;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        key[t] = is_fin(fin, t) ? order_key(sc[t]) : 0u;
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
        for (int t = 0; t < NT; ++t) sel |= (key[t] != 0u ? 1u : 0u) << t;
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
          const bool s = key[t] > T || (tie && carry + (incl - v) < tau);
          sel |= (s ? 1u : 0u) << t;
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
    }
  }
  // forced columns / rows, sink, causal; ascending emission by ballot scan
  // (over the scores every lane has already read).  An eligible column is
  // forced when its kv block is not similar (it is eligible but not
  // selectable), when the q block is not similar, or for the sink.
  __syncwarp();
  const size_t row = (size_t)rowid;
  int32_t *lut = a.lut + row * a.nk;
  int run = 0;
  uint32_t keepm = 0;  // bit t: column lane + 32 t is kept
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int j = lane + 32 * t;
    const bool elig = j < n_elig;
    const bool keep = elig && (((sel >> t) & 1u) || !is_fin(fin, t) || !q_similar ||
                               (a.sink && j == 0));
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (keep) lut[run + __popc(bal & lt_mask)] = j;
    keepm |= (keep ? 1u : 0u) << t;
    run += __popc(bal);
  }
  for (int p = run + lane; p < a.nk; p += 32) lut[p] = -1;
  if (a.bmap) {
    // the optional 0/1 block map, kept out of the unrolled loops above
    uint8_t *brow = a.bmap + row * a.nk;
#pragma unroll 1
    for (int t = 0; t < NT; ++t) {
      const int j = lane + 32 * t;
      if (j < ncols) brow[j] = (uint8_t)((keepm >> t) & 1u);
    }
    for (int j = ncols + lane; j < a.nk; j += 32) brow[j] = 0;
  }
  if (lane == 0) a.cnt[row] = run;
}

// one warp per q block (row): 8 warps per CTA.  NT = ceil(nk / 32) scores per
// lane; a causal row whose eligible prefix is shorter runs the body of a
// smaller NT (the branch is uniform over the warp).  Up to NT = 16, four CTAs
// per SM (64 registers): with a few spilled bytes this measured faster than
// three CTAs at 80 registers, the rows waiting mostly on their loads.
template <int NT, bool CDF>
__global__ void __launch_bounds__(256, NT <= 16 ? 4 : 1)
    k_select(SelectArgs a, const __grid_constant__ HeadParams hp) {
  __shared__ __align__(16) int hist_all[8][256];  // radix-select counters, one set per warp
  const int lane = threadIdx.x & 31;
  int *hist = hist_all[threadIdx.x >> 5];
  const int rowid = blockIdx.x * 8 + (threadIdx.x >> 5);  // (batch, head, q block)
  if (rowid >= a.b * a.hq * a.nq) return;
  const int i = rowid % a.nq;
  const int last_q = (i + 1) * a.blkq - 1;
  const int n_elig = a.causal ? min(a.nk, last_q / a.blkk + 1) : a.nk;
  pdl_wait();  // the scores kernel's output
  constexpr int kQ = NT / 4;  // quarter steps (NT is a multiple of 4)
  if (NT >= 8 && n_elig <= 32 * kQ) select_row<kQ, CDF>(a, hp, rowid, n_elig, hist, lane);
  else if (NT >= 8 && n_elig <= 64 * kQ) select_row<2 * kQ, CDF>(a, hp, rowid, n_elig, hist, lane);
  else if (NT >= 8 && n_elig <= 96 * kQ) select_row<3 * kQ, CDF>(a, hp, rowid, n_elig, hist, lane);
  else select_row<NT, CDF>(a, hp, rowid, n_elig, hist, lane);
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------

template <int NT>
static cudaError_t launch_select(const SelectArgs &a, const HeadParams &hp, cudaStream_t st) {
  const int rows = a.b * a.hq * a.nq;
  const dim3 grid((rows + 7) / 8);
  if (a.mode_cdf) return launch_pdl(k_select<NT, true>, grid, dim3(256), 0, st, a, hp);
  return launch_pdl(k_select<NT, false>, grid, dim3(256), 0, st, a, hp);
}

static cudaError_t launch_select_nt(const SelectArgs &a, const HeadParams &hp, cudaStream_t st) {
  if (a.nk <= 256) return launch_select<8>(a, hp, st);
  if (a.nk <= 512) return launch_select<16>(a, hp, st);
  return launch_select<32>(a, hp, st);
}

int device_sm_count();  // fmha_tc.cu

constexpr int kMaxPoolDevices = 64;

template <class E, int D, bool SMOOTH, bool QUANT>
static cudaError_t launch_pool_t(const PoolSide &qs, const PoolSide &ks, uint32_t *err,
                                 cudaStream_t st) {
  // the shared-memory attribute is per device: set it once on each
  static std::atomic<bool> attr_done[kMaxPoolDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxPoolDevices || !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_pool_sim<E, D, SMOOTH, QUANT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PoolRing<D>::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxPoolDevices) attr_done[dev].store(true, std::memory_order_release);
  }
  const int total = qs.nunits + ks.nunits;
  if (total == 0) return cudaSuccess;
  const int grid = std::min(total, device_sm_count());
  k_pool_sim<E, D, SMOOTH, QUANT><<<grid, kPoolThreads, PoolRing<D>::kSmem, st>>>(qs, ks, err);
  return cudaGetLastError();
}

template <bool SMOOTH>
static cudaError_t launch_pool(const BlockMapLaunch &L, const PoolSide &qs, const PoolSide &ks,
                               cudaStream_t st) {
  if constexpr (!SMOOTH) {
    // e4m3 codes of Q and K requested (d = 128, checked by the caller)
    if (qs.codes)
      return L.bf16 ? launch_pool_t<BF16, 128, false, true>(qs, ks, L.err, st)
                    : launch_pool_t<F16, 128, false, true>(qs, ks, L.err, st);
  }
  if (L.d == 128)
    return L.bf16 ? launch_pool_t<BF16, 128, SMOOTH, false>(qs, ks, L.err, st)
                  : launch_pool_t<F16, 128, SMOOTH, false>(qs, ks, L.err, st);
  return L.bf16 ? launch_pool_t<BF16, 64, SMOOTH, false>(qs, ks, L.err, st)
                : launch_pool_t<F16, 64, SMOOTH, false>(qs, ks, L.err, st);
}

cudaError_t launch_block_map(const BlockMapLaunch &L, cudaStream_t st) {
  PoolSide qs{static_cast<const uint16_t *>(L.q), L.qpl, L.qsim, L.s, L.nq, L.b * L.hq * L.nq,
              nullptr};
  PoolSide ks{static_cast<const uint16_t *>(L.k), L.kpl, L.ksim, L.s, L.nk, L.b * L.hk * L.nk,
              nullptr};
  qs.codes = L.q8; qs.scales = L.q_scale;
  ks.codes = L.k8; ks.scales = L.k_scale;
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
    none.codes = nullptr;
    ks.mu = L.kmu;
    ks.codes = nullptr;
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
