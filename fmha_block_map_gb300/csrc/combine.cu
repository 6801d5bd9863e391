// LSE combine of split-KV partials (Incremental_FlashAttention updating_log,
// Stage 1: the lse_max trick; ROCm/aiter pull 4919: the split-KV reduce).
//
// One warp per output row: lanes read the S partial LSEs, form
// m = max_s LSE_s and the weights w_s = exp(LSE_s - m), and stream the S
// partial rows with 128-bit loads, up to 8 partials in flight per lane (the
// first 8 issued before the weights are known), writing
// sum_s w_s O_s / sum_s w_s.  A row whose partials are all -inf (empty) writes
// O = 0 and LSE = -inf.  The kernel is bandwidth-bound: it reads
// S * (dv + 1) * 4 bytes and writes dv elements (+ 4 bytes of LSE) per row.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

constexpr int kBatch = 8;  // partial rows loaded per lane before they are weighted

template <int OUT>  // 0 = f16, 1 = bf16, 2 = f32
__global__ void __launch_bounds__(256) k_attn_combine(const CombineLaunch L) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= L.rows) return;
  pdl_wait();  // the partials' writer (launched just before, on the same stream)
  // weights: lane s holds split s (and s + 32)
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < L.num_splits) l0 = L.lse_part[(int64_t)lane * L.rows + row];
  if (lane + 32 < L.num_splits) l1 = L.lse_part[(int64_t)(lane + 32) * L.rows + row];
  // the partial rows of a batch are loaded before they are weighted, so their
  // latency overlaps (for the first batch, the weights' own load and shuffles)
  auto load_batch = [&](float4 (&x)[kBatch], int c, int s0) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int s = s0 + j;
      x[j] = (s < L.num_splits && c < L.dv)
                 ? __ldg(reinterpret_cast<const float4 *>(
                       L.o_part + ((int64_t)s * L.rows + row) * L.dv + c))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  float4 x[kBatch];
  load_batch(x, lane * 4, 0);
  const float m = warp_max(fmaxf(l0, l1));
  const bool live = m != -INFINITY;
  const float w0 = live ? expf(l0 - m) : 0.f;
  const float w1 = live ? expf(l1 - m) : 0.f;
  const float wsum = warp_sum(w0 + w1);
  const float inv = live ? 1.0f / wsum : 0.f;
  // every lane runs the same trip counts: the weight shuffles need the full warp
  for (int c0 = 0; c0 < L.dv; c0 += 128) {
    const int c = c0 + lane * 4;
    const bool act = c < L.dv;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < L.num_splits; s0 += kBatch) {
      if (c0 > 0 || s0 > 0) load_batch(x, c, s0);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int s = s0 + j;
        const float w = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
        // an empty partial (weight 0) adds nothing, whatever its row holds
        if (s < L.num_splits && w != 0.f) {
          acc.x = fmaf(w, x[j].x, acc.x);
          acc.y = fmaf(w, x[j].y, acc.y);
          acc.z = fmaf(w, x[j].z, acc.z);
          acc.w = fmaf(w, x[j].w, acc.w);
        }
      }
    }
    if (!act) continue;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    if constexpr (OUT == 2) {
      *reinterpret_cast<float4 *>(static_cast<float *>(L.out) + row * L.dv + c) = acc;
    } else {
      using E = typename std::conditional<OUT == 1, BF16, F16>::type;
      uint2 pk = make_uint2(E::from_f2(acc.x, acc.y), E::from_f2(acc.z, acc.w));
      *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(L.out) + row * L.dv + c) = pk;
    }
  }
  if (L.lse_out && lane == 0) L.lse_out[row] = live ? m + logf(wsum) : -INFINITY;
}

// Few splits (S <= 8): one thread per (row, CH chunks of 4 columns), unrolled
// for at most SMAX splits.  Each thread reads the row's S LSEs itself (the
// threads of a row share them through L1) and all of its S x CH partial
// chunks at once, then weights them: no cross-lane reduction and no load
// waiting on another, and with few registers many threads keep loads in
// flight.  Same order of operations as the warp kernel above, so the results
// are identical.  Both kernels are chained launches (launch_pdl): they wait
// for the kernel that wrote the partials before reading them.
constexpr int kSmallSplits = 8;

template <int OUT, int SMAX, int CH>
__global__ void __launch_bounds__(256) k_attn_combine_few(const CombineLaunch L) {
  const int per_row = L.dv / (4 * CH);
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= L.rows * per_row) return;
  pdl_wait();  // the partials' writer (launched just before, on the same stream)
  const int64_t row = t / per_row;
  const int c = (int)(t - row * per_row) * 4 * CH;
  float l[SMAX];
  float4 x[SMAX][CH];
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    const bool in = s < L.num_splits;
    l[s] = in ? __ldg(L.lse_part + (int64_t)s * L.rows + row) : -INFINITY;
    const float4 *src = reinterpret_cast<const float4 *>(L.o_part + ((int64_t)s * L.rows + row) * L.dv + c);
#pragma unroll
    for (int h = 0; h < CH; ++h) x[s][h] = in ? __ldg(src + h) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) m = fmaxf(m, l[s]);
  const bool live = m != -INFINITY;
  float4 acc[CH];
#pragma unroll
  for (int h = 0; h < CH; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    const float w = live ? expf(l[s] - m) : 0.f;
    wsum += w;
    // an empty partial (weight 0) adds nothing, whatever its row holds
    if (w != 0.f) {
#pragma unroll
      for (int h = 0; h < CH; ++h) {
        acc[h].x = fmaf(w, x[s][h].x, acc[h].x);
        acc[h].y = fmaf(w, x[s][h].y, acc[h].y);
        acc[h].z = fmaf(w, x[s][h].z, acc[h].z);
        acc[h].w = fmaf(w, x[s][h].w, acc[h].w);
      }
    }
  }
  const float inv = live ? 1.0f / wsum : 0.f;
#pragma unroll
  for (int h = 0; h < CH; ++h) {
    float4 a = acc[h];
    a.x *= inv; a.y *= inv; a.z *= inv; a.w *= inv;
    if constexpr (OUT == 2) {
      reinterpret_cast<float4 *>(static_cast<float *>(L.out) + row * L.dv + c)[h] = a;
    } else {
      using E = typename std::conditional<OUT == 1, BF16, F16>::type;
      reinterpret_cast<uint2 *>(static_cast<uint16_t *>(L.out) + row * L.dv + c)[h] =
          make_uint2(E::from_f2(a.x, a.y), E::from_f2(a.z, a.w));
    }
  }
  if (L.lse_out && c == 0) L.lse_out[row] = live ? m + logf(wsum) : -INFINITY;
}

template <int SMAX, int CH>
cudaError_t launch_few(const CombineLaunch &L, cudaStream_t st) {
  const int64_t threads = L.rows * (L.dv / (4 * CH));
  const dim3 grid((unsigned)((threads + 255) / 256));
  if (L.out_dtype == FBM_F32) return launch_pdl(k_attn_combine_few<2, SMAX, CH>, grid, dim3(256), 0, st, L);
  if (L.out_dtype == FBM_BF16) return launch_pdl(k_attn_combine_few<1, SMAX, CH>, grid, dim3(256), 0, st, L);
  return launch_pdl(k_attn_combine_few<0, SMAX, CH>, grid, dim3(256), 0, st, L);
}

}  // namespace

cudaError_t launch_combine(const CombineLaunch &L, cudaStream_t st) {
  // few splits: the per-thread kernel (its grid must fit one dimension)
  if (L.num_splits <= kSmallSplits && L.rows * (L.dv / 4) / 256 < 0x7fffffff) {
    const bool two = L.dv % 8 == 0;  // two chunks of 4 columns per thread
    if (L.num_splits <= 2) return two ? launch_few<2, 2>(L, st) : launch_few<2, 1>(L, st);
    if (L.num_splits <= 4) return two ? launch_few<4, 2>(L, st) : launch_few<4, 1>(L, st);
    return launch_few<8, 1>(L, st);
  }
  const int64_t threads = L.rows * 32;
  const dim3 grid((unsigned)((threads + 255) / 256));
  if (L.out_dtype == FBM_F32) return launch_pdl(k_attn_combine<2>, grid, dim3(256), 0, st, L);
  if (L.out_dtype == FBM_BF16) return launch_pdl(k_attn_combine<1>, grid, dim3(256), 0, st, L);
  return launch_pdl(k_attn_combine<0>, grid, dim3(256), 0, st, L);
}

}  // namespace fbm
