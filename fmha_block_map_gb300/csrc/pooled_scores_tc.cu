// Pooled scores of the block map on 5th-generation tensor cores.
//
// The block map ranks kv blocks by S_ij = scale * qbar_i . kbar_j ("Sparge
// Attention (Composable Kernel)" README: pooled QK), a [nq x nk x d] product
// of fp32 block means per (batch, head).  Its result decides integer
// selections, so it must keep fp32 accuracy; bf16 tensor-core products alone
// would not.  Each fp32 operand x is therefore cut into three bf16 terms,
//   x0 = bf16(x),  x1 = bf16(x - x0),  x2 = bf16(x - x0 - x1),
// which carry its 24 significand bits, and the six products x_a y_b with
// a + b <= 2 are accumulated in fp32 (the three-term bf16 scheme of Henry,
// Tang and Heinecke, "Leveraging the bfloat16 Artificial Intelligence Datatype
// For Higher-Precision Computations", ARITH 2019); the dropped terms are below
// 2^-24 of the product.
//
// One CTA per (batch, head, 128 q blocks), 8 warps.  Per N tile of 256 kv
// blocks and per 64-wide d chunk, all threads read the fp32 means (coalesced),
// split them and write the three bf16 planes of A (128 rows) and B (256 rows)
// into shared memory in the 128-byte-swizzled K-major layout; one thread then
// issues 4 K-steps x 6 products of tcgen05.mma (M = 128, N = 256, K = 16,
// fp32 accumulator in TMEM, 256 columns).  Warps 0-3 read the accumulator
// back (lane = q block) and write scale * S into the caller's LUT buffer, which
// has exactly the size of the score matrix.
#include <atomic>
#include <climits>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {
namespace {

using namespace tc;

constexpr int kTM = 128;                 // q blocks per CTA (MMA M)
constexpr int kTN = 256;                 // kv blocks per N tile (MMA N)
constexpr int kKC = 64;                  // d values per staged chunk: 128 B of bf16 per row
constexpr int kAPlane = kTM * 128;       // one bf16 plane of A: 16 KB
constexpr int kBPlane = kTN * 128;       // one bf16 plane of B: 32 KB
constexpr int OFF_A = 0;                 // planes x0, x1, x2 of A
constexpr int OFF_B = 3 * kAPlane;       // planes y0, y1, y2 of B
constexpr int OFF_BAR = OFF_B + 3 * kBPlane;
constexpr int OFF_TMEM = OFF_BAR + 8;
constexpr int OFF_FLAG = OFF_TMEM + 4;
constexpr int SMEM_ALLOC = OFF_FLAG + 4 + 1024;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");

FBM_DEVICE uint16_t bf16_bits(__nv_bfloat16 v) { return __bfloat16_as_ushort(v); }

// x = x0 + x1 + x2 in bf16 (each difference is exact in fp32)
FBM_DEVICE void split3(float x, uint16_t &h0, uint16_t &h1, uint16_t &h2) {
  const __nv_bfloat16 b0 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(b0);
  const __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b1);
  h0 = bf16_bits(b0);
  h1 = bf16_bits(b1);
  h2 = bf16_bits(__float2bfloat16_rn(r2));
}

// Rows [0, CAP) of the fp32 matrix src ([rows, D], rows past `valid` read as
// zero), d values [d0, d0 + 64), as three bf16 planes of CAP rows of 128
// bytes in the 128-byte-swizzled K-major layout (16-byte piece c of row r at
// r * 128 + ((c ^ (r mod 8)) * 16)).  A thread's loads are all issued before
// its first split, so their latencies overlap.
template <int D, int CAP>
FBM_DEVICE void stage_split(uint8_t *planes, const float *src, int valid, int d0, int tid) {
  constexpr int kPlane = CAP * 128;
  constexpr int kTasks = CAP * 8 / kThreads;  // (row, 16-byte piece) tasks per thread
  float4 in[kTasks][2];
#pragma unroll
  for (int i = 0; i < kTasks; ++i) {
    const int task = tid + i * kThreads, r = task >> 3, c = task & 7;
    if (r < valid) {
      const float4 *p = reinterpret_cast<const float4 *>(src + (size_t)r * D + d0 + c * 8);
      in[i][0] = __ldg(p);
      in[i][1] = __ldg(p + 1);
    } else {
      in[i][0] = in[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int i = 0; i < kTasks; ++i) {
    const int task = tid + i * kThreads, r = task >> 3, c = task & 7;
    const float v[8] = {in[i][0].x, in[i][0].y, in[i][0].z, in[i][0].w,
                        in[i][1].x, in[i][1].y, in[i][1].z, in[i][1].w};
    uint32_t w[3][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint16_t a0, a1, a2, b0, b1, b2;
      split3(v[2 * e], a0, a1, a2);
      split3(v[2 * e + 1], b0, b1, b2);
      w[0][e] = (uint32_t)a0 | ((uint32_t)b0 << 16);
      w[1][e] = (uint32_t)a1 | ((uint32_t)b1 << 16);
      w[2][e] = (uint32_t)a2 | ((uint32_t)b2 << 16);
    }
    const int off = r * 128 + ((c ^ (r & 7)) << 4);
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint4 *>(planes + t * kPlane + off) =
          make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_pooled_scores_tc(const SelectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, bi = blockIdx.z;
  const int g = h / (a.hq / a.hk);
  const int i0 = blockIdx.x * kTM;
  const int nrow = min(kTM, a.nq - i0);
  const float *qbar = a.qbar + ((size_t)(bi * a.hq + h) * a.nq + i0) * D;
  const float *kbar = a.kbar + (size_t)(bi * a.hk + g) * a.nk * D;
  float *S = reinterpret_cast<float *>(a.lut) + (size_t)(bi * a.hq + h) * a.nq * a.nk;
  const uint32_t bar = sbase + OFF_BAR;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM);
  volatile int *flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    *flag = 1;
  }
  if (warp == 0) {
    tmem_alloc(sbase + OFF_TMEM, kTN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t idesc = idesc_f16(true, false, false, kTM, kTN);
  constexpr uint32_t dhi = sdesc_hi_sw128(1024);  // 8-row atoms of 1024 bytes
  uint32_t phase = 0;
  bool ok = true;
  for (int n0 = 0; n0 < a.nk && ok; n0 += kTN) {
    const int ncol = min(kTN, a.nk - n0);
    for (int d0 = 0; d0 < D && ok; d0 += kKC) {
      stage_split<D, kTM>(smem + OFF_A, qbar, nrow, d0, tid);
      stage_split<D, kTN>(smem + OFF_B, kbar + (size_t)n0 * D, ncol, d0, tid);
      fence_proxy_async();  // the planes, written by threads, are read by the tensor core
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
        // the six products x_a y_b (a + b <= 2), smaller terms first:
        // (2,0) (1,1) (0,2) (1,0) (0,1) (0,0)
#pragma unroll
        for (int ks = 0; ks < kKC / 16; ++ks)
#pragma unroll
          for (int t = 0; t < 6; ++t) {
            const int ta = t < 3 ? 2 - t : (t < 5 ? 4 - t : 0);
            const int tb = t < 3 ? t : (t < 5 ? t - 3 : 0);
            mma_f16_lo(tmem, sdesc_lo(sbase + OFF_A + ta * kAPlane + ks * 32, 16),
                       sdesc_lo(sbase + OFF_B + tb * kBPlane + ks * 32, 16), dhi, idesc,
                       (d0 > 0 || ks > 0 || t > 0) ? 1u : 0u);
          }
        mma_commit(bar);
        // the planes are restaged (and TMEM read) only after the MMAs finish
        if (!mbar_wait_for(bar, phase, kWaitNs)) {
          set_error(a.err, FBM_DEVERR_TIMEOUT);
          *flag = 0;
        }
      }
      phase ^= 1;
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      ok = *flag != 0;
    }
    if (!ok) break;
    // epilogue: warp w < 4 reads TMEM lanes 32 w .. 32 w + 31 (q blocks)
    if (warp < 4) {
      const int row = warp * 32 + lane;
      const bool vec = (a.nk & 3) == 0;
      for (int c0 = 0; c0 < ncol; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        tmem_wait_ld();
        if (row < nrow) {
          float *dst = S + (size_t)(i0 + row) * a.nk + n0 + c0;
          const int nv = min(32, ncol - c0);
          if (vec && nv == 32) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              reinterpret_cast<float4 *>(dst)[e] =
                  make_float4(a.scale * __uint_as_float(v[4 * e]), a.scale * __uint_as_float(v[4 * e + 1]),
                              a.scale * __uint_as_float(v[4 * e + 2]),
                              a.scale * __uint_as_float(v[4 * e + 3]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e < nv) dst[e] = a.scale * __uint_as_float(v[e]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM is free for the next N tile
    tc_fence_after();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, kTN);
  }
}

constexpr int kMaxDevices = 64;

template <int D>
cudaError_t launch_d(const SelectArgs &a, cudaStream_t st) {
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_pooled_scores_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev].store(true, std::memory_order_release);
  }
  dim3 grid((a.nq + kTM - 1) / kTM, a.hq, a.b);
  k_pooled_scores_tc<D><<<grid, kThreads, SMEM_ALLOC, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pooled_scores_tc(const SelectArgs &a, int d, cudaStream_t st) {
  return d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace fbm
