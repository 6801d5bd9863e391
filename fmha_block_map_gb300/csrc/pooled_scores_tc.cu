// Pooled scores of the block map on 5th-generation tensor cores.
//
// The block map ranks kv blocks by S_ij = scale * qbar_i . kbar_j ("Sparge
// Attention (Composable Kernel)" README: pooled QK), a [nq x nk x d] product
// of fp32 block means per (batch, head).  Its result decides integer
// selections, so it must keep fp32 accuracy; bf16 tensor-core products alone
// would not.  The pooling kernel therefore leaves each fp32 mean x as three
// bf16 terms x = x0 + x1 + x2 (kernels.h: the split planes), and this kernel
// accumulates the six products x_a y_b with a + b <= 2 in fp32 (the
// three-term bf16 scheme of Henry, Tang and Heinecke, "Leveraging the bfloat16
// Artificial Intelligence Datatype For Higher-Precision Computations",
// ARITH 2019); the dropped terms are below 2^-24 of the product.
//
// One CTA per (batch, head, 128 q blocks, 128 kv blocks), 8 warps, two CTAs
// per SM (96 KB of shared memory).  The planes are already in the
// 128-byte-swizzled K-major layout the MMA reads, so per 64-wide d chunk one
// thread fetches the three planes of A (128 q blocks) and of B (128 kv
// blocks) with two bulk copies (48 KB each), then issues 4 K-steps x 6
// products of tcgen05.mma (M = 128, N = 128, K = 16, fp32 accumulator in
// TMEM, 128 columns).  Epilogue: warp w reads TMEM lanes 32 (w mod 4) .. +31
// (q blocks) and columns 64 (w / 4) .. +63 (kv blocks) and writes scale * S
// into shared memory (rows padded to 528 bytes, so the stores of 32 rows hit
// distinct banks); then each warp writes whole rows of the tile to the
// caller's LUT buffer, which has exactly the size of the score matrix.  Under
// the causal mask a tile stops at the last kv block its last q block may see,
// and tiles wholly past it exit at once.
#include <atomic>
#include <climits>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {
namespace {

using namespace tc;

constexpr int kTM = 128;                           // q blocks per CTA (MMA M)
constexpr int kTN = 128;                           // kv blocks per CTA (MMA N)
constexpr int kKC = 64;                            // d values per chunk: 128 B of bf16 per row
constexpr int OFF_A = 0;                           // planes x0, x1, x2 of A
constexpr int OFF_B = (int)(3 * kPlaneBytes);      // planes y0, y1, y2 of B
constexpr int kSPitch = kTN + 4;                   // floats per staged row of S (528 bytes)
constexpr int OFF_BAR = (int)(6 * kPlaneBytes);    // 96 KB
constexpr int OFF_TMEM = OFF_BAR + 16;
constexpr int OFF_FLAG = OFF_TMEM + 4;
constexpr int SMEM_ALLOC = OFF_FLAG + 4 + 1024;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(kTM * kSPitch * 4 <= OFF_BAR, "the staged S tile fits in the plane buffers");
static_assert(kTN == kPlaneRows && kTM == kPlaneRows, "one plane tile per operand");
static_assert(2 * (SMEM_ALLOC + 1024) <= 228 * 1024, "two CTAs per SM");

template <int D>
__global__ void __launch_bounds__(kThreads, 2) k_pooled_scores_tc(const SelectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntn = (a.nk + kTN - 1) / kTN;
  const int h = blockIdx.y, bi = blockIdx.z;
  const int g = h / (a.hq / a.hk);
  const int tq = blockIdx.x / ntn, tn = blockIdx.x % ntn;
  const int i0 = tq * kTM, n0 = tn * kTN;
  const int nrow = min(kTM, a.nq - i0);
  // causal: no row of this tile reads a kv block past the last one its last
  // q block may see (the selection reads eligible columns only)
  const int kv_end = a.causal ? min(a.nk, ((i0 + nrow) * a.blkq - 1) / a.blkk + 1) : a.nk;
  if (n0 >= kv_end) return;  // uniform over the CTA, before any barrier or allocation
  const int ncol = min(kTN, kv_end - n0);
  const uint8_t *pa = a.qpl + (size_t)(bi * a.hq + h) * plane_head_bytes(a.nq, D) +
                      (size_t)tq * plane_tile_bytes(D);
  const uint8_t *pb = a.kpl + (size_t)(bi * a.hk + g) * plane_head_bytes(a.nk, D) +
                      (size_t)tn * plane_tile_bytes(D);
  float *S = reinterpret_cast<float *>(a.lut) + (size_t)(bi * a.hq + h) * a.nq * a.nk;
  const uint32_t full = sbase + OFF_BAR, done = sbase + OFF_BAR + 8;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM);
  volatile int *flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
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
  // the setup above overlaps the pooling kernel's tail; its planes are read
  // (and this tile written) only after it completes
  pdl_trigger();
  pdl_wait();
  if (warp == 0) {
    // the whole warp runs the loop; one lane issues the copies, one elected
    // lane each MMA (issued from a lone lane in a divergent branch, the 24 MMAs
    // of a chunk took about twice their execution time)
    constexpr uint32_t idesc = idesc_f16(true, false, false, kTM, kTN);
    constexpr uint32_t dhi = sdesc_hi_sw128(1024);  // 8-row atoms of 1024 bytes
    constexpr uint32_t kChunk = (uint32_t)(3 * kPlaneBytes);
    bool ok = true;
    for (int c = 0; c < D / kKC; ++c) {
      // the chunk's planes of A and B: two bulk copies on one barrier
      if (lane == 0) {
        mbar_arrive_tx(full, 2 * kChunk);
        bulk_load(sbase + OFF_A, pa + (size_t)c * kChunk, kChunk, full);
        bulk_load(sbase + OFF_B, pb + (size_t)c * kChunk, kChunk, full);
      }
      __syncwarp();
      if (!mbar_wait_for_w(full, c & 1, kWaitNs)) {
        ok = false;
        mbar_wait_for_w(full, c & 1, kWaitNs);  // drain the copies in flight (bounded)
        break;
      }
      tc_fence_after();
      // the six products x_a y_b (a + b <= 2), smaller terms first:
      // (2,0) (1,1) (0,2) (1,0) (0,1) (0,0)
#pragma unroll
      for (int ks = 0; ks < kKC / 16; ++ks)
#pragma unroll
        for (int t = 0; t < 6; ++t) {
          const int ta = t < 3 ? 2 - t : (t < 5 ? 4 - t : 0);
          const int tb = t < 3 ? t : (t < 5 ? t - 3 : 0);
          mma_f16_lo_w(tmem, sdesc_lo(sbase + OFF_A + ta * (uint32_t)kPlaneBytes + ks * 32, 16),
                       sdesc_lo(sbase + OFF_B + tb * (uint32_t)kPlaneBytes + ks * 32, 16), dhi, idesc,
                       (c > 0 || ks > 0 || t > 0) ? 1u : 0u);
        }
      mma_commit_w(done);
      // the planes are refilled (and TMEM read) only after the MMAs finish
      if (!mbar_wait_for_w(done, c & 1, kWaitNs)) {
        ok = false;
        mbar_wait_for_w(done, c & 1, kWaitNs);  // drain the MMAs in flight (bounded)
        break;
      }
    }
    if (!ok && lane == 0) {
      set_error(a.err, FBM_DEVERR_TIMEOUT);
      *flag = 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*flag) {  // uniform over the CTA
    // TMEM -> padded rows in shared memory (the plane buffers are free now)
    float *stage = reinterpret_cast<float *>(smem);
    const int row = (warp & 3) * 32 + lane;
    const int cbase = (warp >> 2) * 64;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c0 = cbase + 32 * half;
      if (c0 >= ncol) break;  // uniform over the warp
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)c0, v);
      tmem_wait_ld();
      float4 *dst = reinterpret_cast<float4 *>(stage + row * kSPitch + c0);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        dst[e] = make_float4(a.scale * __uint_as_float(v[4 * e]), a.scale * __uint_as_float(v[4 * e + 1]),
                             a.scale * __uint_as_float(v[4 * e + 2]),
                             a.scale * __uint_as_float(v[4 * e + 3]));
    }
    // whole rows of the tile.  Aligned full rows leave as bulk copies (one per
    // row, issued by lanes 0-15 of every warp, asynchronous: the row loop of
    // 16-byte stores took ~4000 cycles per tile); otherwise plain stores.
    const bool bulk = ncol % 4 == 0 && (a.nk & 3) == 0 && (reinterpret_cast<uintptr_t>(S) & 15) == 0;
    if (bulk) fence_proxy_async();  // this thread's staged values, for the async proxy
    __syncthreads();
    if (bulk) {
      const int r = warp * 16 + lane;  // 8 warps x 16 lanes = the 128 rows of a full tile
      if (lane < 16 && r < nrow) {
        bulk_store(S + (size_t)(i0 + r) * a.nk + n0, smem_u32(stage + r * kSPitch), (uint32_t)ncol * 4);
        bulk_commit();
        bulk_wait_read0();  // the staged row is read before the CTA leaves
      }
    } else {
      for (int r = warp; r < nrow; r += kThreads / 32) {
        float *grow = S + (size_t)(i0 + r) * a.nk + n0;
        const float *srow = stage + r * kSPitch;
        for (int c = lane; c < ncol; c += 32) grow[c] = srow[c];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
  dim3 grid(((a.nq + kTM - 1) / kTM) * ((a.nk + kTN - 1) / kTN), a.hq, a.b);
  return launch_pdl(k_pooled_scores_tc<D>, grid, dim3(kThreads), SMEM_ALLOC, st, a);
}

}  // namespace

cudaError_t launch_pooled_scores_tc(const SelectArgs &a, int d, cudaStream_t st) {
  return d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace fbm
