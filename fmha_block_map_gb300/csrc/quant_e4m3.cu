// fp8 (e4m3) quantisation of Q or K with one scale per 64-row block, the
// operands of the fp8 S = Q.K^T product (the "Sparge Attention (Composable
// Kernel)" README lists Q/K quantisation fused into the pool kernel as not yet
// ported; ROCm/aiter pull 6841 measures a bf16fp8 recipe).
//
// One warp per 64-row block of one (batch, head): pass 1 streams the block
// (16-byte loads, two rows per warp step) and reduces amax = max |x| in fp32;
// qscale = amax / 448 and inv = 448 / amax (IEEE round to nearest; 1 and 1 for
// an all-zero block); pass 2 reads the block again (from L2) and writes
// e4m3(x * inv), rounded to nearest even with saturation, eight codes per
// lane.  HBM-bound: 2 bytes read (plus the L2 re-read) and 1 byte written per
// element, 4 bytes of scale per block.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

template <class E>
__global__ void __launch_bounds__(256) k_quant_e4m3(const QuantLaunch L) {
  constexpr int D = 128;
  const int lane = threadIdx.x & 31;
  const int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (unit >= L.units) return;
  const int64_t bh = unit / L.nb;
  const int j = (int)(unit - bh * L.nb);
  const int row0 = j * kBlk;
  const int n = min(kBlk, L.s - row0);
  const uint16_t *src = static_cast<const uint16_t *>(L.x) + ((size_t)bh * L.s + row0) * D;
  uint8_t *dst = L.codes + ((size_t)bh * L.s + row0) * D;
  const int sub = lane & 15;   // 8 elements (16 bytes) of a row
  const int rsel = lane >> 4;  // even / odd row of the step

  float amax = 0.f;
#pragma unroll 4
  for (int r = rsel; r < n; r += 2) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)r * D) + sub);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = E::to_f2(ws[p]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  amax = warp_max(amax);
  const float qscale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  if (lane == 0) L.scales[unit] = qscale;

#pragma unroll 4
  for (int r = rsel; r < n; r += 2) {
    const uint4 w = *(reinterpret_cast<const uint4 *>(src + (size_t)r * D) + sub);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[2];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 f = E::to_f2(ws[p]);
      const float2 y = make_float2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
      const uint32_t c2 = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);  // .x low
      if (p & 1) out[p >> 1] |= c2 << 16;
      else out[p >> 1] = c2;
    }
    *(reinterpret_cast<uint2 *>(dst + (size_t)r * D) + sub) = make_uint2(out[0], out[1]);
  }
}

}  // namespace

cudaError_t launch_quant_e4m3(const QuantLaunch &L, cudaStream_t st) {
  const int64_t blocks = (L.units + 7) / 8;
  if (L.bf16) k_quant_e4m3<BF16><<<(unsigned)blocks, 256, 0, st>>>(L);
  else k_quant_e4m3<F16><<<(unsigned)blocks, 256, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace fbm
