// Shared device helpers of libfbm (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fbm.h"

#define FBM_DEVICE __device__ __forceinline__

namespace fbm {

constexpr int kBlk = 64;  // BLKQ = BLKK = 64 tokens per block

// fp16 / bf16 element traits ------------------------------------------------
struct F16 {
  using T = __half;
  using T2 = __half2;
  static FBM_DEVICE float2 to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
  }
  static FBM_DEVICE uint32_t from_f2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  static FBM_DEVICE T from_f(float a) { return __float2half_rn(a); }
  static FBM_DEVICE uint16_t bits(float a) { return __half_as_ushort(__float2half_rn(a)); }
  static constexpr bool kIsBf16 = false;
};
struct BF16 {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  static FBM_DEVICE float2 to_f2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
  }
  static FBM_DEVICE uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  static FBM_DEVICE T from_f(float a) { return __float2bfloat16_rn(a); }
  static FBM_DEVICE uint16_t bits(float a) { return __bfloat16_as_ushort(__float2bfloat16_rn(a)); }
  static constexpr bool kIsBf16 = true;
};

FBM_DEVICE void set_error(uint32_t *err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

FBM_DEVICE uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async (16 B, zero-filled when src_bytes == 0) ---------------------------
FBM_DEVICE void cp_async16(uint32_t dst, const void *src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
FBM_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
FBM_DEVICE void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the kernel before it on the stream is still finishing; it runs
// pdl_wait() (griddepcontrol.wait: all prerequisite grids complete, their
// memory visible) before it reads that kernel's output or writes anything the
// earlier kernels read.  pdl_trigger() lets the next launch_pdl kernel start
// launching before this one ends.  Without the launch attribute both are
// no-ops.
FBM_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
FBM_DEVICE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

FBM_DEVICE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
FBM_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace fbm
