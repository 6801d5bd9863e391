// sparge_block_map_static: the block map with its scratch in a file-scope
// device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the library: a
// runtime that plans every device buffer before it starts and hands each
// operation only its inputs and outputs has no workspace to give, and code
// whose hot path must never enter the allocator (cudaMalloc can synchronise
// the device and takes unbounded time) cannot make one either.  This entry
// point serves them: it runs the same kernels as sparge_block_map, with
// the pooled means and self-similarities placed in g_block_map_scratch.
//
// The array is part of the library's device image, so every GPU that loads
// the library holds its FBM_STATIC_SCRATCH_BYTES until the process exits.
// Its device address is looked up once per device, by the first call made
// with that device current.  Under CUDA's lazy module loading (the default)
// that lookup may itself load this file's module and so reserve the array's
// memory: make one warm-up call per device at start-up, outside any stream
// capture and outside the hot path.
// All calls share the one array and nothing in it needs to start at zero (the
// pooling kernel overwrites every byte the later kernels read), so calls that overlap
// on the GPU, e.g. on two streams, race on it.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fbm {
fbm_status set_message(fbm_status st, const char *msg);
}

namespace {

__device__ __align__(256) uint8_t g_block_map_scratch[FBM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void *g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// device address of the scratch array on the current device, or nullptr
void *scratch_address(cudaError_t *err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDev) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_block_map_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" fbm_status sparge_block_map_static(const void *q, const void *k, int dtype, int b,
                                              int hq, int hk, int s, int d, int blkq, int blkk,
                                              const float *topk, const float *cdfthreshd,
                                              const float *simthreshd1, float scale, int causal,
                                              int attention_sink, int smooth_k, int32_t *lut,
                                              int32_t *lut_count, uint8_t *block_map,
                                              void *stream) {
  const size_t need = fbm_block_map_workspace_bytes(b, hq, hk, s, d, blkq, blkk);
  if (need > FBM_STATIC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "sparge_block_map_static: this shape needs %zu bytes of scratch, more than the "
             "%u-byte static array; use sparge_block_map with a workspace",
             need, (unsigned)FBM_STATIC_SCRATCH_BYTES);
    return fbm::set_message(FBM_ERR_UNSUPPORTED, msg);
  }
  cudaError_t err = cudaSuccess;
  void *ws = scratch_address(&err);
  if (!ws) {
    char msg[256];
    snprintf(msg, sizeof(msg), "sparge_block_map_static: scratch address lookup failed: %s",
             cudaGetErrorString(err));
    return fbm::set_message(FBM_ERR_CUDA, msg);
  }
  return sparge_block_map(q, k, dtype, b, hq, hk, s, d, blkq, blkk, topk, cdfthreshd, simthreshd1,
                          scale, causal, attention_sink, smooth_k, lut, lut_count, block_map, ws,
                          FBM_STATIC_SCRATCH_BYTES, stream);
}
