// C ABI layer of libfbm: host-side argument checks, workspace carving and
// kernel dispatch.  Every check runs before any launch; nothing is allocated
// per call.  The device error word is a file-scope __device__ variable whose
// address is looked up once per device.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fbm {
size_t decode_smem_bytes(int topk, int num_splits);
}

namespace {

__device__ uint32_t g_fbm_error_word;

thread_local char g_msg[512] = "";

fbm_status fail(fbm_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
uint32_t *g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

// device address of the error word for the current device (nullptr on failure)
uint32_t *error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fbm_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t *>(p);
  }
  return g_err_ptr[dev];
}

fbm_status cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return FBM_OK;
  return fail(FBM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t qpl, qsim, kpl, ksim, kmu, total;
};

WsLayout ws_layout(int b, int hq, int hk, int s, int d) {
  const size_t nq = (size_t)(s + 63) / 64, nk = nq;
  WsLayout w{};
  size_t off = 0;
  w.qpl = off; off = align256(off + (size_t)b * hq * fbm::plane_head_bytes((int)nq, d));
  w.qsim = off; off = align256(off + sizeof(float) * b * hq * nq);
  w.kpl = off; off = align256(off + (size_t)b * hk * fbm::plane_head_bytes((int)nk, d));
  w.ksim = off; off = align256(off + sizeof(float) * b * hk * nk);
  w.kmu = off; off = align256(off + sizeof(float) * b * hk * d);
  w.total = off;
  return w;
}

}  // namespace

namespace fbm {
// Records the calling thread's failure message (for entry points defined in
// other files of the library).
fbm_status set_message(fbm_status st, const char *msg) {
  snprintf(g_msg, sizeof(g_msg), "%s", msg);
  return st;
}
// The device error word of the current device (for other files of the library).
uint32_t *device_error_word() { return error_word(); }
}  // namespace fbm

extern "C" {

int fbm_version(void) { return 100; }

const char *fbm_last_error_message(void) { return g_msg; }

fbm_status fbm_get_error(void *stream, uint32_t *detail) {
  if (detail) *detail = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, "cudaStreamSynchronize");
  uint32_t *w = error_word();
  if (!w) return fail(FBM_ERR_CUDA, "error word lookup failed");
  uint32_t v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e, "read error word");
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_status(e, "clear error word");
  }
  if (detail) *detail = v;
  return v ? fail(FBM_ERR_DEVICE, "device error bits 0x%x", v) : FBM_OK;
}

size_t fbm_block_map_workspace_bytes(int b, int hq, int hk, int s, int d, int blkq, int blkk) {
  if (b <= 0 || hq <= 0 || hk <= 0 || s <= 0 || d <= 0 || blkq != 64 || blkk != 64) return 0;
  return ws_layout(b, hq, hk, s, d).total;
}

size_t fbm_workspace_bytes(int b, int hq, int hk, int s, int d) {
  return fbm_block_map_workspace_bytes(b, hq, hk, s, d, 64, 64);
}

namespace {

// the block map, and (q8 != NULL) the e4m3 codes of Q and K from the same pass
fbm_status block_map_impl(const void *q, const void *k, int dtype, int b, int hq, int hk, int s,
                          int d, int blkq, int blkk, const float *topk, const float *cdfthreshd,
                          const float *simthreshd1, float scale, int causal, int attention_sink,
                          int smooth_k, int32_t *lut, int32_t *lut_count, uint8_t *block_map,
                          void *workspace, size_t workspace_bytes, uint8_t *q8, float *q_scale,
                          uint8_t *k8, float *k_scale, void *stream) {
  if (!q || !k || !lut || !lut_count || !workspace || !simthreshd1)
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: null pointer argument");
  if (b <= 0 || hq <= 0 || hk <= 0 || s <= 0 || d <= 0)
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: sizes must be positive");
  if (hq % hk != 0) return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: hq %% hk != 0");
  if (hq > FBM_MAX_HEADS)
    return fail(FBM_ERR_UNSUPPORTED, "sparge_block_map: hq > %d", FBM_MAX_HEADS);
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: dtype must be f16 or bf16");
  if (blkq != 64 || blkk != 64)
    return fail(FBM_ERR_UNSUPPORTED, "sparge_block_map: blkq = blkk = 64 only");
  if (d != 64 && d != 128) return fail(FBM_ERR_UNSUPPORTED, "sparge_block_map: d in {64, 128}");
  if ((topk == nullptr) == (cdfthreshd == nullptr))
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: exactly one of topk / cdfthreshd");
  const int nq = (s + 63) / 64;
  if (nq > 1024) return fail(FBM_ERR_UNSUPPORTED, "sparge_block_map: s > 65536");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: scale must be positive and finite");
  if (!aligned16(q) || !aligned16(k) || !aligned16(workspace))
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: q, k and workspace must be 16-byte aligned");
  const WsLayout w = ws_layout(b, hq, hk, s, d);
  if (workspace_bytes < w.total)
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: workspace too small (%zu < %zu)",
                workspace_bytes, w.total);
  fbm::BlockMapLaunch L{};
  const float *sel = topk ? topk : cdfthreshd;
  for (int h = 0; h < hq; ++h) {
    if (!(sel[h] > 0.f && sel[h] <= 1.f))
      return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: %s[%d] = %g not in (0, 1]",
                  topk ? "topk" : "cdfthreshd", h, (double)sel[h]);
    if (std::isnan(simthreshd1[h]))
      return fail(FBM_ERR_INVALID_ARG, "sparge_block_map: simthreshd1[%d] is NaN", h);
    L.hp.sel[h] = sel[h];
    L.hp.theta[h] = simthreshd1[h];
  }
  L.q = q; L.k = k;
  L.bf16 = dtype == FBM_BF16;
  L.b = b; L.hq = hq; L.hk = hk; L.s = s; L.d = d; L.nq = nq; L.nk = nq;
  L.scale = scale; L.causal = causal != 0; L.sink = attention_sink != 0;
  L.mode_cdf = topk == nullptr;
  L.smooth_k = smooth_k != 0;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  L.qpl = ws + w.qpl;
  L.qsim = reinterpret_cast<float *>(ws + w.qsim);
  L.kpl = ws + w.kpl;
  L.ksim = reinterpret_cast<float *>(ws + w.ksim);
  L.kmu = reinterpret_cast<float *>(ws + w.kmu);
  L.lut = lut; L.cnt = lut_count; L.bmap = block_map;
  L.q8 = q8; L.q_scale = q_scale; L.k8 = k8; L.k_scale = k_scale;
  L.err = error_word();
  if (!L.err) return fail(FBM_ERR_CUDA, "sparge_block_map: error word lookup failed");
  return cuda_status(fbm::launch_block_map(L, static_cast<cudaStream_t>(stream)),
                     "sparge_block_map launch");
}

}  // namespace

fbm_status sparge_block_map(const void *q, const void *k, int dtype, int b, int hq, int hk,
                            int s, int d, int blkq, int blkk, const float *topk,
                            const float *cdfthreshd, const float *simthreshd1, float scale,
                            int causal, int attention_sink, int smooth_k, int32_t *lut,
                            int32_t *lut_count, uint8_t *block_map, void *workspace,
                            size_t workspace_bytes, void *stream) {
  return block_map_impl(q, k, dtype, b, hq, hk, s, d, blkq, blkk, topk, cdfthreshd, simthreshd1,
                        scale, causal, attention_sink, smooth_k, lut, lut_count, block_map,
                        workspace, workspace_bytes, nullptr, nullptr, nullptr, nullptr, stream);
}

fbm_status sparge_block_map_e4m3(const void *q, const void *k, int dtype, int b, int hq, int hk,
                                 int s, int d, int blkq, int blkk, const float *topk,
                                 const float *cdfthreshd, const float *simthreshd1, float scale,
                                 int causal, int attention_sink, int smooth_k, int32_t *lut,
                                 int32_t *lut_count, uint8_t *block_map, void *workspace,
                                 size_t workspace_bytes, uint8_t *q8, float *q_scale, uint8_t *k8,
                                 float *k_scale, void *stream) {
  if (!q8 || !q_scale || !k8 || !k_scale)
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map_e4m3: null code or scale buffer");
  if (d != 128) return fail(FBM_ERR_UNSUPPORTED, "sparge_block_map_e4m3: d = 128 only");
  if (!aligned16(q8) || !aligned16(k8))
    return fail(FBM_ERR_INVALID_ARG, "sparge_block_map_e4m3: code buffers must be 16-byte aligned");
  return block_map_impl(q, k, dtype, b, hq, hk, s, d, blkq, blkk, topk, cdfthreshd, simthreshd1,
                        scale, causal, attention_sink, smooth_k, lut, lut_count, block_map,
                        workspace, workspace_bytes, q8, q_scale, k8, k_scale, stream);
}

int fbm_fmha_kernel_kind(int dtype, int d, int dv, int num_splits, int s_q, int s_k) {
  if (dtype != FBM_F16 && dtype != FBM_BF16) return 0;
  if (d != dv || (d != 64 && d != 128) || num_splits < 1 || num_splits > 64) return 0;
  return fbm::fmha_tc_supported(d, dv, num_splits, s_q, s_k) ? 1 : 0;
}

fbm_status sparse_fmha_fwd(const void *q, const void *k, const void *v, int dtype, int b,
                           int hq, int hk, int s_q, int s_k, int d, int dv, int blkq, int blkk,
                           const int32_t *lut, const int32_t *lut_count, int lut_stride,
                           int num_splits, float scale, int causal, int key_offset,
                           float pv_threshold, void *out, float *lse, float *o_partial,
                           float *lse_partial, void *stream) {
  if (!q || !k || !v) return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: null q / k / v");
  if ((lut == nullptr) != (lut_count == nullptr))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: lut and lut_count must both be set or both NULL");
  if (b <= 0 || hq <= 0 || hk <= 0 || s_q <= 0 || s_k <= 0 || d <= 0 || dv <= 0)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: sizes must be positive");
  if (hq % hk != 0) return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: hq %% hk != 0");
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: dtype must be f16 or bf16");
  if (blkq != 64 || blkk != 64)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd: blkq = blkk = 64 only");
  if (d != dv || (d != 64 && d != 128))
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd: d = dv in {64, 128}");
  const int nq = (s_q + 63) / 64, nk = (s_k + 63) / 64;
  if (lut && lut_stride < 1)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: lut_stride must be >= 1");
  if (causal && (key_offset < -(1 << 30) || key_offset > (1 << 30)))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: |key_offset| must be at most 2^30");
  if (num_splits < 1 || num_splits > 64)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: num_splits in [1, 64]");
  const bool partial = num_splits > 1 || out == nullptr;
  if (partial && (!o_partial || !lse_partial))
    return fail(FBM_ERR_INVALID_ARG,
                num_splits > 1 ? "sparse_fmha_fwd: split mode needs o_partial and lse_partial"
                               : "sparse_fmha_fwd: null out (and no o_partial / lse_partial)");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: scale must be positive and finite");
  if (!(pv_threshold >= 0.f))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: pv_threshold must be >= 0 (+inf: off)");
  if (pv_threshold < INFINITY && partial)
    return fail(FBM_ERR_UNSUPPORTED,
                "sparse_fmha_fwd: pv_threshold needs whole rows (num_splits = 1, out given)");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (out && !aligned16(out)) ||
      (o_partial && !aligned16(o_partial)))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd: tensors must be 16-byte aligned");
  if ((long long)b * hq * nq * num_splits > 0x7fffffffLL)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd: grid too large");
  fbm::FmhaLaunch L{};
  L.q = q; L.k = k; L.v = v;
  L.bf16 = dtype == FBM_BF16;
  L.b = b; L.hq = hq; L.hk = hk; L.s_q = s_q; L.s_k = s_k; L.d = d; L.nq = nq; L.nk = nk;
  L.lut = lut; L.cnt = lut_count; L.lut_stride = lut ? lut_stride : nk;
  L.num_splits = num_splits; L.causal = causal != 0; L.scale = scale;
  L.key_offset = causal ? key_offset : 0;
  L.pv_threshold = pv_threshold;
  L.out = partial ? nullptr : out;
  L.lse = partial ? nullptr : lse;
  L.o_part = partial ? o_partial : nullptr;
  L.lse_part = partial ? lse_partial : nullptr;
  L.err = error_word();
  if (!L.err) return fail(FBM_ERR_CUDA, "sparse_fmha_fwd: error word lookup failed");
  return cuda_status(fbm::launch_fmha_tc(L, static_cast<cudaStream_t>(stream)),
                     "sparse_fmha_fwd launch");
}

fbm_status attn_combine(const float *o_part, const float *lse_part, int num_splits,
                        int64_t rows, int dv, int out_dtype, void *out, float *lse_out,
                        void *stream) {
  if (!o_part || !lse_part || !out) return fail(FBM_ERR_INVALID_ARG, "attn_combine: null pointer");
  if (num_splits < 1 || num_splits > 64)
    return fail(FBM_ERR_INVALID_ARG, "attn_combine: num_splits in [1, 64]");
  if (rows <= 0 || dv <= 0) return fail(FBM_ERR_INVALID_ARG, "attn_combine: sizes must be positive");
  if (dv % 4 != 0 || dv > 1024) return fail(FBM_ERR_UNSUPPORTED, "attn_combine: dv %% 4 == 0 and dv <= 1024");
  if (out_dtype != FBM_F16 && out_dtype != FBM_BF16 && out_dtype != FBM_F32)
    return fail(FBM_ERR_INVALID_ARG, "attn_combine: bad out_dtype");
  if (!aligned16(o_part) || !aligned16(out))
    return fail(FBM_ERR_INVALID_ARG, "attn_combine: o_part and out must be 16-byte aligned");
  if (rows > (int64_t)0x7fffffff * 8)
    return fail(FBM_ERR_UNSUPPORTED, "attn_combine: too many rows");
  fbm::CombineLaunch L{o_part, lse_part, num_splits, rows, dv, out_dtype, out, lse_out};
  return cuda_status(fbm::launch_combine(L, static_cast<cudaStream_t>(stream)),
                     "attn_combine launch");
}

fbm_status quantize_e4m3_blocks(const void *x, int dtype, int64_t bh, int s, int d,
                                uint8_t *codes, float *scales, void *stream) {
  if (!x || !codes || !scales) return fail(FBM_ERR_INVALID_ARG, "quantize_e4m3_blocks: null pointer");
  if (bh <= 0 || s <= 0) return fail(FBM_ERR_INVALID_ARG, "quantize_e4m3_blocks: sizes must be positive");
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "quantize_e4m3_blocks: dtype must be f16 or bf16");
  if (d != 128) return fail(FBM_ERR_UNSUPPORTED, "quantize_e4m3_blocks: d = 128 only");
  if (!aligned16(x) || !aligned16(codes))
    return fail(FBM_ERR_INVALID_ARG, "quantize_e4m3_blocks: x and codes must be 16-byte aligned");
  const int nb = (s + 63) / 64;
  if (bh * nb > (int64_t)0x7fffffff * 8)
    return fail(FBM_ERR_UNSUPPORTED, "quantize_e4m3_blocks: too many blocks");
  fbm::QuantLaunch L{x, dtype == FBM_BF16, s, nb, bh * nb, codes, scales};
  return cuda_status(fbm::launch_quant_e4m3(L, static_cast<cudaStream_t>(stream)),
                     "quantize_e4m3_blocks launch");
}

fbm_status sparse_fmha_fwd_fp8(const uint8_t *q8, const float *q_scale, const uint8_t *k8,
                               const float *k_scale, const void *v, int dtype, int b, int hq,
                               int hk, int s_q, int s_k, int d, int dv, const int32_t *lut,
                               const int32_t *lut_count, int lut_stride, float scale, int causal,
                               void *out, float *lse, void *stream) {
  if (!q8 || !q_scale || !k8 || !k_scale || !v || !out)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: null pointer argument");
  if ((lut == nullptr) != (lut_count == nullptr))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: lut and lut_count must both be set or both NULL");
  if (b <= 0 || hq <= 0 || hk <= 0 || s_q <= 0 || s_k <= 0)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: sizes must be positive");
  if (hq % hk != 0) return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: hq %% hk != 0");
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: dtype (of v and out) must be f16 or bf16");
  if (d != 128 || dv != 128) return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_fp8: d = dv = 128 only");
  if (causal && s_q != s_k)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_fp8: causal needs s_q == s_k");
  const int nq = (s_q + 63) / 64, nk = (s_k + 63) / 64;
  if (lut && lut_stride < 1)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: lut_stride must be >= 1");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: scale must be positive and finite");
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v) || !aligned16(out))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_fp8: tensors must be 16-byte aligned");
  if ((long long)b * hq * nq > 0x7fffffffLL)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_fp8: grid too large");
  fbm::FmhaLaunch L{};
  L.q = q8; L.k = k8; L.v = v;
  L.bf16 = dtype == FBM_BF16;
  L.b = b; L.hq = hq; L.hk = hk; L.s_q = s_q; L.s_k = s_k; L.d = d; L.nq = nq; L.nk = nk;
  L.lut = lut; L.cnt = lut_count; L.lut_stride = lut ? lut_stride : nk;
  L.num_splits = 1; L.causal = causal != 0; L.scale = scale;
  L.pv_threshold = INFINITY;
  L.q_scale = q_scale; L.k_scale = k_scale;
  L.out = out; L.lse = lse;
  L.err = error_word();
  if (!L.err) return fail(FBM_ERR_CUDA, "sparse_fmha_fwd_fp8: error word lookup failed");
  return cuda_status(fbm::launch_fmha_tc(L, static_cast<cudaStream_t>(stream)),
                     "sparse_fmha_fwd_fp8 launch (tcgen05)");
}

fbm_status lut_shard(const int32_t *lut, const int32_t *lut_count, int64_t rows, int lut_stride,
                     int lo, int hi, int32_t *out_lut, int32_t *out_count, int out_stride,
                     void *stream) {
  if (!lut || !lut_count || !out_lut || !out_count)
    return fail(FBM_ERR_INVALID_ARG, "lut_shard: null pointer");
  if (rows <= 0 || lut_stride < 1 || out_stride < 1)
    return fail(FBM_ERR_INVALID_ARG, "lut_shard: rows, lut_stride and out_stride must be positive");
  if (lo < 0 || hi <= lo)
    return fail(FBM_ERR_INVALID_ARG, "lut_shard: need 0 <= lo < hi");
  if (out_stride < hi - lo)
    return fail(FBM_ERR_INVALID_ARG, "lut_shard: out_stride (%d) < hi - lo (%d)", out_stride,
                hi - lo);
  if (rows > (int64_t)0x7fffffff * 8) return fail(FBM_ERR_UNSUPPORTED, "lut_shard: too many rows");
  fbm::LutShardLaunch L{lut, lut_count, rows, lut_stride, lo, hi, out_stride, out_lut, out_count,
                        error_word()};
  if (!L.err) return fail(FBM_ERR_CUDA, "lut_shard: error word lookup failed");
  return cuda_status(fbm::launch_lut_shard(L, static_cast<cudaStream_t>(stream)),
                     "lut_shard launch");
}

fbm_status lut_validate(const int32_t *lut, const int32_t *lut_count, int64_t rows,
                        int lut_stride, int nk, void *stream) {
  if (!lut || !lut_count) return fail(FBM_ERR_INVALID_ARG, "lut_validate: null pointer");
  if (rows <= 0 || lut_stride < 1 || nk < 1)
    return fail(FBM_ERR_INVALID_ARG, "lut_validate: rows, lut_stride and nk must be positive");
  if (rows > (int64_t)0x7fffffff * 8) return fail(FBM_ERR_UNSUPPORTED, "lut_validate: too many rows");
  fbm::LutValidateLaunch L{lut, lut_count, rows, lut_stride, nk, error_word()};
  if (!L.err) return fail(FBM_ERR_CUDA, "lut_validate: error word lookup failed");
  return cuda_status(fbm::launch_lut_validate(L, static_cast<cudaStream_t>(stream)),
                     "lut_validate launch");
}

fbm_status lut_pair_union(const int32_t *lut, const int32_t *lut_count, int64_t bh, int nq,
                          int lut_stride, int nk, int32_t *pair_lut, int32_t *pair_count,
                          int pair_stride, void *stream) {
  if (!lut || !lut_count || !pair_lut || !pair_count)
    return fail(FBM_ERR_INVALID_ARG, "lut_pair_union: null pointer");
  if (bh <= 0 || nq <= 0 || lut_stride < 1 || nk < 1)
    return fail(FBM_ERR_INVALID_ARG, "lut_pair_union: bh, nq, lut_stride and nk must be positive");
  if (nk > 1024) return fail(FBM_ERR_UNSUPPORTED, "lut_pair_union: nk <= 1024");
  if (pair_stride < nk)
    return fail(FBM_ERR_INVALID_ARG, "lut_pair_union: pair_stride (%d) < nk (%d)", pair_stride, nk);
  if (bh * ((nq + 1) / 2) > (int64_t)0x7fffffff * 8)
    return fail(FBM_ERR_UNSUPPORTED, "lut_pair_union: too many rows");
  fbm::PairUnionLaunch L{lut, lut_count, bh, nq, lut_stride, nk, pair_stride, pair_lut, pair_count,
                         error_word()};
  if (!L.err) return fail(FBM_ERR_CUDA, "lut_pair_union: error word lookup failed");
  return cuda_status(fbm::launch_lut_pair_union(L, static_cast<cudaStream_t>(stream)),
                     "lut_pair_union launch");
}

fbm_status sparse_fmha_fwd_pairs(const void *q, const void *k, const void *v, int dtype, int b,
                                 int hq, int hk, int s_q, int s_k, int d, int dv,
                                 const int32_t *pair_lut, const int32_t *pair_count,
                                 int pair_stride, float scale, int causal, int key_offset,
                                 void *out, float *lse, void *stream) {
  if (!q || !k || !v || !out)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: null q / k / v / out");
  if ((pair_lut == nullptr) != (pair_count == nullptr))
    return fail(FBM_ERR_INVALID_ARG,
                "sparse_fmha_fwd_pairs: pair_lut and pair_count must both be set or both NULL");
  if (b <= 0 || hq <= 0 || hk <= 0 || s_q <= 0 || s_k <= 0 || d <= 0 || dv <= 0)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: sizes must be positive");
  if (hq % hk != 0) return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: hq %% hk != 0");
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: dtype must be f16 or bf16");
  if (d != dv || (d != 64 && d != 128))
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_pairs: d = dv in {64, 128}");
  const int nq = (s_q + 63) / 64, nk = (s_k + 63) / 64;
  if (pair_lut && pair_stride < 1)
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: pair_stride must be >= 1");
  if (nk > (1 << 29)) return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_pairs: too many kv blocks");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: scale must be positive and finite");
  if (causal && (key_offset < -(1 << 30) || key_offset > (1 << 30)))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: |key_offset| must be at most 2^30");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(FBM_ERR_INVALID_ARG, "sparse_fmha_fwd_pairs: tensors must be 16-byte aligned");
  if ((long long)b * hq * ((nq + 1) / 2) > 0x7fffffffLL)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_fmha_fwd_pairs: grid too large");
  fbm::FmhaLaunch L{};
  L.q = q; L.k = k; L.v = v;
  L.bf16 = dtype == FBM_BF16;
  L.b = b; L.hq = hq; L.hk = hk; L.s_q = s_q; L.s_k = s_k; L.d = d; L.nq = nq; L.nk = nk;
  L.lut = pair_lut; L.cnt = pair_count; L.lut_stride = pair_lut ? pair_stride : nk;
  L.num_splits = 1; L.causal = causal != 0; L.scale = scale;
  L.key_offset = causal ? key_offset : 0;
  L.pv_threshold = INFINITY;
  L.out = out; L.lse = lse;
  L.err = error_word();
  if (!L.err) return fail(FBM_ERR_CUDA, "sparse_fmha_fwd_pairs: error word lookup failed");
  return cuda_status(fbm::launch_fmha_pair(L, static_cast<cudaStream_t>(stream)),
                     "sparse_fmha_fwd_pairs launch");
}

fbm_status sparse_decode_fwd(const void *q, const void *kv_cache, int dtype, int n_q, int hq,
                             int d, int dv, int page_size, int64_t n_pages,
                             const int32_t *page_table, int pages_per_query,
                             const int32_t *indices, int topk, int num_splits, float scale,
                             float *o_partial, float *lse_partial, void *stream) {
  if (!q || !kv_cache || !page_table || !indices || !o_partial || !lse_partial)
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: null pointer");
  if (n_q <= 0 || hq <= 0 || d <= 0 || dv <= 0 || page_size <= 0 || n_pages <= 0 ||
      pages_per_query <= 0 || topk <= 0)
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: sizes must be positive");
  if (dtype != FBM_F16 && dtype != FBM_BF16)
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: dtype must be f16 or bf16");
  if (hq != 16 || d != 576 || dv != 512 || page_size != 64)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_decode_fwd: hq = 16, d = 576, dv = 512, page_size = 64 only");
  if (num_splits < 1 || num_splits > 64)
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: num_splits in [1, 64]");
  if (n_pages * page_size > 0x7fffffffLL)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_decode_fwd: cache rows exceed int32");
  if ((int64_t)pages_per_query * page_size > 0x7fffffffLL)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_decode_fwd: positions exceed int32");
  if (fbm::decode_smem_bytes(topk, num_splits) > 227 * 1024)
    return fail(FBM_ERR_UNSUPPORTED, "sparse_decode_fwd: topk / num_splits too large for one CTA");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: scale must be positive and finite");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(o_partial))
    return fail(FBM_ERR_INVALID_ARG, "sparse_decode_fwd: q, kv_cache, o_partial must be 16-byte aligned");
  fbm::DecodeLaunch L{};
  L.q = q; L.cache = kv_cache; L.bf16 = dtype == FBM_BF16;
  L.n_q = n_q; L.hq = hq; L.d = d; L.dv = dv; L.page = page_size; L.n_pages = n_pages;
  L.page_table = page_table; L.pages_per_query = pages_per_query;
  L.idx = indices; L.topk = topk; L.num_splits = num_splits; L.scale = scale;
  L.o_part = o_partial; L.lse_part = lse_partial;
  L.err = error_word();
  if (!L.err) return fail(FBM_ERR_CUDA, "sparse_decode_fwd: error word lookup failed");
  return cuda_status(fbm::launch_decode(L, static_cast<cudaStream_t>(stream)),
                     "sparse_decode_fwd launch");
}

}  // extern "C"
