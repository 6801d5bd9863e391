// Sparse decode over per-query token index lists through a page table
// (ROCm/aiter pull 4919: sparse MLA decode; a K row holds 512 latent + 64
// rotary values and V is its latent plane; split-KV partials).
//
// One CTA (4 warps) per (query, split).  Prologue: the CTA resolves every
// listed token of its chunk to a physical cache row (index list, then page
// table) into shared memory before any row is fetched, so the dependent
// lookups are off the streaming loop.  Main loop over tiles of 32 tokens:
//   - cp.async gathers the 32 rows (1152 B each) into a double-buffered,
//     XOR-swizzled shared tile (a sentinel or invalid token is zero-filled and
//     masked);
//   - S = Q K^T [16 heads x 32 tokens] on mma.sync, the 576-wide contraction
//     split over the 4 warps (each keeps its 144-column slice of Q in
//     registers) and summed in a fixed order through shared memory;
//   - online softmax per head (base 2); P goes to shared memory as the A
//     operand of O += P V, whose 512 output columns are split over the warps.
// The 16 heads share each gathered row, so every selected row is read once
// per query: the kernel is bound by HBM bandwidth.
#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

constexpr int kDTok = 32;     // tokens per tile
constexpr int kDHeads = 16;   // query heads (the MMA M dimension)

template <class E>
FBM_DEVICE void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (E::kIsBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
FBM_DEVICE void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
FBM_DEVICE void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <int D>
FBM_DEVICE uint32_t swz(int r, int ch) {
  return (uint32_t)(r * (D * 2) + ((ch ^ (r & 7)) << 4));
}

template <class E, int D, int DV>
__global__ void __launch_bounds__(128) k_sparse_decode(const DecodeLaunch L) {
  static_assert(D % 64 == 0 && DV % 64 == 0 && DV <= D, "shape");
  constexpr int KS_PER_WARP = D / 64;          // 16-wide k-steps per warp for S
  constexpr int TILE = kDTok * D * 2;
  constexpr int P_LD = kDTok + 8;              // padded P row (elements)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *p = smem;
  const uint32_t sQ = smem_u32(p);               p += kDHeads * D * 2;
  const uint32_t sKV = smem_u32(p);              p += 2 * TILE;
  float *s_part = reinterpret_cast<float *>(p);  p += 4 * kDHeads * kDTok * sizeof(float);
  uint16_t *s_p = reinterpret_cast<uint16_t *>(p); p += kDHeads * P_LD * 2;
  float *s_alpha = reinterpret_cast<float *>(p); p += kDHeads * sizeof(float);
  float *s_l = reinterpret_cast<float *>(p);     p += kDHeads * sizeof(float);
  int32_t *s_rows = reinterpret_cast<int32_t *>(p);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int split = blockIdx.x % L.num_splits;
  const int c = blockIdx.x / L.num_splits;
  const int base = L.topk / L.num_splits, extra = L.topk % L.num_splits;
  const int lo = split * base + min(split, extra);
  const int n = base + (split < extra ? 1 : 0);
  const uint16_t *cache = static_cast<const uint16_t *>(L.cache);
  const int max_pos = L.pages_per_query * L.page;

  // prologue: token list -> physical rows (-1 = masked)
  for (int t = tid; t < n; t += 128) {
    const int pos = __ldg(L.idx + (size_t)c * L.topk + lo + t);
    int row = -1;
    if (pos >= 0) {
      if (pos < max_pos) {
        const int pg = __ldg(L.page_table + (size_t)c * L.pages_per_query + pos / L.page);
        if (pg >= 0 && pg < L.n_pages) row = pg * L.page + pos % L.page;
        else set_error(L.err, FBM_DEVERR_LUT_RANGE);
      } else {
        set_error(L.err, FBM_DEVERR_LUT_RANGE);
      }
    }
    s_rows[t] = row;
  }
  // Q [16][D]
  {
    const uint16_t *qg = static_cast<const uint16_t *>(L.q) + (size_t)c * L.hq * D;
    for (int ch = tid; ch < kDHeads * (D / 8); ch += 128) {
      const int r = ch / (D / 8), cc = ch % (D / 8);
      cp_async16(sQ + swz<D>(r, cc), qg + (size_t)r * D + cc * 8, true);
    }
  }
  __syncthreads();
  auto load_tile = [&](int tile, int stage) {
    const uint32_t dst = sKV + stage * TILE;
    for (int ch = tid; ch < kDTok * (D / 8); ch += 128) {
      const int r = ch / (D / 8), cc = ch % (D / 8);
      const int tok = tile * kDTok + r;
      const int row = tok < n ? s_rows[tok] : -1;
      const bool ok = row >= 0;
      cp_async16(dst + swz<D>(r, cc), cache + (size_t)(ok ? row : 0) * D + cc * 8, ok);
    }
  };
  const int ntiles = (n + kDTok - 1) / kDTok;
  if (ntiles > 0) load_tile(0, 0);
  cp_async_commit();

  float o[DV / 4 / 8][4];  // this warp's DV/4 columns: DV/32 n-tiles
#pragma unroll
  for (int a = 0; a < DV / 32; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
  // softmax role: thread -> head tid/8, tokens (tid%8)*4 .. +3
  const int sm_head = tid >> 3, sm_tok = (tid & 7) * 4;
  float m_run = -INFINITY, l_run = 0.f;
  const float sl2 = L.scale * 1.4426950408889634f;
  uint32_t qf[KS_PER_WARP][4];

  for (int t = 0; t < ntiles; ++t) {
    const int stage = t & 1;
    if (t + 1 < ntiles) {
      load_tile(t + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int ks = 0; ks < KS_PER_WARP; ++ks) {
        const int ch = (warp * KS_PER_WARP + ks) * 2 + (lane >> 4);
        ldsm_x4(sQ + swz<D>(lane & 15, ch), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const uint32_t kv = sKV + stage * TILE;
    // partial S over this warp's slice of the contraction
    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS_PER_WARP; ++ks) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int mi = lane >> 3;
        const int tok = np * 16 + (mi >> 1) * 8 + (lane & 7);
        const int ch = (warp * KS_PER_WARP + ks) * 2 + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kv + swz<D>(tok, ch), b0, b1, b2, b3);
        mma16816<E>(s[2 * np], qf[ks], b0, b1);
        mma16816<E>(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
    float *sp = s_part + warp * kDHeads * kDTok;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int head = (lane >> 2) + (cc >= 2 ? 8 : 0);
        const int tok = a * 8 + (lane & 3) * 2 + (cc & 1);
        sp[head * kDTok + tok] = s[a][cc];
      }
    __syncthreads();
    // online softmax for (sm_head, 4 tokens)
    {
      float x[4];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tok = sm_tok + u;
        const int gtok = t * kDTok + tok;
        float v = s_part[sm_head * kDTok + tok] + s_part[kDHeads * kDTok + sm_head * kDTok + tok] +
                  s_part[2 * kDHeads * kDTok + sm_head * kDTok + tok] +
                  s_part[3 * kDHeads * kDTok + sm_head * kDTok + tok];
        if (gtok >= n || s_rows[gtok] < 0) v = -INFINITY;
        x[u] = v;
        mx = fmaxf(mx, v);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      const float m_new = fmaxf(m_run, mx * sl2);
      const float b = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_run - b);
      m_run = m_new;
      float ls = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = exp2f(fmaf(x[u], sl2, -b));
        ls += x[u];
      }
      l_run = l_run * alpha + ls;
      uint2 pk = make_uint2(E::from_f2(x[0], x[1]), E::from_f2(x[2], x[3]));
      *reinterpret_cast<uint2 *>(s_p + sm_head * P_LD + sm_tok) = pk;
      if ((tid & 7) == 0) s_alpha[sm_head] = alpha;
    }
    __syncthreads();
    // O = alpha * O + P V over this warp's DV/4 columns
    {
      const float a0 = s_alpha[lane >> 2], a1 = s_alpha[(lane >> 2) + 8];
#pragma unroll
      for (int a = 0; a < DV / 32; ++a) {
        o[a][0] *= a0; o[a][1] *= a0; o[a][2] *= a1; o[a][3] *= a1;
      }
      const uint32_t sP = smem_u32(s_p);
#pragma unroll
      for (int kk = 0; kk < kDTok / 16; ++kk) {
        uint32_t pa[4];
        ldsm_x4(sP + (lane & 15) * (P_LD * 2) + (kk * 2 + (lane >> 4)) * 16, pa[0], pa[1], pa[2],
                pa[3]);
#pragma unroll
        for (int dp = 0; dp < DV / 64; ++dp) {
          const int mi = lane >> 3;
          const int tok = kk * 16 + (mi & 1) * 8 + (lane & 7);
          const int ch = (warp * (DV / 4) + dp * 16) / 8 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(kv + swz<D>(tok, ch), b0, b1, b2, b3);
          mma16816<E>(o[2 * dp], pa, b0, b1);
          mma16816<E>(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  // epilogue
  {
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    if ((tid & 7) == 0) {
      s_l[sm_head] = l;
      const bool live = l > 0.f;
      L.lse_part[((size_t)split * L.n_q + c) * kDHeads + sm_head] =
          live ? m_run * 0.6931471805599453f + logf(l) : -INFINITY;
    }
  }
  __syncthreads();
  const float l0 = s_l[lane >> 2], l1 = s_l[(lane >> 2) + 8];
  const float i0 = l0 > 0.f ? 1.0f / l0 : 0.f, i1 = l1 > 0.f ? 1.0f / l1 : 0.f;
  float *dst = L.o_part + ((size_t)split * L.n_q + c) * kDHeads * DV;
#pragma unroll
  for (int a = 0; a < DV / 32; ++a) {
    const int col = warp * (DV / 4) + a * 8 + (lane & 3) * 2;
    const int h0 = lane >> 2;
    *reinterpret_cast<float2 *>(dst + (size_t)h0 * DV + col) = make_float2(o[a][0] * i0, o[a][1] * i0);
    *reinterpret_cast<float2 *>(dst + (size_t)(h0 + 8) * DV + col) =
        make_float2(o[a][2] * i1, o[a][3] * i1);
  }
}

template <class E, int D, int DV>
size_t decode_smem(int chunk) {
  return (size_t)kDHeads * D * 2 + 2 * (size_t)kDTok * D * 2 + 4 * kDHeads * kDTok * 4 +
         kDHeads * (kDTok + 8) * 2 + 2 * kDHeads * 4 + (size_t)chunk * 4;
}

template <class E>
cudaError_t launch_e(const DecodeLaunch &L, cudaStream_t st) {
  const int chunk = (L.topk + L.num_splits - 1) / L.num_splits;
  const size_t smem = decode_smem<E, 576, 512>(chunk);
  cudaError_t e = cudaFuncSetAttribute(k_sparse_decode<E, 576, 512>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_sparse_decode<E, 576, 512><<<L.n_q * L.num_splits, 128, smem, st>>>(L);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int topk, int num_splits) {
  return decode_smem<BF16, 576, 512>((topk + num_splits - 1) / num_splits);
}

cudaError_t launch_decode(const DecodeLaunch &L, cudaStream_t st) {
  return L.bf16 ? launch_e<BF16>(L, st) : launch_e<F16>(L, st);
}

}  // namespace fbm
