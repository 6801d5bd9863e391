// Sparse FMHA forward with warp-level mma.sync (m16n8k16, fp32 accumulate).
//
// One CTA of 4 warps per (batch, head, q block, split); each warp owns 16 query
// rows.  The kv blocks listed in the q block's LUT row (or every kv block in
// dense mode) are streamed through a double-buffered cp.async pipeline into
// XOR-swizzled shared memory; S = Q K^T and O += P V run on mma.sync with an
// online softmax in the base-2 domain (scale * log2(e) folded into one FMA).
// This is the d = 64 path (whole rows, split-KV and fp32 partials); the
// tcgen05 kernel covers d = 128.
//
// Loop shape: the per-row-block loop over a block list of the
// Incremental_FlashAttention updating_log, Stage 3 (prefetch the next listed
// K/V tile while the current one is consumed; an empty list writes O = 0 and
// LSE = -inf).
#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

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

// byte offset of 16-byte chunk `ch` of row `r` in a swizzled [64][D] tile
template <int D>
FBM_DEVICE uint32_t swz(int r, int ch) {
  return (uint32_t)(r * (D * 2) + ((ch ^ (r & 7)) << 4));
}

template <int D>
FBM_DEVICE void load_tile(uint32_t dst, const uint16_t *src, int row0, int nrows_valid, bool ok) {
  constexpr int CH = D / 8;
  for (int c = threadIdx.x; c < kBlk * CH; c += 128) {
    const int r = c / CH, ch = c % CH;
    const bool valid = ok && r < nrows_valid;
    const uint16_t *g = src + (size_t)(valid ? row0 + r : 0) * D + ch * 8;
    cp_async16(dst + swz<D>(r, ch), g, valid);
  }
}

template <class E, int D, bool SPLIT>
__global__ void __launch_bounds__(128) k_fmha_mma(const FmhaLaunch L) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int TILE = kBlk * D * 2;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + TILE;          // 2 stages
  const uint32_t sV = sQ + 3 * TILE;      // 2 stages
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int unit = blockIdx.x;
  const int split = unit % L.num_splits;
  unit /= L.num_splits;
  const int i = unit % L.nq;
  unit /= L.nq;
  const int h = unit % L.hq;
  const int bi = unit / L.hq;
  const int g = h / (L.hq / L.hk);

  const uint16_t *q = static_cast<const uint16_t *>(L.q) + ((size_t)(bi * L.hq + h) * L.s_q) * D;
  const uint16_t *k = static_cast<const uint16_t *>(L.k) + ((size_t)(bi * L.hk + g) * L.s_k) * D;
  const uint16_t *v = static_cast<const uint16_t *>(L.v) + ((size_t)(bi * L.hk + g) * L.s_k) * D;

  // the kv-block list of this (q block, split)
  const int32_t *lut_row = nullptr;
  int n_list;
  if (L.lut) {
    const size_t row = (size_t)(bi * L.hq + h) * L.nq + i;
    lut_row = L.lut + row * L.lut_stride;
    n_list = L.cnt[row];
    if (n_list < 0 || n_list > L.nk || n_list > L.lut_stride) {
      if (threadIdx.x == 0) set_error(L.err, FBM_DEVERR_LUT_RANGE);
      n_list = max(0, min(n_list, min(L.nk, L.lut_stride)));
    }
  } else {
    n_list = L.causal ? min(L.nk, (i * kBlk + kBlk - 1) / kBlk + 1) : L.nk;
  }
  const int base = n_list / L.num_splits, extra = n_list % L.num_splits;
  const int lo = split * base + min(split, extra);
  const int n = base + (split < extra ? 1 : 0);

  const int q_row0 = i * kBlk;
  const int q_rows = min(kBlk, L.s_q - q_row0);
  // kv block of entry t of this chunk, or -1 for an unusable LUT entry
  // (lut_entry: out of range, or not above the entry before it)
  auto block_of = [&](int t, uint32_t *why) -> int {
    if (!lut_row) {
      *why = 0;
      return lo + t;
    }
    return lut_entry(lut_row, lo + t, L.nk, why);
  };

  float o[D / 8][4];
#pragma unroll
  for (int a = 0; a < D / 8; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const float sl2 = L.scale * 1.4426950408889634f;

  if (n > 0) {
    load_tile<D>(sQ, q, q_row0, q_rows, true);
    {
      uint32_t why;
      const int j0 = block_of(0, &why);
      const bool ok = j0 >= 0;
      load_tile<D>(sK, k, j0 * kBlk, ok ? L.s_k - j0 * kBlk : 0, ok);
      load_tile<D>(sV, v, j0 * kBlk, ok ? L.s_k - j0 * kBlk : 0, ok);
    }
    cp_async_commit();
    uint32_t qf[D / 16][4];
    for (int t = 0; t < n; ++t) {
      const int stage = t & 1;
      if (t + 1 < n) {
        uint32_t why;
        const int jn = block_of(t + 1, &why);
        const bool ok = jn >= 0;
        load_tile<D>(sK + (stage ^ 1) * TILE, k, jn * kBlk, ok ? L.s_k - jn * kBlk : 0, ok);
        load_tile<D>(sV + (stage ^ 1) * TILE, v, jn * kBlk, ok ? L.s_k - jn * kBlk : 0, ok);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      if (t == 0) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ldsm_x4(sQ + swz<D>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)), qf[ks][0], qf[ks][1],
                  qf[ks][2], qf[ks][3]);
      }
      uint32_t why;
      const int j = block_of(t, &why);
      const bool jok = j >= 0;
      if (!jok && threadIdx.x == 0) set_error(L.err, why);
      const uint32_t kt = sK + stage * TILE, vt = sV + stage * TILE;
      // S = Q K^T (16 rows x 64 keys per warp)
      float s[8][4];
#pragma unroll
      for (int a = 0; a < 8; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int mi = lane >> 3;
          const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt + swz<D>(key, ks * 2 + (mi & 1)), b0, b1, b2, b3);
          mma16816<E>(s[2 * np], qf[ks], b0, b1);
          mma16816<E>(s[2 * np + 1], qf[ks], b2, b3);
        }
      }
      // masks: keys past s_k, causal, invalid LUT entries
      const int key0 = j * kBlk;
      const int row_a = q_row0 + warp * 16 + (lane >> 2);
      const bool need_mask = !jok || key0 + kBlk > L.s_k || (L.causal && key0 + kBlk - 1 > q_row0);
      if (need_mask) {
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int key = key0 + a * 8 + (lane & 3) * 2 + (c & 1);
            const int row = row_a + (c >= 2 ? 8 : 0);
            if (!jok || key >= L.s_k || (L.causal && key > row)) s[a][c] = -INFINITY;
          }
      }
      // online softmax (base 2)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mx = -INFINITY;
#pragma unroll
        for (int a = 0; a < 8; ++a) mx = fmaxf(mx, fmaxf(s[a][2 * r], s[a][2 * r + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_r[r], mx * sl2);
        const float base = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m_r[r] - base);
        m_r[r] = m_new;
        float ls = 0.f;
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          s[a][2 * r] = exp2f(fmaf(s[a][2 * r], sl2, -base));
          s[a][2 * r + 1] = exp2f(fmaf(s[a][2 * r + 1], sl2, -base));
          ls += s[a][2 * r] + s[a][2 * r + 1];
        }
        l_r[r] = l_r[r] * alpha + ls;
#pragma unroll
        for (int a = 0; a < D / 8; ++a) {
          o[a][2 * r] *= alpha;
          o[a][2 * r + 1] *= alpha;
        }
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = E::from_f2(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = E::from_f2(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = E::from_f2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = E::from_f2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int mi = lane >> 3;
          const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vt + swz<D>(key, dp * 2 + (mi >> 1)), b0, b1, b2, b3);
          mma16816<E>(o[2 * dp], pa, b0, b1);
          mma16816<E>(o[2 * dp + 1], pa, b2, b3);
        }
      }
      __syncthreads();
    }
  }
  // epilogue: O / l, LSE = m ln2 + ln l
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_r[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const bool live = l > 0.f;
    const float inv = live ? 1.0f / l : 0.f;
    const int row = q_row0 + warp * 16 + (lane >> 2) + r * 8;
    if (row < L.s_q) {
      const size_t orow = (size_t)(bi * L.hq + h) * L.s_q + row;
      const float lse = live ? m_r[r] * 0.6931471805599453f + logf(l) : -INFINITY;
      if constexpr (SPLIT) {
        const size_t plane = (size_t)L.b * L.hq * L.s_q;
        float *dst = L.o_part + ((size_t)split * plane + orow) * D;
#pragma unroll
        for (int a = 0; a < D / 8; ++a) {
          const int col = a * 8 + (lane & 3) * 2;
          *reinterpret_cast<float2 *>(dst + col) = make_float2(o[a][2 * r] * inv, o[a][2 * r + 1] * inv);
        }
        if ((lane & 3) == 0) L.lse_part[(size_t)split * plane + orow] = lse;
      } else {
        uint16_t *dst = static_cast<uint16_t *>(L.out) + orow * D;
#pragma unroll
        for (int a = 0; a < D / 8; ++a) {
          const int col = a * 8 + (lane & 3) * 2;
          *reinterpret_cast<uint32_t *>(dst + col) = E::from_f2(o[a][2 * r] * inv, o[a][2 * r + 1] * inv);
        }
        if (L.lse && (lane & 3) == 0) L.lse[orow] = lse;
      }
    }
  }
}

template <class E, int D, bool SPLIT>
cudaError_t launch3(const FmhaLaunch &L, cudaStream_t st) {
  const int smem = 5 * kBlk * D * 2;
  cudaError_t e = cudaFuncSetAttribute(k_fmha_mma<E, D, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)L.b * L.hq * L.nq * L.num_splits;
  k_fmha_mma<E, D, SPLIT><<<(unsigned)grid, 128, smem, st>>>(L);
  return cudaGetLastError();
}

template <class E, int D>
cudaError_t launch2(const FmhaLaunch &L, cudaStream_t st) {
  // fp32 partials for a split, or for one whole row when the caller asks for
  // them instead of out (num_splits = 1, out = NULL)
  const bool partial = L.num_splits > 1 || L.out == nullptr;
  return partial ? launch3<E, D, true>(L, st) : launch3<E, D, false>(L, st);
}

}  // namespace

cudaError_t launch_fmha_mma(const FmhaLaunch &L, cudaStream_t st) {
  if (L.bf16) return L.d == 128 ? launch2<BF16, 128>(L, st) : launch2<BF16, 64>(L, st);
  return L.d == 128 ? launch2<F16, 128>(L, st) : launch2<F16, 64>(L, st);
}

}  // namespace fbm
