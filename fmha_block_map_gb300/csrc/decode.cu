// Sparse decode over per-query token index lists through a page table
// (ROCm/aiter pull 4919: sparse MLA decode; a K row holds 512 latent + 64
// rotary values and V is its latent plane; split-KV partials).
//
// One CTA (two groups of 4 warps) per (query, split).  Prologue: the CTA
// resolves every listed token of its chunk to a physical cache row (index
// list, then page table) into shared memory before any row is fetched, so the
// dependent lookups are off the streaming loop, and stages Q.  The two warp
// groups then work independently, group g on the 16-token tiles g, g + 2, ...
// of the chunk, each with its own online-softmax state; per tile:
//   - cp.async gathers the 16 rows (1152 B each) into the group's
//     double-buffered, XOR-swizzled shared tile (a sentinel or invalid token
//     is zero-filled and masked);
//   - S = Q K^T [16 heads x 16 tokens] on mma.sync, the 576-wide contraction
//     split over the group's 4 warps and summed in a fixed order through
//     shared memory;
//   - online softmax per head (base 2); P goes to shared memory as the A
//     operand of O += P V, whose 512 output columns are split over the warps.
// At the end the two groups' states merge like two split-KV partials (the
// Stage 1 combine of "Incremental_FlashAttention updating_log.md").  The 16
// heads share each gathered row, so every selected row is read once per
// query; two independent groups per CTA and two CTAs per SM keep 16 warps of
// per-tile chains in flight on each SM.
#include "common.cuh"
#include "kernels.h"

namespace fbm {
namespace {

constexpr int kDTok = 16;     // tokens per tile
constexpr int kDHeads = 16;   // query heads (the MMA M dimension)
constexpr int kDGroups = 2;   // independent 4-warp groups per CTA
constexpr int kDThreads = 128 * kDGroups;

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
// the 128 threads of one warp group (named barrier 1 + group)
FBM_DEVICE void group_sync(int grp) {
  asm volatile("bar.sync %0, 128;\n" ::"r"(1 + grp) : "memory");
}

template <int D>
FBM_DEVICE uint32_t swz(int r, int ch) {
  return (uint32_t)(r * (D * 2) + ((ch ^ (r & 7)) << 4));
}

// shared memory of one warp group: two KV tiles, the warps' partial scores,
// P and the per-head rescale factors
template <int D>
struct DecGroup {
  static constexpr int kTile = kDTok * D * 2;
  static constexpr int kPLd = kDTok + 8;  // padded P row (elements)
  static constexpr int kPart = 2 * kTile;
  static constexpr int kP = kPart + 4 * kDHeads * kDTok * 4;
  static constexpr int kAlpha = kP + kDHeads * kPLd * 2;
  static constexpr int kBytes = (kAlpha + kDHeads * 4 + 127) / 128 * 128;
};

template <int D>
constexpr size_t dec_fixed_bytes() {
  return (size_t)kDHeads * D * 2 + (size_t)kDGroups * DecGroup<D>::kBytes + 4 * kDHeads * 4;
}

template <class E, int D, int DV>
__global__ void __launch_bounds__(kDThreads, 2) k_sparse_decode(const DecodeLaunch L) {
  static_assert(D % 64 == 0 && DV % 64 == 0 && DV <= D, "shape");
  using G = DecGroup<D>;
  constexpr int KS_PER_WARP = D / 64;  // 16-wide k-steps per warp for S
  static_assert(4 * (DV / 4) * 16 * 4 <= 2 * G::kTile, "group 1's O fits in its KV tiles");
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const int tid = threadIdx.x, grp = tid >> 7, gtid = tid & 127;
  const int warp = gtid >> 5, lane = tid & 31;
  uint8_t *gb = smem + kDHeads * D * 2 + grp * G::kBytes;
  const uint32_t sKV = smem_u32(gb);
  float *s_part = reinterpret_cast<float *>(gb + G::kPart);
  uint16_t *s_p = reinterpret_cast<uint16_t *>(gb + G::kP);
  float *s_alpha = reinterpret_cast<float *>(gb + G::kAlpha);
  float *s_ml = reinterpret_cast<float *>(smem + kDHeads * D * 2 + kDGroups * G::kBytes);
  int32_t *s_rows = reinterpret_cast<int32_t *>(s_ml + 4 * kDHeads);

  const int split = blockIdx.x % L.num_splits;
  const int c = blockIdx.x / L.num_splits;
  const int base = L.topk / L.num_splits, extra = L.topk % L.num_splits;
  const int lo = split * base + min(split, extra);
  const int n = base + (split < extra ? 1 : 0);
  const uint16_t *cache = static_cast<const uint16_t *>(L.cache);
  const int max_pos = L.pages_per_query * L.page;
  // a chained launch: it reads its inputs and writes its partials only once
  // the kernel before it is done (no early trigger: a following decode's CTAs
  // dispatched early would crowd onto the idle SMs and unbalance it)
  pdl_wait();

  // prologue: Q [16][D] first (its copy overlaps the lookups), then the token
  // list -> physical rows (-1 = masked).  A thread issues the index loads of
  // all its tokens before their page-table loads, so the prologue waits for
  // two dependent loads rather than two per token.
  {
    const uint16_t *qg = static_cast<const uint16_t *>(L.q) + (size_t)c * L.hq * D;
    for (int ch = tid; ch < kDHeads * (D / 8); ch += kDThreads) {
      const int r = ch / (D / 8), cc = ch % (D / 8);
      cp_async16(sQ + swz<D>(r, cc), qg + (size_t)r * D + cc * 8, true);
    }
    cp_async_commit();
  }
  constexpr int kLook = 4;  // tokens resolved per thread per round
  for (int t0 = tid; t0 < n; t0 += kDThreads * kLook) {
    int pos[kLook], pg[kLook];
#pragma unroll
    for (int u = 0; u < kLook; ++u) {
      const int t = t0 + u * kDThreads;
      pos[u] = t < n ? __ldg(L.idx + (size_t)c * L.topk + lo + t) : -1;
    }
#pragma unroll
    for (int u = 0; u < kLook; ++u)
      pg[u] = (pos[u] >= 0 && pos[u] < max_pos)
                  ? __ldg(L.page_table + (size_t)c * L.pages_per_query + pos[u] / L.page)
                  : -1;
#pragma unroll
    for (int u = 0; u < kLook; ++u) {
      const int t = t0 + u * kDThreads;
      if (t < n) {
        int row = -1;
        if (pos[u] >= 0) {
          if (pos[u] < max_pos && pg[u] >= 0 && pg[u] < L.n_pages) row = pg[u] * L.page + pos[u] % L.page;
          else set_error(L.err, FBM_DEVERR_LUT_RANGE);
        }
        s_rows[t] = row;
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // this group's tiles: grp, grp + 2, ...  Each thread gathers the 16-byte
  // chunks ld_c, ld_c + 8, ... of row ld_r of a tile: one row lookup, then
  // fixed strides (the swizzle only permutes the low three chunk bits)
  static_assert(128 == kDTok * 8 && (D / 8) % 8 == 0, "8 threads per row");
  const int ld_r = gtid >> 3, ld_c = gtid & 7;
  const uint32_t ld_dst = (uint32_t)(ld_r * (D * 2) + ((ld_c ^ (ld_r & 7)) << 4));
  auto load_tile = [&](int tile, int stage) {
    const int tok = tile * kDTok + ld_r;
    const int row = tok < n ? s_rows[tok] : -1;
    const bool ok = row >= 0;
    const uint16_t *src = cache + (size_t)(ok ? row : 0) * D + ld_c * 8;
    const uint32_t dst = sKV + stage * G::kTile + ld_dst;
#pragma unroll
    for (int k = 0; k < D / 64; ++k) cp_async16(dst + k * 128, src + k * 64, ok);
  };
  const int ntiles = (n + kDTok - 1) / kDTok;
  const int mine = ntiles > grp ? (ntiles - grp + 1) / kDGroups : 0;
  if (mine > 0) load_tile(grp, 0);
  cp_async_commit();

  float o[DV / 4 / 8][4];  // this warp's DV/4 columns: DV/32 n-tiles
#pragma unroll
  for (int a = 0; a < DV / 32; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
  // softmax role: thread -> head gtid/8, tokens (gtid%8)*2 .. +1
  const int sm_head = gtid >> 3, sm_tok = (gtid & 7) * 2;
  float m_run = -INFINITY, l_run = 0.f;
  const float sl2 = L.scale * 1.4426950408889634f;

  for (int j = 0; j < mine; ++j) {
    const int tile = kDGroups * j + grp;
    const int stage = j & 1;
    if (j + 1 < mine) {
      load_tile(tile + kDGroups, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    group_sync(grp);
    const uint32_t kv = sKV + stage * G::kTile;
    // partial S over this warp's slice of the contraction
    float s[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS_PER_WARP; ++ks) {
      uint32_t qf[4];
      const int qch = (warp * KS_PER_WARP + ks) * 2 + (lane >> 4);
      ldsm_x4(sQ + swz<D>(lane & 15, qch), qf[0], qf[1], qf[2], qf[3]);
      const int mi = lane >> 3;
      const int tok = (mi >> 1) * 8 + (lane & 7);
      const int ch = (warp * KS_PER_WARP + ks) * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kv + swz<D>(tok, ch), b0, b1, b2, b3);
      mma16816<E>(s[0], qf, b0, b1);
      mma16816<E>(s[1], qf, b2, b3);
    }
    // the warp's partial scores, two adjacent tokens per 8-byte store (the
    // softmax threads below read them back the same way, without conflicts)
    float *sp = s_part + warp * kDHeads * kDTok;
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int head = (lane >> 2) + 8 * hh;
        const int tok = a * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2 *>(sp + head * kDTok + tok) =
            make_float2(s[a][2 * hh], s[a][2 * hh + 1]);
      }
    group_sync(grp);
    // online softmax for (sm_head, 2 tokens)
    {
      float x[2];
      float mx = -INFINITY;
      {
        const float *pp = s_part + sm_head * kDTok + sm_tok;
        const float2 p0 = *reinterpret_cast<const float2 *>(pp);
        const float2 p1 = *reinterpret_cast<const float2 *>(pp + kDHeads * kDTok);
        const float2 p2 = *reinterpret_cast<const float2 *>(pp + 2 * kDHeads * kDTok);
        const float2 p3 = *reinterpret_cast<const float2 *>(pp + 3 * kDHeads * kDTok);
        x[0] = p0.x + p1.x + p2.x + p3.x;
        x[1] = p0.y + p1.y + p2.y + p3.y;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int gtok = tile * kDTok + sm_tok + u;
        if (gtok >= n || s_rows[gtok] < 0) x[u] = -INFINITY;
        mx = fmaxf(mx, x[u]);
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
      for (int u = 0; u < 2; ++u) {
        x[u] = exp2f(fmaf(x[u], sl2, -b));
        ls += x[u];
      }
      l_run = l_run * alpha + ls;
      *reinterpret_cast<uint32_t *>(s_p + sm_head * G::kPLd + sm_tok) = E::from_f2(x[0], x[1]);
      if ((gtid & 7) == 0) s_alpha[sm_head] = alpha;
    }
    group_sync(grp);
    // O = alpha * O + P V over this warp's DV/4 columns
    {
      const float a0 = s_alpha[lane >> 2], a1 = s_alpha[(lane >> 2) + 8];
      // alpha is exactly 1 for a head whose running max did not move
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int a = 0; a < DV / 32; ++a) {
          o[a][0] *= a0; o[a][1] *= a0; o[a][2] *= a1; o[a][3] *= a1;
        }
      }
      const uint32_t sP = smem_u32(s_p);
      uint32_t pa[4];
      ldsm_x4(sP + (lane & 15) * (G::kPLd * 2) + (lane >> 4) * 16, pa[0], pa[1], pa[2], pa[3]);
#pragma unroll
      for (int dp = 0; dp < DV / 64; ++dp) {
        const int mi = lane >> 3;
        const int tok = (mi & 1) * 8 + (lane & 7);
        const int ch = (warp * (DV / 4) + dp * 16) / 8 + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(kv + swz<D>(tok, ch), b0, b1, b2, b3);
        mma16816<E>(o[2 * dp], pa, b0, b1);
        mma16816<E>(o[2 * dp + 1], pa, b2, b3);
      }
    }
    group_sync(grp);
  }

  // merge the two groups' states (running max m in base 2, sum l, O) per head
  {
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    if ((gtid & 7) == 0) {
      s_ml[(2 * grp) * kDHeads + sm_head] = m_run;
      s_ml[(2 * grp + 1) * kDHeads + sm_head] = l;
    }
  }
  // group 1's O goes to its own (now idle) KV tiles, laid out by thread
  float *s_o1 = reinterpret_cast<float *>(smem + kDHeads * D * 2 + G::kBytes);
  if (grp == 1) {
#pragma unroll
    for (int a = 0; a < DV / 32; ++a)
      *reinterpret_cast<float4 *>(s_o1 + ((size_t)a * 128 + gtid) * 4) =
          make_float4(o[a][0], o[a][1], o[a][2], o[a][3]);
  }
  __syncthreads();
  if (grp != 0) return;
  float w0[2], w1[2], inv[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = (lane >> 2) + 8 * hh;
    const float m0 = s_ml[h], l0 = s_ml[kDHeads + h];
    const float m1 = s_ml[2 * kDHeads + h], l1 = s_ml[3 * kDHeads + h];
    const float m = fmaxf(m0, m1);
    w0[hh] = m == -INFINITY ? 0.f : exp2f(m0 - m);
    w1[hh] = m == -INFINITY ? 0.f : exp2f(m1 - m);
    const float l = w0[hh] * l0 + w1[hh] * l1;
    inv[hh] = l > 0.f ? 1.0f / l : 0.f;
  }
  if ((gtid & 7) == 0) {
    const int h = sm_head;
    const float m0 = s_ml[h], l0 = s_ml[kDHeads + h];
    const float m1 = s_ml[2 * kDHeads + h], l1 = s_ml[3 * kDHeads + h];
    const float m = fmaxf(m0, m1);
    const float l = m == -INFINITY ? 0.f : exp2f(m0 - m) * l0 + exp2f(m1 - m) * l1;
    L.lse_part[((size_t)split * L.n_q + c) * kDHeads + h] =
        l > 0.f ? m * 0.6931471805599453f + logf(l) : -INFINITY;
  }
  float *dst = L.o_part + ((size_t)split * L.n_q + c) * kDHeads * DV;
#pragma unroll
  for (int a = 0; a < DV / 32; ++a) {
    const float4 p1 = *reinterpret_cast<const float4 *>(s_o1 + ((size_t)a * 128 + gtid) * 4);
    const int col = warp * (DV / 4) + a * 8 + (lane & 3) * 2;
    const int h0 = lane >> 2;
    *reinterpret_cast<float2 *>(dst + (size_t)h0 * DV + col) =
        make_float2((w0[0] * o[a][0] + w1[0] * p1.x) * inv[0], (w0[0] * o[a][1] + w1[0] * p1.y) * inv[0]);
    *reinterpret_cast<float2 *>(dst + (size_t)(h0 + 8) * DV + col) =
        make_float2((w0[1] * o[a][2] + w1[1] * p1.z) * inv[1], (w0[1] * o[a][3] + w1[1] * p1.w) * inv[1]);
  }
}

template <class E, int D, int DV>
size_t decode_smem(int chunk) {
  return dec_fixed_bytes<D>() + (size_t)chunk * 4;
}

template <class E>
cudaError_t launch_e(const DecodeLaunch &L, cudaStream_t st) {
  const int chunk = (L.topk + L.num_splits - 1) / L.num_splits;
  const size_t smem = decode_smem<E, 576, 512>(chunk);
  cudaError_t e = cudaFuncSetAttribute(k_sparse_decode<E, 576, 512>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_sparse_decode<E, 576, 512>, dim3(L.n_q * L.num_splits), dim3(kDThreads), smem,
                    st, L);
}

}  // namespace

size_t decode_smem_bytes(int topk, int num_splits) {
  return decode_smem<BF16, 576, 512>((topk + num_splits - 1) / num_splits);
}

cudaError_t launch_decode(const DecodeLaunch &L, cudaStream_t st) {
  return L.bf16 ? launch_e<BF16>(L, st) : launch_e<F16>(L, st);
}

}  // namespace fbm
