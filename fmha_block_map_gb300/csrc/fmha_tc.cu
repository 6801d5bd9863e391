// Sparse FMHA forward for sm_103a on 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA loads), d = 128.
//
// The per-q-block work of the sparse FMHA stage (the "Sparge Attention
// (Composable Kernel)" README) visits only the kv blocks of the q block's LUT
// row.  A q block holds 64 query rows, less than the 128-row tile of a full-rate
// tcgen05.mma, and neighbouring q blocks select different kv blocks, so the
// kernel computes the transposed problem: two LUT-selected kv blocks (128 keys)
// form the M dimension and the 64 queries the N dimension.
//
//   S^T [128 keys x 64 q]  = K_pair [128 x d] . Q^T          (A, B K-major)
//   O^T [d x 64 q]        += V_pair^T [d x 128] . P^T [128 x 64] (A, B MN-major)
//
// No MMA row is spent on a kv block the q block did not select (an odd count
// leaves one half-empty pair per row).  The softmax runs along TMEM lanes
// (keys): each of the 128 softmax threads owns one key and holds that key's 64
// scores; the running max per query is kept lazily (rescale only when a score
// exceeds it by more than 2^8), so the cross-lane column maximum is needed only
// on those rare pairs.
//
// Roles (one persistent CTA per SM, 20 warps):
//   warp 0    TMA producer of Q (double buffer) and K pairs (2-slot ring)
//   warp 19   TMA producer of V pairs (2-slot ring)
//   warp 1    TMEM owner and single-thread S^T issuer
//   warp 18   single-thread PV issuer (so S^T never queues behind a PV that
//             waits for the softmax)
//   warps 2-17 four softmax + epilogue warpgroups, each owning 16 of the 64
//             query columns (each group covers TMEM lane quadrants 2, 3, 0, 1:
//             all 128 keys)
// Pipeline: S^T(p) is issued once K(p) has landed and its TMEM slot (two
// slots) is free; PV(p) once P(p) is written.  The softmax of pair p+1
// overlaps the PV MMA of pair p.  Every wait is bounded:
// on expiry the kernel raises FBM_DEVERR_TIMEOUT, every role leaves its loop,
// in-flight copies and MMAs are drained with bounded waits and TMEM is freed.
//
// Loop shape: the Incremental_FlashAttention updating_log's Stage 3/4 sparse
// mainloop (listed blocks only, next K prefetched while the current tile is
// consumed, an empty list writes O = 0 and LSE = -inf).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kQBytes = 64 * kD * 2;      // 16 KB: a 64-row Q tile
constexpr int kPairBytes = 128 * kD * 2;  // 32 KB: two 64-row kv blocks
constexpr int kQChunk = 64 * 128;         // 8 KB: one 64-wide d chunk of a 64-row tile
constexpr int kPairChunk = 128 * 128;     // 16 KB: one 64-wide d chunk of a 128-row pair
constexpr int kPBytes = 128 * 128;        // 16 KB: P^T, 128 keys x 64 queries (MN-major)

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 2 * kQBytes;
constexpr int OFF_V = OFF_K + 2 * kPairBytes;
constexpr int OFF_P = OFF_V + 2 * kPairBytes;
constexpr int OFF_STAGE = OFF_P + 2 * kPBytes;   // 16 KB: output staging [64 q][128 d]
constexpr int kGroups = 4;                         // softmax warpgroups per CTA
constexpr int kCW = 64 / kGroups;                  // query columns per group
constexpr int OFF_RED = OFF_STAGE + kQBytes;       // float [groups][4 quadrants][kCW]
constexpr int OFF_ALPHA = OFF_RED + kGroups * 4 * kCW * 4;  // float [groups][kCW]
constexpr int OFF_INVL = OFF_ALPHA + kGroups * kCW * 4;     // float [groups][kCW]
constexpr int OFF_M = OFF_INVL + kGroups * kCW * 4;         // float [groups][kCW]
constexpr int OFF_BAR = OFF_M + kGroups * kCW * 4;
enum {
  B_QF = 0, B_QE = 2, B_KF = 4, B_KE = 6, B_VF = 8, B_VE = 10, B_SF = 12, B_SE = 14,
  B_PF = 16, B_PV = 18, B_OF = 20, B_DRAIN = 21, B_DRAIN2 = 22, NBAR = 23
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;      // [0] tmem base, [1] abort flag
constexpr int SMEM_BYTES = OFF_MISC + 16;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
constexpr uint32_t kTmemCols = 256;                // S0 @0, S1 @64, O @128
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s per wait
constexpr int kGroupThreads = 128;                 // one softmax warpgroup
constexpr int kSoftmaxThreads = kGroups * kGroupThreads;
constexpr int kPvWarp = 2 + kSoftmaxThreads / 32;  // the PV issuer follows the softmax warps
constexpr int kVWarp = kPvWarp + 1;                 // then the V producer
constexpr int kThreads = 64 + kSoftmaxThreads + 64; // + Q/K producer, S^T issuer, PV issuer, V producer

// N consecutive TMEM columns of 32 lanes (a query group's columns)
template <int N>
FBM_DEVICE void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 16) tmem_ld16(taddr, r);
  else tmem_ld32(taddr, r);
}
template <int N>
FBM_DEVICE void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 16) tmem_st16(taddr, r);
  else tmem_st32(taddr, r);
}

struct TcParams {
  CUtensorMap tq, tk, tv;
  const int32_t *lut, *cnt;
  void *out;
  float *lse;
  uint32_t *err;
  int b, hq, hk, s_q, s_k, nq, nk, lut_stride, causal, units;
  float sl2;  // scale * log2(e)
};

struct Unit {
  int bh_q, bh_k, i, n;
  const int32_t *row;
};

FBM_DEVICE Unit unit_of(const TcParams &P, int u) {
  Unit U;
  U.bh_q = u / P.nq;
  U.i = u - U.bh_q * P.nq;
  const int b = U.bh_q / P.hq, h = U.bh_q - b * P.hq;
  U.bh_k = b * P.hk + h / (P.hq / P.hk);
  if (P.lut) {
    U.row = P.lut + (size_t)u * P.lut_stride;
    int n = __ldg(P.cnt + u);
    U.n = max(0, min(n, min(P.nk, P.lut_stride)));
  } else {
    U.row = nullptr;
    U.n = P.causal ? min(P.nk, U.i + 1) : P.nk;
  }
  return U;
}

FBM_DEVICE int entry_of(const Unit &U, int t) { return U.row ? __ldg(U.row + t) : t; }

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1) k_fmha_tc(const __grid_constant__ TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *misc = reinterpret_cast<volatile int *>(smem + OFF_MISC);
  volatile int *abort_flag = misc + 1;
  auto bar = [&](int k) -> uint32_t { return sbase + OFF_BAR + 8 * k; };

  if (threadIdx.x == 0) {
    for (int k = 0; k < NBAR; ++k) {
      uint32_t cnt = 1;
      if (k == B_SE || k == B_SE + 1 || k == B_PF || k == B_PF + 1 || k == B_OF)
        cnt = kSoftmaxThreads;  // every query group arrives
      mbar_init(bar(k), cnt);
    }
    misc[1] = 0;
    fence_mbar_init();
    prefetch_map(&P.tq);
    prefetch_map(&P.tk);
    prefetch_map(&P.tv);
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = (uint32_t)misc[0];

  auto fail = [&](uint32_t bits) {
    set_error(P.err, bits);
    *abort_flag = 1;
  };

  // K or V pair g (= pc + p) of a q block into its ring slot, once the MMA that
  // last read the slot has completed
  auto load_pair = [&](const Unit &U, int pc, int p, bool is_v) -> bool {
    const int g = pc + p, slot = g & 1;
    const int fb = (is_v ? B_VF : B_KF) + slot, eb = (is_v ? B_VE : B_KE) + slot;
    if (!mbar_wait(bar(eb), ((g >> 1) & 1) ^ 1, abort_flag, kWaitNs)) return false;
    int js[2] = {-1, -1};
    uint32_t bytes = 0;
    for (int hf = 0; hf < 2; ++hf) {
      const int t = 2 * p + hf;
      if (t >= U.n) break;
      int j = entry_of(U, t);
      if (j < 0 || j >= P.nk) {
        // out of range: flagged; block 0 is fetched in its place so that the
        // masked keys (P = 0) meet finite V rows
        set_error(P.err, FBM_DEVERR_LUT_RANGE);
        j = 0;
      }
      js[hf] = j;
      bytes += 2 * kQChunk;
    }
    mbar_arrive_tx(bar(fb), bytes);
    const uint32_t dst0 = sbase + (is_v ? OFF_V : OFF_K) + slot * kPairBytes;
    for (int hf = 0; hf < 2; ++hf) {
      if (js[hf] < 0) continue;
      for (int c = 0; c < 2; ++c)
        tma_load_3d(dst0 + c * kPairChunk + hf * kQChunk, is_v ? &P.tv : &P.tk, c * 64,
                    js[hf] * 64, U.bh_k, bar(fb));
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    if (lane == 0) {
      int pc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of(P, u);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        const int qb = uc & 1;
        if (!(ok = mbar_wait(bar(B_QE + qb), ((uc >> 1) & 1) ^ 1, abort_flag, kWaitNs))) break;
        mbar_arrive_tx(bar(B_QF + qb), kQBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sbase + OFF_Q + qb * kQBytes + c * kQChunk, &P.tq, c * 64, U.i * 64,
                      U.bh_q, bar(B_QF + qb));
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc, p, false);
        pc += npairs;
        uc += 1;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ V producer
    // (its own thread, so a K load never waits behind a V slot that a late PV
    // still holds)
    if (lane == 0) {
      int pc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of(P, u);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc, p, true);
        pc += npairs;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S^T issuer
    // S^T(g) runs as soon as its K pair is loaded and its TMEM slot is free;
    // it never waits for P, so it stays ahead of the softmax.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(kBf16, false, false, 128, 64);
      int pc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of(P, u);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        const int qb = uc & 1;
        if (!(ok = mbar_wait(bar(B_QF + qb), (uc >> 1) & 1, abort_flag, kWaitNs))) break;
        tc_fence_after();
        const uint32_t qaddr = sbase + OFF_Q + qb * kQBytes;
        for (int p = 0; p < npairs; ++p) {
          const int g = pc + p, slot = g & 1;
          if (!(ok = mbar_wait(bar(B_KF + slot), (g >> 1) & 1, abort_flag, kWaitNs))) break;
          if (!(ok = mbar_wait(bar(B_SE + slot), ((g >> 1) & 1) ^ 1, abort_flag, kWaitNs))) break;
          tc_fence_after();
          const uint32_t kaddr = sbase + OFF_K + slot * kPairBytes;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(kaddr + (kk >> 2) * kPairChunk + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(qaddr + (kk >> 2) * kQChunk + (kk & 3) * 32, 16, 1024);
            mma_f16(tbase + slot * 64, ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SF + slot));
          mma_commit(bar(B_KE + slot));
        }
        if (ok) mma_commit(bar(B_QE + qb));  // Q free once every S^T of the row is done
        pc += npairs;
        uc += 1;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
      // drain: every MMA this thread issued has completed before TMEM is freed
      mma_commit(bar(B_DRAIN));
      if (!mbar_wait_for(bar(B_DRAIN), 0, kWaitNs)) set_error(P.err, FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t idO = idesc_f16(kBf16, true, true, 128, 64);
      const uint32_t tO = tbase + 128;
      int pc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of(P, u);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        for (int p = 0; p < npairs; ++p) {
          const int g = pc + p, slot = g & 1;
          if (!(ok = mbar_wait(bar(B_PF + slot), (g >> 1) & 1, abort_flag, kWaitNs))) break;
          if (!(ok = mbar_wait(bar(B_VF + slot), (g >> 1) & 1, abort_flag, kWaitNs))) break;
          if (p == 0 && !(ok = mbar_wait(bar(B_OF), (uc & 1) ^ 1, abort_flag, kWaitNs))) break;
          tc_fence_after();
          const uint32_t vaddr = sbase + OFF_V + slot * kPairBytes;
          const uint32_t paddr = sbase + OFF_P + slot * kPBytes;
          const int ksteps = (2 * p + 1 < U.n) ? 8 : 4;  // a half pair has 64 keys
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t ad = sdesc_sw128(vaddr + kk * 2048, kPairChunk, 1024);
            const uint64_t bd = sdesc_sw128(paddr + kk * 2048, kPairChunk, 1024);
            mma_f16(tO, ad, bd, idO, (p > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_PV + slot));
          mma_commit(bar(B_VE + slot));
        }
        pc += npairs;
        uc += 1;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
      mma_commit(bar(B_DRAIN2));
      if (!mbar_wait_for(bar(B_DRAIN2), 0, kWaitNs)) set_error(P.err, FBM_DEVERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wg = (warp - 2) >> 2;          // query group: columns kCW*wg .. kCW*wg+kCW-1
    const int cb = wg * kCW;
    const int qd = warp & 3;
    const int key = qd * 32 + lane;          // TMEM lane: key of the pair (S^T) / d (O^T)
    const int tg = (threadIdx.x - 64) & 127; // 0..127 within the group
    const int barid = 1 + wg;                // named barrier of this group
    const uint32_t tl = tbase + ((uint32_t)(qd * 32) << 16);
    float *red = reinterpret_cast<float *>(smem + OFF_RED) + wg * 4 * kCW;   // [4][kCW]
    float *alpha_s = reinterpret_cast<float *>(smem + OFF_ALPHA) + wg * kCW;
    float *invl_s = reinterpret_cast<float *>(smem + OFF_INVL) + wg * kCW;
    float *m_s = reinterpret_cast<float *>(smem + OFF_M) + wg * kCW;
    using E = typename std::conditional<kBf16, BF16, F16>::type;
    // Every softmax thread of a group runs the same loop trip counts and named
    // barriers whatever happens: a failed (timed-out) wait only clears `ok`,
    // and later waits return at once, so no thread is left behind at a barrier.
    int pc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units; u += gridDim.x) {
      const Unit U = unit_of(P, u);
      const int q0 = U.i * 64;
      const int rows = min(64, P.s_q - q0);
      const int my_rows = max(0, min(kCW, rows - cb));  // this group's valid query rows
      uint16_t *orow = static_cast<uint16_t *>(P.out) + ((size_t)U.bh_q * P.s_q + q0 + cb) * kD;
      float *lrow = P.lse ? P.lse + (size_t)U.bh_q * P.s_q + q0 + cb : nullptr;
      if (U.n == 0) {
        for (int e = tg * 8; e < my_rows * kD; e += kGroupThreads * 8)
          *reinterpret_cast<uint4 *>(orow + e) = make_uint4(0, 0, 0, 0);
        if (lrow && tg < my_rows) lrow[tg] = -INFINITY;
        continue;
      }
      const int npairs = (U.n + 1) >> 1;
      // running max per query (log2 domain) lives in m_s; l holds this key's
      // share of the row sums, as packed fp32 pairs (queries 2i, 2i+1)
      uint64_t l2[kCW / 2];
#pragma unroll
      for (int i = 0; i < kCW / 2; ++i) l2[i] = 0ull;
      if (tg < kCW) m_s[tg] = -INFINITY;
      named_sync(barid, kGroupThreads);
      const uint64_t sl2x2 = f2_pack(P.sl2, P.sl2);
      int j_next = (key >> 6) < U.n ? entry_of(U, key >> 6) : -1;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, slot = g & 1;
        // this thread's key: block t of the row, offset key & 63
        const int j = j_next;
        {
          const int tn = 2 * (p + 1) + (key >> 6);
          j_next = (p + 1 < npairs && tn < U.n) ? entry_of(U, tn) : -1;
        }
        const bool jvalid = j >= 0 && j < P.nk;
        const int kpos = (jvalid ? j : 0) * 64 + (key & 63);
        const bool kvalid = jvalid && kpos < P.s_k;
        // queries cb + q with q < qmin cannot see this key (causal)
        const int qmin = P.causal ? kpos - q0 - cb : -1;
        const bool plain = kvalid && qmin <= 0;  // the whole column range is visible
        ok = ok && mbar_wait(bar(B_SF + slot), (g >> 1) & 1, abort_flag, kWaitNs);
        tc_fence_after();
        uint32_t r[kCW];
        tmem_ld_cols(tl + slot * 64 + cb, r);
        tmem_wait_ld();
        uint64_t x2[kCW / 2];
        float mx;
        if (plain) {
#pragma unroll
          for (int i4 = 0; i4 < kCW / 4; ++i4) {
            const float4 mv = reinterpret_cast<const float4 *>(m_s)[i4];
            x2[2 * i4] = f2_fma(f2_pack(__uint_as_float(r[4 * i4]), __uint_as_float(r[4 * i4 + 1])),
                                sl2x2, f2_pack(-mv.x, -mv.y));
            x2[2 * i4 + 1] = f2_fma(f2_pack(__uint_as_float(r[4 * i4 + 2]), __uint_as_float(r[4 * i4 + 3])),
                                    sl2x2, f2_pack(-mv.z, -mv.w));
          }
        } else {
#pragma unroll
          for (int i = 0; i < kCW / 2; ++i) {
            const int q = 2 * i;
            const float a = (kvalid && q >= qmin) ? fmaf(__uint_as_float(r[q]), P.sl2, -m_s[q]) : -INFINITY;
            const float b = (kvalid && q + 1 >= qmin) ? fmaf(__uint_as_float(r[q + 1]), P.sl2, -m_s[q + 1]) : -INFINITY;
            x2[i] = f2_pack(a, b);
          }
        }
        {
          float t[kCW / 4];
#pragma unroll
          for (int i = 0; i < kCW / 4; ++i) {
            const float2 a = f2_unpack(x2[2 * i]), b = f2_unpack(x2[2 * i + 1]);
            t[i] = fmax3(a.x, a.y, fmaxf(b.x, b.y));
          }
          mx = t[0];
#pragma unroll
          for (int i = 1; i < kCW / 4; i += 2)
            mx = (i + 1 < kCW / 4) ? fmax3(mx, t[i], t[i + 1]) : fmaxf(mx, t[i]);
        }
        if (named_or(barid, kGroupThreads, mx > 8.0f)) {
          // rare: some score exceeds the running max by > 2^8 (always on the
          // first pair): exact column max over the 128 keys, then rescale
          float v[kCW];
#pragma unroll
          for (int q = 0; q < kCW; ++q)
            v[q] = (kvalid && q >= qmin) ? __uint_as_float(r[q]) * P.sl2 : -INFINITY;
          // transpose-reduce within the warp: lanes l and l + 16 end with column l & 15
#pragma unroll
          for (int o = kCW / 2; o >= 1; o >>= 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int x = 0; x < o; ++x) {
              const float send = hi ? v[x] : v[x + o];
              const float keep = hi ? v[x + o] : v[x];
              v[x] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
            }
          }
          if constexpr (kCW == 16) v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 16));
          if (lane < kCW) red[qd * kCW + lane] = v[0];
          named_sync(barid, kGroupThreads);
          if (tg < kCW) {
            const int q = tg;
            const float cm = fmaxf(fmaxf(red[q], red[kCW + q]), fmaxf(red[2 * kCW + q], red[3 * kCW + q]));
            const float mo = m_s[q];
            const float mn = fmaxf(mo, cm);
            alpha_s[q] = (mn == -INFINITY) ? 1.f : fast_exp2(mo - mn);
            m_s[q] = mn;
          }
          named_sync(barid, kGroupThreads);
#pragma unroll
          for (int i = 0; i < kCW / 2; ++i)
            l2[i] = f2_mul(l2[i], f2_pack(alpha_s[2 * i], alpha_s[2 * i + 1]));
          if (p > 0) {
            // O^T holds PV(0 .. p-1): wait for the last of them, then scale
            const int gp = g - 1;
            ok = ok && mbar_wait(bar(B_PV + (gp & 1)), (gp >> 1) & 1, abort_flag, kWaitNs);
            tc_fence_after();
            uint32_t o[kCW];
            tmem_ld_cols(tl + 128 + cb, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < kCW; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha_s[q]);
            tmem_st_cols(tl + 128 + cb, o);
            tmem_wait_st();
            tc_fence_before();
          }
#pragma unroll
          for (int i = 0; i < kCW / 2; ++i) {
            const int q = 2 * i;
            const float a = (kvalid && q >= qmin) ? fmaf(__uint_as_float(r[q]), P.sl2, -m_s[q]) : -INFINITY;
            const float b = (kvalid && q + 1 >= qmin) ? fmaf(__uint_as_float(r[q + 1]), P.sl2, -m_s[q + 1]) : -INFINITY;
            x2[i] = f2_pack(a, b);
          }
        }
        // P(p) goes to buffer `slot`, last read by PV(g - 2)
        if (p >= 2) {
          const int gp = g - 2;
          ok = ok && mbar_wait(bar(B_PV + slot), (gp >> 1) & 1, abort_flag, kWaitNs);
        }
        uint8_t *prow = smem + OFF_P + slot * kPBytes + key * 128;
#pragma unroll
        for (int c = 0; c < kCW / 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const float2 xv = f2_unpack(x2[4 * c + z]);
            const float e0 = fast_exp2(xv.x), e1 = fast_exp2(xv.y);
            l2[4 * c + z] = f2_add(l2[4 * c + z], f2_pack(e0, e1));
            pk[z] = E::from_f2(e0, e1);
          }
          const int chunk = wg * (kCW / 8) + c;
          *reinterpret_cast<uint4 *>(prow + ((chunk ^ (key & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(bar(B_PF + slot));
        mbar_arrive(bar(B_SE + slot));
      }
      // ---- epilogue: O = O^T / l, LSE = m ln2 + ln l (this group's kCW queries)
      {
        const int gl = pc + npairs - 1;
        ok = ok && mbar_wait(bar(B_PV + (gl & 1)), (gl >> 1) & 1, abort_flag, kWaitNs);
        tc_fence_after();
        // sum l over the 128 keys
        float l[kCW];
#pragma unroll
        for (int i = 0; i < kCW / 2; ++i) {
          const float2 v = f2_unpack(l2[i]);
          l[2 * i] = v.x;
          l[2 * i + 1] = v.y;
        }
#pragma unroll
        for (int o = kCW / 2; o >= 1; o >>= 1) {
          const bool hi = (lane & o) != 0;
#pragma unroll
          for (int x = 0; x < o; ++x) {
            const float send = hi ? l[x] : l[x + o];
            const float keep = hi ? l[x + o] : l[x];
            l[x] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        if constexpr (kCW == 16) l[0] += __shfl_xor_sync(0xffffffffu, l[0], 16);
        if (lane < kCW) red[qd * kCW + lane] = l[0];
        named_sync(barid, kGroupThreads);
        if (tg < kCW) {
          const int q = tg;
          const float lt = (red[q] + red[kCW + q]) + (red[2 * kCW + q] + red[3 * kCW + q]);
          invl_s[q] = lt > 0.f ? 1.0f / lt : 0.f;
          if (lrow && q < my_rows)
            lrow[q] = lt > 0.f ? m_s[q] * 0.6931471805599453f + logf(lt) : -INFINITY;
        }
        named_sync(barid, kGroupThreads);
        // O^T row `key` (= d), columns cb.. -> staging rows cb.. of [64 q][128 d]
        uint16_t *stage = reinterpret_cast<uint16_t *>(smem + OFF_STAGE);
        {
          uint32_t r[kCW];
          tmem_ld_cols(tl + 128 + cb, r);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < kCW; ++q)
            stage[(cb + q) * kD + key] = E::bits(__uint_as_float(r[q]) * invl_s[q]);
        }
        tc_fence_before();
        mbar_arrive(bar(B_OF));
        fence_proxy_async();
        named_sync(barid, kGroupThreads);
        if (tg == 0 && my_rows > 0) {
          bulk_store(orow, sbase + OFF_STAGE + cb * kD * 2, (uint32_t)(my_rows * kD * 2));
          bulk_commit();
          bulk_wait_read0();
        }
        named_sync(barid, kGroupThreads);
      }
      pc += npairs;
    }
    if (!ok) fail(FBM_DEVERR_TIMEOUT);
    if (tg == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [bh, s, d=128] 16-bit tensor, box = 64 d x 64 rows x 1 head, 128B swizzle
bool make_map(CUtensorMap *m, const void *base, int bh, int s, bool bf16) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)s, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)s * kD * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

template <bool BF16>
cudaError_t launch_t(const FmhaLaunch &L, cudaStream_t st) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k_fmha_tc<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  TcParams P;
  memset(&P, 0, sizeof(P));
  if (!make_map(&P.tq, L.q, L.b * L.hq, L.s_q, BF16) || !make_map(&P.tk, L.k, L.b * L.hk, L.s_k, BF16) ||
      !make_map(&P.tv, L.v, L.b * L.hk, L.s_k, BF16))
    return cudaErrorInvalidValue;
  P.lut = L.lut;
  P.cnt = L.cnt;
  P.out = L.out;
  P.lse = L.lse;
  P.err = L.err;
  P.b = L.b; P.hq = L.hq; P.hk = L.hk; P.s_q = L.s_q; P.s_k = L.s_k; P.nq = L.nq; P.nk = L.nk;
  P.lut_stride = L.lut_stride;
  P.causal = L.causal;
  P.units = L.b * L.hq * L.nq;
  P.sl2 = L.scale * 1.4426950408889634f;
  const int grid = std::min(P.units, sm_count());
  k_fmha_tc<BF16><<<grid, kThreads, SMEM_ALLOC, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

bool fmha_tc_supported(int d, int dv, int num_splits, int s_q, int s_k) {
  return d == kD && dv == kD && num_splits == 1 && s_q > 0 && s_k > 0;
}

cudaError_t launch_fmha_tc(const FmhaLaunch &L, cudaStream_t st) {
  return L.bf16 ? launch_t<true>(L, st) : launch_t<false>(L, st);
}

}  // namespace fbm
