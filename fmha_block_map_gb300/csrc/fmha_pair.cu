// Sparse FMHA forward on 128-row tiles: two adjacent q blocks of a (batch,
// head) attend together.
//
// A 64-row q block can only feed M = 64 tensor-core MMAs, which run at half
// the M = 128 rate and read every K / V byte from shared memory once per 64
// query rows.  Here q blocks 2p and 2p + 1 form one 128-row tile that walks
// the union of their LUT rows (lut_pair_union: ascending, each entry flagged
// with the rows it belongs to); a row masks (-inf) every kv block outside its
// own LUT row, so the result is exactly that of the two q blocks attending
// alone, while each MMA now covers 128 query rows.  With LUT rows A and B the
// tensor work is |A u B| 128-row tiles instead of |A| + |B| 64-row ones, and
// in dense mode (every kv block) the union is the row itself.
//
// Per union pair g (two kv blocks, 128 keys):
//   S [128 q x 128 keys]  = Q . K_pair^T      M = 128, N = 128 (A, B in smem)
//   P = exp2(S * scale * log2 e - m)           16-bit, into TMEM (A operand layout)
//   O [128 q x D]        += P . V_pair         M = 128, N = D (A = P in TMEM, B = V)
//
// TMEM (512 columns, lane = query row): S slots at 0 and 128, P buffers at 256
// and 320 (two 16-bit values per column), O at 384.
// Roles (one persistent CTA per SM, 12 warps):
//   warp 0     TMA producer of Q (128-row tile, double buffer) and K pairs
//   warp 1     TMA producer of V pairs
//   warp 2     TMEM owner and S issuer
//   warp 3     PV issuer
//   warps 4-11 softmax and epilogue: warp w reads TMEM lanes 32 (w mod 4) ..
//              (rows; q block 2p for subpartitions 0-1, 2p + 1 for 2-3) and
//              handles kv block (w - 4) / 4 of each pair, one row per thread;
//              the two warps of a subpartition agree on the row max through
//              one OR-barrier per pair, exchanging their block maxima in
//              shared memory only when either must move it.
// The output tile is staged in the (dead) Q slot of its unit: that slot's
// release needs the last S MMA's commit and the epilogue's arrival.  Every
// wait is bounded; on expiry the kernel raises FBM_DEVERR_TIMEOUT, every role
// leaves its loop, in-flight MMAs are drained and TMEM is freed.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <type_traits>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {

// shared with fmha_tc.cu (host helpers)
PFN_cuTensorMapEncodeTiled_v12000 tma_encoder();
int device_sm_count();

namespace {

using namespace tc;

constexpr int kChunk = 128 * 128;   // 16 KB: a 64-wide d chunk of 128 rows
constexpr int kBlkRows = 64 * 128;  // 8 KB: the 64 rows of one kv block within a chunk
constexpr int kKSlots = 2, kVSlots = 2, kSSlots = 2, kPBufs = 2;
enum {
  B_QF = 0, B_QE = 2, B_KF = 4, B_KE = B_KF + kKSlots, B_VF = B_KE + kKSlots,
  B_VE = B_VF + kVSlots, B_SF = B_VE + kVSlots, B_SE = B_SF + kSSlots, B_PF = B_SE + kSSlots,
  B_PV = B_PF + kPBufs, B_OF = B_PV + kPBufs, B_DRAIN = B_OF + 1, B_DRAIN2 = B_DRAIN + 1,
  NBAR = B_DRAIN2 + 1
};

template <int D>
struct PLay {
  static constexpr int NCH = D / 64;
  static constexpr int TileBytes = 128 * D * 2;  // a 128-row Q / output tile, or a K / V pair
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * TileBytes;
  static constexpr int OFF_V = OFF_K + kKSlots * TileBytes;
  static constexpr int OFF_BAR = OFF_V + kVSlots * TileBytes;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] tmem base, [1] abort flag
  // block maxima [pair parity][kv block][128 rows], then row sums [kv block][128 rows]
  static constexpr int OFF_XCH = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = OFF_XCH + (2 * 2 * 128 + 2 * 128) * 4 + 1024;
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTS = 0, kTP = 256, kTO = 384;
constexpr uint32_t kDescHi = sdesc_hi_sw128(1024);
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kWarpQK = 0, kWarpV = 1, kWarpS = 2, kWarpPV = 3, kWarpSm = 4;
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 32 * (kWarpSm + kSoftmaxWarps);
constexpr int kSoftmaxBar = 1, kPairBar0 = 2;
constexpr int kEntryMask = (1 << 29) - 1;  // union entry: block | in-row-A << 29 | in-row-B << 30

struct PairParams {
  CUtensorMap tq, tk, tv, to;
  const int32_t *lut, *cnt;  // pair-union LUT [b * hq * npq, stride] or nullptr (dense)
  void *out;
  float *lse;
  uint32_t *err;
  int b, hq, hk, s_q, s_k, nq, nk, npq, lut_stride, causal, koff, units;
  float sl2;
};

struct PUnit {
  int bh_q, bh_k, p, n;
  const int32_t *row;
};

FBM_DEVICE PUnit punit_of(const PairParams &P, int u, bool *bad) {
  PUnit U;
  U.bh_q = u / P.npq;
  U.p = u - U.bh_q * P.npq;
  const int b = U.bh_q / P.hq, h = U.bh_q - b * P.hq;
  U.bh_k = b * P.hk + h / (P.hq / P.hk);
  *bad = false;
  if (P.lut) {
    U.row = P.lut + (size_t)u * P.lut_stride;
    const int raw = __ldg(P.cnt + u), lim = min(P.nk, P.lut_stride);
    *bad = raw < 0 || raw > lim;
    U.n = max(0, min(raw, lim));
  } else {
    U.row = nullptr;
    const int lastk = U.p * 128 + 127 + P.koff;
    U.n = !P.causal ? P.nk : (lastk < 0 ? 0 : min(P.nk, lastk / 64 + 1));
  }
  return U;
}

// union entry t (block | membership bits); dense rows belong to both q blocks
FBM_DEVICE int pentry(const PUnit &U, int t) {
  return U.row ? __ldg(U.row + t) : (t | (3 << 29));
}

template <int D, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1) k_fmha_pair(const __grid_constant__ PairParams P) {
  using Ly = PLay<D>;
  constexpr int kNch = Ly::NCH, kTile = Ly::TileBytes;
  constexpr int OFF_Q = Ly::OFF_Q, OFF_K = Ly::OFF_K, OFF_V = Ly::OFF_V, OFF_BAR = Ly::OFF_BAR,
                OFF_MISC = Ly::OFF_MISC, OFF_XCH = Ly::OFF_XCH;
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
      if ((k >= B_SE && k < B_SE + kSSlots) || (k >= B_PF && k < B_PF + kPBufs) || k == B_OF)
        cnt = kSoftmaxWarps;  // one elected arrive per softmax warp
      if (k >= B_QE && k < B_QE + 2) cnt = 2;  // the last S commit + the epilogue
      mbar_init(bar(k), cnt);
    }
    misc[1] = 0;
    fence_mbar_init();
    prefetch_map(&P.tq);
    prefetch_map(&P.tk);
    prefetch_map(&P.tv);
    prefetch_map(&P.to);
  }
  if (warp == kWarpS) {
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

  // K or V pair g of a unit into its ring slot, once the MMA that last read
  // the slot has completed
  auto load_pair = [&](const PUnit &U, int g, int p, bool is_v) -> bool {
    const int ns = is_v ? kVSlots : kKSlots;
    const int slot = g % ns;
    const int fb = (is_v ? B_VF : B_KF) + slot, eb = (is_v ? B_VE : B_KE) + slot;
    if (!mbar_wait(bar(eb), ((g / ns) & 1) ^ 1, abort_flag, kWaitNs)) return false;
    int js[2] = {-1, -1};
    uint32_t bytes = 0;
    for (int hf = 0; hf < 2; ++hf) {
      const int t = 2 * p + hf;
      if (t >= U.n) break;
      const int e = pentry(U, t);
      int j = e & kEntryMask;
      if (e < 0 || j >= P.nk) {
        // out of range: flagged (by the K producer); block 0 is fetched in
        // its place so that the masked keys (P = 0) meet finite V rows
        if (!is_v) set_error(P.err, FBM_DEVERR_LUT_RANGE);
        j = 0;
      }
      js[hf] = j;
      bytes += kNch * kBlkRows;
    }
    mbar_arrive_tx(bar(fb), bytes);
    const uint32_t dst0 = sbase + (is_v ? OFF_V : OFF_K) + slot * kTile;
    for (int hf = 0; hf < 2; ++hf) {
      if (js[hf] < 0) continue;
      for (int c = 0; c < kNch; ++c)
        tma_load_3d(dst0 + c * kChunk + hf * kBlkRows, is_v ? &P.tv : &P.tk, c * 64, js[hf] * 64,
                    U.bh_k, bar(fb));
    }
    return true;
  };

  if (warp == kWarpQK) {
    // ------------------------------------------------------------ Q and K producer
    if (lane == 0) {
      int pc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        bool bad;
        const PUnit U = punit_of(P, u, &bad);
        if (bad) set_error(P.err, FBM_DEVERR_LUT_RANGE);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        const int qb = uc & 1;
        if (!(ok = mbar_wait(bar(B_QE + qb), ((uc >> 1) & 1) ^ 1, abort_flag, kWaitNs))) break;
        mbar_arrive_tx(bar(B_QF + qb), kNch * kChunk);
        for (int c = 0; c < kNch; ++c)
          tma_load_3d(sbase + OFF_Q + qb * kTile + c * kChunk, &P.tq, c * 64, U.p * 128, U.bh_q,
                      bar(B_QF + qb));
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc + p, p, false);
        pc += npairs;
        uc += 1;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kWarpV) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      int pc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        bool bad;
        const PUnit U = punit_of(P, u, &bad);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc + p, p, true);
        pc += npairs;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kWarpS) {
    // ------------------------------------------------------------ S issuer
    // (the whole warp runs the loop; one elected lane issues each MMA)
    constexpr uint32_t idS = idesc_f16(kBf16, false, false, 128, 128);
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
      bool bad;
      const PUnit U = punit_of(P, u, &bad);
      if (U.n == 0) continue;
      const int npairs = (U.n + 1) >> 1;
      const int qb = uc & 1;
      if (!(ok = mbar_wait_w(bar(B_QF + qb), (uc >> 1) & 1, abort_flag, kWaitNs))) break;
      tc_fence_after();
      const uint32_t q_lo = sdesc_lo(sbase + OFF_Q + qb * kTile, 16);
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, slot = g % kKSlots, ss = g % kSSlots;
        if (!(ok = mbar_wait_w(bar(B_KF + slot), (g / kKSlots) & 1, abort_flag, kWaitNs))) break;
        if (!(ok = mbar_wait_w(bar(B_SE + ss), ((g / kSSlots) & 1) ^ 1, abort_flag, kWaitNs))) break;
        tc_fence_after();
        const uint32_t k_lo = sdesc_lo(sbase + OFF_K + slot * kTile, 16);
        const uint32_t dS = tbase + kTS + ss * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
          mma_f16_lo_w(dS, q_lo + off, k_lo + off, kDescHi, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar(B_SF + ss));
        mma_commit_w(bar(B_KE + slot));
      }
      // Q's first release: every S of the unit is done (the epilogue, which
      // stages the output tile in the slot, gives the second)
      if (ok) mma_commit_w(bar(B_QE + qb));
      pc += npairs;
      uc += 1;
    }
    if (!ok && lane == 0) fail(FBM_DEVERR_TIMEOUT);
    mma_commit_w(bar(B_DRAIN));
    if (!mbar_wait_for_w(bar(B_DRAIN), 0, kWaitNs) && lane == 0) set_error(P.err, FBM_DEVERR_TIMEOUT);
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ PV issuer
    // (the whole warp runs the loop; one elected lane issues each MMA)
    // A = P (TMEM, K-major), B = V pair (MN-major: d contiguous)
    constexpr uint32_t idO = idesc_f16(kBf16, false, true, 128, D);
    const uint32_t tO = tbase + kTO;
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
      bool bad;
      const PUnit U = punit_of(P, u, &bad);
      if (U.n == 0) continue;
      const int npairs = (U.n + 1) >> 1;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, slot = g % kVSlots, pb = g % kPBufs;
        if (!(ok = mbar_wait_w(bar(B_PF + pb), (g / kPBufs) & 1, abort_flag, kWaitNs))) break;
        if (!(ok = mbar_wait_w(bar(B_VF + slot), (g / kVSlots) & 1, abort_flag, kWaitNs))) break;
        if (p == 0 && !(ok = mbar_wait_w(bar(B_OF), (uc & 1) ^ 1, abort_flag, kWaitNs))) break;
        tc_fence_after();
        const uint32_t v_lo = sdesc_lo(sbase + OFF_V + slot * kTile, kChunk);
        const uint32_t tP = tbase + kTP + pb * 64;
        const int steps = (2 * p + 1 >= U.n) ? 4 : 8;  // a half pair has 64 keys
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < steps)
            mma_f16_ta_w(tO, tP + kk * 8, v_lo + kk * 128, kDescHi, idO, (p > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(bar(B_PV + pb));
        mma_commit_w(bar(B_VE + slot));
      }
      pc += npairs;
      uc += 1;
    }
    if (!ok && lane == 0) fail(FBM_DEVERR_TIMEOUT);
    mma_commit_w(bar(B_DRAIN2));
    if (!mbar_wait_for_w(bar(B_DRAIN2), 0, kWaitNs) && lane == 0) set_error(P.err, FBM_DEVERR_TIMEOUT);
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    using E = typename std::conditional<kBf16, BF16, F16>::type;
    const int sw = warp & 3;                  // TMEM subpartition: rows 32 sw .. 32 sw + 31
    const int blk = (warp - kWarpSm) >> 2;    // kv block of each pair
    const int row = sw * 32 + lane;           // query row within the 128-row tile
    const int my_bit = sw < 2 ? 29 : 30;      // union-entry bit of this row's q block
    const int tid = threadIdx.x - kWarpSm * 32;
    const int pair_bar = kPairBar0 + sw;
    const uint32_t tl = tbase + ((uint32_t)(sw * 32) << 16);
    constexpr int kOC = D / 2;                // O columns of this thread: kOC * blk ..
    const uint64_t sl2x2 = f2_pack(P.sl2, P.sl2);
    volatile float *xmax = reinterpret_cast<volatile float *>(smem + OFF_XCH);
    volatile float *xsum = xmax + 2 * 2 * 128;
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units; u += gridDim.x) {
      bool bad;
      const PUnit U = punit_of(P, u, &bad);
      const int q0 = U.p * 128;
      const int rows = min(128, P.s_q - q0);
      if (U.n == 0) {
        uint16_t *o = static_cast<uint16_t *>(P.out) + ((size_t)U.bh_q * P.s_q + q0) * D;
        for (int e = tid * 8; e < rows * D; e += kSoftmaxThreads * 8)
          *reinterpret_cast<uint4 *>(o + e) = make_uint4(0, 0, 0, 0);
        if (P.lse && tid < rows) P.lse[(size_t)U.bh_q * P.s_q + q0 + tid] = -INFINITY;
        continue;
      }
      const int npairs = (U.n + 1) >> 1;
      const int qpos = q0 + row;
      const int qb = uc & 1;
      float m = -INFINITY;                 // running max of the row (log2 domain)
      uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};
      int e_next = blk < U.n ? pentry(U, blk) : -1;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, ss = g % kSSlots, pb = g % kPBufs;
        const int e = e_next;
        {
          const int tn = 2 * (p + 1) + blk;
          e_next = (p + 1 < npairs && tn < U.n) ? pentry(U, tn) : -1;
        }
        const int j = e & kEntryMask;
        const bool jvalid = e >= 0 && j < P.nk && ((e >> my_bit) & 1);
        const int kpos0 = (jvalid ? j : 0) * 64;
        const bool plain = jvalid && kpos0 + 64 <= P.s_k && (!P.causal || kpos0 + 63 <= qpos + P.koff);
        ok = mbar_wait_ok(ok, bar(B_SF + ss), (g / kSSlots) & 1, abort_flag, kWaitNs);
        tc_fence_after();
        uint32_t sv[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv + 32);
          tmem_ld32(tl + kTS + ss * 128 + blk * 64, lo);
          tmem_ld32(tl + kTS + ss * 128 + blk * 64 + 32, hi);
        }
        tmem_wait_ld();
        // the S slot is free for S(g + kSSlots) as soon as it is in registers
        tc_fence_before();
        __syncwarp();
        mbar_arrive_lane0(bar(B_SE + ss), lane);
        if (!plain) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int kpos = kpos0 + c;
            const bool vis = jvalid && kpos < P.s_k && (!P.causal || kpos <= qpos + P.koff);
            if (!vis) sv[c] = __float_as_uint(-INFINITY);
          }
        }
        float mx;
        {
          float t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float *v = reinterpret_cast<const float *>(sv) + 8 * i;
            t[i] = fmaxf(fmax3(fmax3(v[0], v[1], v[2]), v[3], v[4]), fmax3(v[5], v[6], v[7]));
          }
          mx = fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
        }
        const float mxs = mx * P.sl2;
        // agree with the partner warp (the other kv block of the same rows)
        volatile float *xm = xmax + (g & 1) * 256;
        xm[blk * 128 + row] = mxs;
        const bool any_need = named_or(pair_bar, 64, mxs > m + 8.0f);
        if (any_need) {
          // rare: a score of these rows exceeds the running max by more than
          // 2^8 (always on the first pair): move the max to the pair's row
          // max, rescale l and this warp's columns of O
          const float mrow = fmaxf(mxs, xm[(blk ^ 1) * 128 + row]);
          const float mn = mrow > m + 8.0f ? mrow : m;
          const float alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - mn);
          m = mn;
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 4; ++i) l2[i] = f2_mul(l2[i], a2);
          if (p > 0) {
            const int gp = g - 1;
            ok = mbar_wait_ok(ok, bar(B_PV + gp % kPBufs), (gp / kPBufs) & 1, abort_flag, kWaitNs);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < kOC / 32; ++h) {
              uint32_t o[32];
              tmem_ld32(tl + kTO + blk * kOC + h * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const float2 w2 = f2_unpack(
                    f2_mul(f2_pack(__uint_as_float(o[c]), __uint_as_float(o[c + 1])), a2));
                o[c] = __float_as_uint(w2.x);
                o[c + 1] = __float_as_uint(w2.y);
              }
              tmem_st32(tl + kTO + blk * kOC + h * 32, o);
            }
            tmem_wait_st();
          }
        }
        // P = exp2(s * scale * log2 e - m), packed to 16-bit pairs.  A block
        // outside this q block's LUT row (the same for the whole warp: its 32
        // rows share a q block) has P = 0 and needs no exponential.
        uint32_t pk[32];
        if (jvalid) {
          const float mu = (m == -INFINITY) ? 0.f : m;
          const uint64_t negm = f2_pack(-mu, -mu);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 xv = f2_unpack(
                f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), sl2x2, negm));
            const float e0 = fast_exp2(xv.x), e1 = fast_exp2(xv.y);
            l2[i & 3] = f2_add(l2[i & 3], f2_pack(e0, e1));
            pk[i] = E::from_f2(e0, e1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = 0u;
        }
        // P buffer pb was last read by PV(g - kPBufs): wait for the previous
        // completion of its barrier (on a fresh barrier the phase before the
        // first counts as complete, so the first uses pass at once)
        ok = mbar_wait_ok(ok, bar(B_PV + pb), ((g / kPBufs) & 1) ^ 1, abort_flag, kWaitNs);
        tc_fence_after();
        tmem_st32(tl + kTP + pb * 64 + blk * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_lane0(bar(B_PF + pb), lane);
      }
      // ---- epilogue: O = O / l, LSE = m ln 2 + ln l
      const int gl = pc + npairs - 1;
      ok = mbar_wait_ok(ok, bar(B_PV + gl % kPBufs), (gl / kPBufs) & 1, abort_flag, kWaitNs);
      tc_fence_after();
      uint32_t o[kOC];
#pragma unroll
      for (int h = 0; h < kOC / 32; ++h) {
        uint32_t (&oh)[32] = *reinterpret_cast<uint32_t(*)[32]>(o + 32 * h);
        tmem_ld32(tl + kTO + blk * kOC + h * 32, oh);
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_lane0(bar(B_OF), lane);  // O may take the next unit's first PV
      float lt;
      {
        const float2 a = f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
        lt = a.x + a.y;
      }
      xsum[blk * 128 + row] = lt;
      named_sync(pair_bar, 64);
      lt += xsum[(blk ^ 1) * 128 + row];
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      if (P.lse && blk == 0 && row < rows)
        P.lse[(size_t)U.bh_q * P.s_q + q0 + row] = lt > 0.f ? m * 0.6931471805599453f + logf(lt)
                                                            : -INFINITY;
      // staging in the (dead) Q slot: columns kOC blk .. of row `row`, 16-byte
      // pieces in the 128-byte-swizzled [chunk][128 rows][128 B] tile
      const uint32_t stage = OFF_Q + qb * kTile;
      const int col0 = kOC * blk;
      uint8_t *srow = smem + stage + (col0 / 64) * kChunk + row * 128;
#pragma unroll
      for (int c = 0; c < kOC / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int z = 0; z < 4; ++z)
          w[z] = E::from_f2(__uint_as_float(o[8 * c + 2 * z]) * inv,
                            __uint_as_float(o[8 * c + 2 * z + 1]) * inv);
        const int piece = (col0 % 64) / 8 + c;
        *reinterpret_cast<uint4 *>(srow + ((piece ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async();
      named_sync(kSoftmaxBar, kSoftmaxThreads);
      if (tid == 0) {
        // rows past the end of the sequence are clipped by the tensor map
#pragma unroll
        for (int c = 0; c < kNch; ++c)
          tma_store_3d(&P.to, sbase + stage + c * kChunk, c * 64, q0, U.bh_q);
        bulk_commit();
        bulk_wait_read0();
        mbar_arrive(bar(B_QE + qb));  // the tile has been read out: the Q slot is free
      }
      named_sync(kSoftmaxBar, kSoftmaxThreads);
      pc += npairs;
      uc += 1;
    }
    if (!ok) fail(FBM_DEVERR_TIMEOUT);
    if (tid == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpS) {
    __syncwarp();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// [bh, s, d] 16-bit tensor, box = 64 d x `rows` rows x 1 head, 128B swizzle
bool pmap(CUtensorMap *m, const void *base, int bh, int s, int d, int rows, bool bf16) {
  auto enc = tma_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)s * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

template <int D, bool BF16>
cudaError_t launch_p(const FmhaLaunch &L, cudaStream_t st) {
  constexpr int SMEM_ALLOC = PLay<D>::SMEM_ALLOC;
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_fmha_pair<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev].store(true, std::memory_order_release);
  }
  PairParams P;
  memset(&P, 0, sizeof(P));
  if (!pmap(&P.tq, L.q, L.b * L.hq, L.s_q, D, 128, BF16) ||
      !pmap(&P.tk, L.k, L.b * L.hk, L.s_k, D, 64, BF16) ||
      !pmap(&P.tv, L.v, L.b * L.hk, L.s_k, D, 64, BF16) ||
      !pmap(&P.to, L.out, L.b * L.hq, L.s_q, D, 128, BF16))
    return cudaErrorInvalidValue;
  P.lut = L.lut;
  P.cnt = L.cnt;
  P.out = L.out;
  P.lse = L.lse;
  P.err = L.err;
  P.b = L.b; P.hq = L.hq; P.hk = L.hk; P.s_q = L.s_q; P.s_k = L.s_k; P.nq = L.nq; P.nk = L.nk;
  P.npq = (L.nq + 1) / 2;
  P.lut_stride = L.lut_stride;
  P.causal = L.causal;
  P.koff = L.key_offset;
  P.units = L.b * L.hq * P.npq;
  P.sl2 = L.scale * 1.4426950408889634f;
  const int grid = std::min(P.units, device_sm_count());
  k_fmha_pair<D, BF16><<<grid, kThreads, SMEM_ALLOC, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fmha_pair(const FmhaLaunch &L, cudaStream_t st) {
  if (L.d == 128) return L.bf16 ? launch_p<128, true>(L, st) : launch_p<128, false>(L, st);
  return L.bf16 ? launch_p<64, true>(L, st) : launch_p<64, false>(L, st);
}

}  // namespace fbm
