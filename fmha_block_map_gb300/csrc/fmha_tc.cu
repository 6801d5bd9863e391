// Sparse FMHA forward for sm_103a on 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA loads and stores), d = 128.
//
// A work unit is one (batch, head, q block, split): with num_splits = S the
// q block's kv list is cut into S contiguous chunks (the first n mod S hold
// ceil(n / S) entries) and each chunk is a unit.  Whole rows (S = 1 with a
// dtype output) leave through a swizzled staging tile and TMA stores; split
// chunks, and whole rows asked for as fp32 partials, are written as fp32 O
// (already divided by the row sum) and LSE straight from registers.
//
// The per-q-block work of the sparse FMHA stage (the "Sparge Attention
// (Composable Kernel)" README) visits only the kv blocks of the q block's LUT
// row, two at a time (a "pair", 128 keys):
//
//   S  [64 q x 128 keys]  = Q [64 x d] . K_pair^T        M = 64, N = 128 (A, B in smem)
//   P  = exp2(S * scale * log2 e - m)                      written to TMEM as fp16 / bf16
//   O  [64 q x 128 d]    += P . V_pair                    M = 64, N = 128 (A = P in TMEM,
//                                                          B = V in smem, MN-major)
//
// Why this orientation: an M = 64 MMA runs at half the rate of an M = 128 one,
// but the tensor core reads its operands from shared memory at about 128 bytes
// per cycle, and with P in TMEM a pair costs 48 KB (S) + 32 KB (PV) of operand
// reads plus 64 KB of TMA writes: about 1100 cycles, close to the 1024 cycles
// the sixteen M = 64 MMAs take.  (The transposed form, S^T = K . Q^T with M = 128
// keys, needs P^T in shared memory: 176 KB per pair.)
//
// TMEM (512 columns): S slots at columns 0 and 128 (fp32), P buffers at 256 and
// 320 (two 16-bit values per column), O at 384.  An M = 64 accumulator keeps
// row i in lane (i mod 16) + 32 (i / 16): softmax warp w (subpartition w) owns
// rows 16w .. 16w + 15, and with the 16x32bx2 load shape thread t holds row
// 16w + (t mod 16), keys 64 (t / 16) .. + 63 of the pair, i.e. one kv block.
// The running max of a row is kept lazily (O and l are rescaled only when a
// score exceeds it by more than 2^8); both threads of a row agree on it through
// one shuffle.
//
// Roles (one persistent CTA per SM; 12 warps for whole rows, 8 for fp32 partials):
//   warp 0   TMA producer of Q (double buffer) and K pairs (3-slot ring)
//   warp 1   TMA producer of V pairs (2-slot ring)
//   warp 2   TMEM owner and S issuer
//   warp 3   PV issuer
//   warps 4-7 softmax (TMEM subpartitions 0-3); fp32 partials leave from here
//   warps 8-11 epilogue of whole rows: a row's sum and max come from the
//            softmax warps through shared memory, O from TMEM once the row's
//            last PV is done, so the softmax warps go straight on to the next
//            row.  setmaxnreg gives the softmax warpgroup 232 registers, the
//            other two 88 and 120.
// Pipeline: S(g) is issued once K(g) has landed and its TMEM slot is free (the
// softmax releases a slot as soon as it holds the scores in registers), so the
// S MMA of pair g + 1 runs during the softmax of pair g; PV(g) once P(g) is in
// TMEM.  Every wait is bounded: on expiry the kernel raises FBM_DEVERR_TIMEOUT,
// every role leaves its loop, in-flight copies and MMAs are drained with
// bounded waits and TMEM is freed.
//
// Loop shape: the Incremental_FlashAttention updating_log's Stage 3/4 sparse
// mainloop (listed blocks only, next K prefetched while the current tile is
// consumed, an empty list writes O = 0 and LSE = -inf).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <type_traits>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {
namespace {

using namespace tc;

constexpr int kQChunk = 64 * 128;         // 8 KB: one 64-wide d chunk of a 64-row tile
constexpr int kPairChunk = 128 * 128;     // 16 KB: one 64-wide d chunk of a 128-row pair
constexpr int kKSlots = 3;                // K ring (S(g) may run ahead of the softmax)
constexpr int kVSlots = 2;                // V ring
constexpr int kSSlots = 2;                // S slots in TMEM
constexpr int kPBufs = 2;                 // P buffers in TMEM

enum {
  B_QF = 0, B_QE = 2, B_KF = 4, B_KE = B_KF + kKSlots, B_VF = B_KE + kKSlots,
  B_VE = B_VF + kVSlots, B_SF = B_VE + kVSlots, B_SE = B_SF + kSSlots, B_PF = B_SE + kSSlots,
  B_PV = B_PF + kPBufs, B_OF = B_PV + kPBufs, B_DRAIN = B_OF + 1, B_DRAIN2 = B_DRAIN + 1,
  B_PVI = B_DRAIN2 + 1,
  // whole rows: the softmax warps hand each row's sum and max to the epilogue
  // warpgroup through two slots (full / free)
  B_STF = B_PVI + 1, B_STE = B_STF + 2, NBAR = B_STE + 2
};
// Shared-memory layout for head dim D (64 or 128): a 64-row tile of D 16-bit
// values is D / 64 chunks of 64 columns (128-byte rows, 128-byte swizzle).
template <int D>
struct Lay {
  static constexpr int NCH = D / 64;             // 64-wide d chunks
  static constexpr int QBytes = 64 * D * 2;      // a 64-row Q (or output) tile
  static constexpr int PairBytes = 128 * D * 2;  // two 64-row kv blocks
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QBytes;
  static constexpr int OFF_V = OFF_K + kKSlots * PairBytes;
  static constexpr int OFF_STAGE = OFF_V + kVSlots * PairBytes;  // output tile [chunk][64 rows][128 B]
  static constexpr int OFF_BAR = OFF_STAGE + QBytes;
  // [0] tmem base, [1] abort flag, bytes 8 .. 15: PV-skip votes [P buffer][softmax warp]
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_STATS = OFF_MISC + 16;  // [slot][64 rows][max, sum] floats
  static constexpr int SMEM_ALLOC = OFF_STATS + 2 * 64 * 2 * 4 + 1024;
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTS = 0;    // S slot s at kTS + 128 s
constexpr uint32_t kTP = 256;  // P buffer b at kTP + 64 b
constexpr uint32_t kTO = 384;  // O (D columns)
constexpr uint32_t kDescHi = sdesc_hi_sw128(1024);  // every operand: 1024-byte 8-row atoms
constexpr uint64_t kWaitNs = 2000000000ull;          // 2 s per wait

constexpr int kWarpQK = 0, kWarpV = 1, kWarpS = 2, kWarpPV = 3, kWarpSm = 4;
constexpr int kSoftmaxWarps = 4;
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 32 * (kWarpSm + kSoftmaxWarps);
// whole rows: warps 8-11 are the epilogue warpgroup
constexpr int kWarpEp = kWarpSm + kSoftmaxWarps;
constexpr int kThreadsEp = kThreads + 32 * kSoftmaxWarps;
constexpr int kSoftmaxBar = 1;  // named barrier of the warps that store O (4 warps)
// register budgets of the three warpgroups with an epilogue warpgroup:
// 128 x (88 + 232 + 120) = 56320, within the 384 x 168 the CTA is launched with
constexpr uint32_t kRegsIo = 88, kRegsSoftmax = 232, kRegsEp = 120;

struct TcParams {
  CUtensorMap tq, tk, tv, to;
  const int32_t *lut, *cnt;
  void *out;      // dtype output (whole rows), or
  float *opart;   // fp32 partials [splits, b * hq * s_q, D] (split-KV / partial mode)
  float *lse;     // [b * hq * s_q], or [splits, b * hq * s_q] with opart
  uint32_t *err;
  int b, hq, hk, s_q, s_k, nq, nk, lut_stride, causal, splits, units;
  int koff;       // causal: key index u visible to query row t when u <= t + koff
  size_t plane;   // b * hq * s_q
  float sl2;      // scale * log2(e)
  float tau2;     // pv_threshold * log2(e) (PV-skip variant)
  const float *qscale, *kscale;  // fp8 variant: [b * hq, nq] and [b * hk, nk] block scales
};

// one (batch, head, q block, split): kv-list entries off .. off + n of the row
struct Unit {
  int bh_q, bh_k, i, split, off, n, nk;
  const int32_t *row;  // the LUT row's first entry (nullptr: dense)
  bool bad_count;      // the row's count lay outside [0, min(nk, lut_stride)]
};

template <bool kPartial>
FBM_DEVICE Unit unit_of(const TcParams &P, int u) {
  Unit U;
  // whole rows (no partial output) are never split: keep the division out of
  // that kernel
  const int qu = kPartial ? u / P.splits : u;
  U.split = u - qu * (kPartial ? P.splits : 1);
  U.bh_q = qu / P.nq;
  U.i = qu - U.bh_q * P.nq;
  const int b = U.bh_q / P.hq, h = U.bh_q - b * P.hq;
  U.bh_k = b * P.hk + h / (P.hq / P.hk);
  int n_list;
  U.nk = P.nk;
  U.bad_count = false;
  if (P.lut) {
    U.row = P.lut + (size_t)qu * P.lut_stride;
    const int raw = __ldg(P.cnt + qu), lim = min(P.nk, P.lut_stride);
    U.bad_count = raw < 0 || raw > lim;
    n_list = max(0, min(raw, lim));
  } else {
    U.row = nullptr;
    // dense: every kv block up to the one holding the q block's last visible key
    const int lastk = U.i * 64 + 63 + P.koff;
    n_list = !P.causal ? P.nk : (lastk < 0 ? 0 : min(P.nk, lastk / 64 + 1));
  }
  if constexpr (kPartial) {
    // contiguous chunks: the first n mod S hold ceil(n / S) entries
    const int base = n_list / P.splits, extra = n_list - base * P.splits;
    U.off = U.split * base + min(U.split, extra);
    U.n = base + (U.split < extra ? 1 : 0);
  } else {
    U.off = 0;
    U.n = n_list;
  }
  return U;
}

// kv block of entry t of the unit's chunk (dense rows: the index itself).  The
// kernel checks the range of every entry (an entry outside [0, nk) is skipped
// and flagged); their order is the caller's contract, checked on request by
// lut_validate, so the read stays a plain load whose value nothing waits on
// until the pair after it.
FBM_DEVICE int entry_of(const Unit &U, int t) {
  return U.row ? __ldg(U.row + U.off + t) : U.off + t;
}

// O of one row as seen by one softmax thread: D / 2 columns (16x32bx2 shape,
// the two threads of a row holding the two halves)
template <int D>
FBM_DEVICE void ld_o(uint32_t taddr, uint32_t (&o)[D / 2]) {
  if constexpr (D == 128) tmem_ld_rowhalf64(taddr, o);
  else tmem_ld_rowhalf32(taddr, o);
}
template <int D>
FBM_DEVICE void st_o(uint32_t taddr, const uint32_t (&o)[D / 2]) {
  if constexpr (D == 128) tmem_st_rowhalf64(taddr, o);
  else tmem_st_rowhalf32(taddr, o);
}

template <int D, bool kBf16, bool kPartial, bool kPvSkip, bool kFp8>
__global__ void __launch_bounds__(kPartial ? kThreads : kThreadsEp, 1)
    k_fmha_tc(const __grid_constant__ TcParams P) {
  // whole rows leave through the epilogue warpgroup; fp32 partials straight
  // from the softmax warps' registers
  constexpr bool kEpi = !kPartial;
  static_assert(!(kFp8 && (kPartial || kPvSkip)), "the fp8 variant runs whole rows");
  static_assert(!kFp8 || D == 128, "fp8 Q / K at d = 128");
  using Ly = Lay<D>;
  constexpr int OFF_Q = Ly::OFF_Q, OFF_K = Ly::OFF_K, OFF_V = Ly::OFF_V,
                OFF_STAGE = Ly::OFF_STAGE, OFF_BAR = Ly::OFF_BAR, OFF_MISC = Ly::OFF_MISC;
  constexpr int kQBytes = Ly::QBytes, kPairBytes = Ly::PairBytes, kNch = Ly::NCH;
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
      if ((k >= B_SE && k < B_SE + kSSlots) || (k >= B_PF && k < B_PF + kPBufs) || k == B_OF ||
          (k >= B_STF && k < B_STE + 2))
        cnt = kSoftmaxWarps;  // one elected arrive per softmax (or epilogue) warp
      mbar_init(bar(k), cnt);
    }
    misc[1] = 0;
    fence_mbar_init();
    prefetch_map(&P.tq);
    prefetch_map(&P.tk);
    prefetch_map(&P.tv);
    if (!kPartial) prefetch_map(&P.to);
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

  // K or V pair g (= pc + p) of a q block into its ring slot, once the MMA that
  // last read the slot has completed
  auto load_pair = [&](const Unit &U, int pc, int p, bool is_v) -> bool {
    const int ns = is_v ? kVSlots : kKSlots;
    const int g = pc + p, slot = g % ns;
    const int fb = (is_v ? B_VF : B_KF) + slot, eb = (is_v ? B_VE : B_KE) + slot;
    if (!mbar_wait(bar(eb), ((g / ns) & 1) ^ 1, abort_flag, kWaitNs)) return false;
    int js[2] = {-1, -1};
    uint32_t bytes = 0;
    // an fp8 K block is one 128-byte-wide box; a 16-bit block is D / 64
    const int nchunk = (kFp8 && !is_v) ? 1 : kNch;
    for (int hf = 0; hf < 2; ++hf) {
      const int t = 2 * p + hf;
      if (t >= U.n) break;
      int j = entry_of(U, t);
      if (j < 0 || j >= P.nk) {
        // out of range: flagged (by the K producer); block 0 is fetched in
        // its place so that the masked keys (P = 0) meet finite V rows
        if (!is_v) set_error(P.err, FBM_DEVERR_LUT_RANGE);
        j = 0;
      }
      js[hf] = j;
      bytes += nchunk * kQChunk;
    }
    mbar_arrive_tx(bar(fb), bytes);
    const uint32_t dst0 = sbase + (is_v ? OFF_V : OFF_K) + slot * kPairBytes;
    for (int hf = 0; hf < 2; ++hf) {
      if (js[hf] < 0) continue;
      for (int c = 0; c < nchunk; ++c)
        tma_load_3d(dst0 + c * kPairChunk + hf * kQChunk, is_v ? &P.tv : &P.tk, c * 64,
                    js[hf] * 64, U.bh_k, bar(fb));
    }
    return true;
  };

  if (warp == kWarpQK) {
    // ------------------------------------------------------------ Q and K producer
    if constexpr (kEpi) regs_decrease<kRegsIo>();
    if (lane == 0) {
      int pc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of<kPartial>(P, u);
        if (U.bad_count && U.split == 0) set_error(P.err, FBM_DEVERR_LUT_RANGE);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        const int qb = uc & 1;
        if (!(ok = mbar_wait(bar(B_QE + qb), ((uc >> 1) & 1) ^ 1, abort_flag, kWaitNs))) break;
        constexpr int qchunks = kFp8 ? 1 : kNch;  // an fp8 Q tile is one 128-byte-wide box
        mbar_arrive_tx(bar(B_QF + qb), qchunks * kQChunk);
        for (int c = 0; c < qchunks; ++c)
          tma_load_3d(sbase + OFF_Q + qb * kQBytes + c * kQChunk, &P.tq, c * 64, U.i * 64,
                      U.bh_q, bar(B_QF + qb));
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc, p, false);
        pc += npairs;
        uc += 1;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kWarpV) {
    // ------------------------------------------------------------ V producer
    if constexpr (kEpi) regs_decrease<kRegsIo>();
    if (lane == 0) {
      int pc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
        const Unit U = unit_of<kPartial>(P, u);
        if (U.n == 0) continue;
        const int npairs = (U.n + 1) >> 1;
        for (int p = 0; p < npairs && ok; ++p) ok = load_pair(U, pc, p, true);
        pc += npairs;
      }
      if (!ok) fail(FBM_DEVERR_TIMEOUT);
    }
  } else if (warp == kWarpS) {
    // ------------------------------------------------------------ S issuer
    if constexpr (kEpi) regs_decrease<kRegsIo>();
    // (the whole warp runs the loop; one elected lane issues each MMA)
    // (kind::f8f6f4 with e4m3 A and B uses format code 0, as f16 does)
    constexpr uint32_t idS = idesc_f16(kFp8 ? false : kBf16, false, false, 64, 128);
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
      const Unit U = unit_of<kPartial>(P, u);
      if (U.n == 0) continue;
      const int npairs = (U.n + 1) >> 1;
      const int qb = uc & 1;
      if (!(ok = mbar_wait_w(bar(B_QF + qb), (uc >> 1) & 1, abort_flag, kWaitNs))) break;
      tc_fence_after();
      const uint32_t q_lo = sdesc_lo(sbase + OFF_Q + qb * kQBytes, 16);
      // the previous row's last PV goes into the tensor pipe before this row's
      // first S, so the previous row's epilogue does not wait behind it
      if (uc > 0 && !(ok = mbar_wait_w(bar(B_PVI), (uc - 1) & 1, abort_flag, kWaitNs))) break;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, slot = g % kKSlots, ss = g % kSSlots;
        if (!(ok = mbar_wait_w(bar(B_KF + slot), (g / kKSlots) & 1, abort_flag, kWaitNs))) break;
        if (!(ok = mbar_wait_w(bar(B_SE + ss), ((g / kSSlots) & 1) ^ 1, abort_flag, kWaitNs))) break;
        tc_fence_after();
        const uint32_t k_lo = sdesc_lo(sbase + OFF_K + slot * kPairBytes, 16);
        const uint32_t dS = tbase + kTS + ss * 128;
        if constexpr (kFp8) {
          // e4m3 rows are 128 bytes: one swizzle atom wide, 32 values of K per MMA
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_f8_lo_w(dS, q_lo + ((kk * 32) >> 4), k_lo + ((kk * 32) >> 4), kDescHi, idS,
                        kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_lo_w(dS, q_lo + (((kk >> 2) * kQChunk + (kk & 3) * 32) >> 4),
                         k_lo + (((kk >> 2) * kPairChunk + (kk & 3) * 32) >> 4), kDescHi, idS,
                         kk > 0 ? 1u : 0u);
        }
        mma_commit_w(bar(B_SF + ss));
        mma_commit_w(bar(B_KE + slot));
      }
      if (ok) mma_commit_w(bar(B_QE + qb));  // Q free once every S of the row is done
      pc += npairs;
      uc += 1;
    }
    if (!ok && lane == 0) fail(FBM_DEVERR_TIMEOUT);
    // drain: every MMA this warp issued has completed before TMEM is freed
    mma_commit_w(bar(B_DRAIN));
    if (!mbar_wait_for_w(bar(B_DRAIN), 0, kWaitNs) && lane == 0) set_error(P.err, FBM_DEVERR_TIMEOUT);
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ PV issuer
    if constexpr (kEpi) regs_decrease<kRegsIo>();
    // (the whole warp runs the loop; one elected lane issues each MMA)
    // A = P (TMEM, K-major), B = V pair (MN-major: d contiguous)
    constexpr uint32_t idO = idesc_f16(kBf16, false, true, 64, D);
    const uint32_t tO = tbase + kTO;
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units && ok; u += gridDim.x) {
      const Unit U = unit_of<kPartial>(P, u);
      if (U.n == 0) continue;
      const int npairs = (U.n + 1) >> 1;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, slot = g % kVSlots, pb = g % kPBufs;
        if (!(ok = mbar_wait_w(bar(B_PF + pb), (g / kPBufs) & 1, abort_flag, kWaitNs))) break;
        if (!(ok = mbar_wait_w(bar(B_VF + slot), (g / kVSlots) & 1, abort_flag, kWaitNs))) break;
        if (p == 0 && !(ok = mbar_wait_w(bar(B_OF), (uc & 1) ^ 1, abort_flag, kWaitNs))) break;
        tc_fence_after();
        const uint32_t v_lo = sdesc_lo(sbase + OFF_V + slot * kPairBytes, kPairChunk);
        const uint32_t tP = tbase + kTP + pb * 64;
        const bool half = 2 * p + 1 >= U.n;  // a half pair has 64 keys: 4 steps
        bool skip_a = false, skip_b = false;
        if constexpr (kPvSkip) {
          // a block is skipped when all four softmax warps voted for it; the
          // first block of a row never is (its running max is still -inf), so
          // the first MMA below always starts the accumulator
          const uint32_t vw = __shfl_sync(
              0xffffffffu, *reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC + 8 + pb * 4), 0);
          const uint32_t all4 = vw & (vw >> 8) & (vw >> 16) & (vw >> 24);
          skip_a = (all4 & 1u) != 0;
          skip_b = (all4 & 2u) != 0;
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < 4 ? !skip_a : (!half && !skip_b))
            mma_f16_ta_w(tO, tP + kk * 8, v_lo + kk * 128, kDescHi, idO,
                         (p > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(bar(B_PV + pb));
        mma_commit_w(bar(B_VE + slot));
        if (p == npairs - 1) mbar_arrive_lane0(bar(B_PVI), lane);  // the row's last PV is issued
      }
      pc += npairs;
      uc += 1;
    }
    if (!ok && lane == 0) fail(FBM_DEVERR_TIMEOUT);
    mma_commit_w(bar(B_DRAIN2));
    if (!mbar_wait_for_w(bar(B_DRAIN2), 0, kWaitNs) && lane == 0) set_error(P.err, FBM_DEVERR_TIMEOUT);
  } else if (kEpi && warp >= kWarpEp) {
    // ------------------------------------------------------------ epilogue warpgroup
    // (whole rows) per row: the row's sum and max from the softmax warps, the
    // row's last PV, O out of TMEM (then O is free for the next row's first
    // PV), O / l through a swizzled staging tile and a tensor store, the LSE.
    // The softmax warps meanwhile work on the next row.
    regs_decrease<kRegsEp>();
    using E = typename std::conditional<kBf16, BF16, F16>::type;
    const int sw = warp - kWarpEp;            // TMEM subpartition
    const int half = lane >> 4;               // d half of O
    const int row = sw * 16 + (lane & 15);    // query row within the q block
    const int tid = threadIdx.x - kWarpEp * 32;
    const uint32_t tl = tbase + ((uint32_t)(sw * 32) << 16);
    volatile float *stats = reinterpret_cast<volatile float *>(smem + Ly::OFF_STATS);
    int pc = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.units; u += gridDim.x) {
      const Unit U = unit_of<false>(P, u);
      const int q0 = U.i * 64;
      const int rows = min(64, P.s_q - q0);
      const size_t orow0 = (size_t)U.bh_q * P.s_q + q0;
      if (U.n == 0) {
        uint16_t *o = static_cast<uint16_t *>(P.out) + orow0 * D;
        for (int e = tid * 8; e < rows * D; e += kSoftmaxThreads * 8)
          *reinterpret_cast<uint4 *>(o + e) = make_uint4(0, 0, 0, 0);
        if (P.lse && tid < rows) P.lse[orow0 + tid] = -INFINITY;
        continue;
      }
      const int npairs = (U.n + 1) >> 1;
      const int gl = pc + npairs - 1, rb = uc & 1;
      ok = mbar_wait_ok(ok, bar(B_STF + rb), (uc >> 1) & 1, abort_flag, kWaitNs);
      const float m = stats[(rb * 64 + row) * 2], lt = stats[(rb * 64 + row) * 2 + 1];
      __syncwarp();
      mbar_arrive_lane0(bar(B_STE + rb), lane);  // the slot may take row uc + 2
      // the softmax warps waited for PV(gl - 2) before the row's last P, and
      // before they handed the row over: the parity wait for PV(gl) is sound
      ok = mbar_wait_ok(ok, bar(B_PV + gl % kPBufs), (gl / kPBufs) & 1, abort_flag, kWaitNs);
      tc_fence_after();
      uint32_t o[D / 2];
      ld_o<D>(tl + kTO, o);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_lane0(bar(B_OF), lane);  // O may take the next row's first PV
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      if (P.lse && half == 0 && row < rows)
        P.lse[orow0 + row] = lt > 0.f ? m * 0.6931471805599453f + logf(lt) : -INFINITY;
      // staging: d half `half` of row `row` as D / 16 pieces of 16 bytes in
      // the 128-byte-swizzled [chunk][64 rows][128 B] tile (d = 128: the half
      // is chunk `half`; d = 64: pieces 4 half .. 4 half + 3 of the one chunk).
      // The previous row's tensor store has long since read the tile.
      if (tid == 0) bulk_wait_read0();
      named_sync(kSoftmaxBar, kSoftmaxThreads);
      uint8_t *srow = smem + OFF_STAGE + (D == 128 ? half * kQChunk : 0) + row * 128;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int z = 0; z < 4; ++z)
          w[z] = E::from_f2(__uint_as_float(o[8 * c + 2 * z]) * inv,
                            __uint_as_float(o[8 * c + 2 * z + 1]) * inv);
        const int piece = D == 128 ? c : 4 * half + c;
        *reinterpret_cast<uint4 *>(srow + ((piece ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async();
      named_sync(kSoftmaxBar, kSoftmaxThreads);
      if (tid == 0) {
        // rows past the end of the sequence are clipped by the tensor map
#pragma unroll
        for (int c = 0; c < kNch; ++c)
          tma_store_3d(&P.to, sbase + OFF_STAGE + c * kQChunk, c * 64, q0, U.bh_q);
        bulk_commit();
      }
      pc += npairs;
      uc += 1;
    }
    if (!ok) fail(FBM_DEVERR_TIMEOUT);
    if (tid == 0) bulk_wait0();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    if constexpr (kEpi) regs_increase<kRegsSoftmax>();
    using E = typename std::conditional<kBf16, BF16, F16>::type;
    const int sw = warp - kWarpSm;            // == warp % 4: TMEM subpartition
    const int half = lane >> 4;               // block of the pair / d half of O
    const int row = sw * 16 + (lane & 15);    // query row within the q block
    const int tid = threadIdx.x - kWarpSm * 32;
    const uint32_t tl = tbase + ((uint32_t)(sw * 32) << 16);
    const uint64_t sl2x2 = f2_pack(P.sl2, P.sl2);
    // Every softmax thread runs the same loop trip counts and barriers whatever
    // happens: a failed (timed-out) wait only clears `ok`, and later waits
    // return at once.
    int pc = 0, uc = 0;
    bool ok = true;
    volatile float *stats = reinterpret_cast<volatile float *>(smem + Ly::OFF_STATS);
    for (int u = blockIdx.x; u < P.units; u += gridDim.x) {
      const Unit U = unit_of<kPartial>(P, u);
      const int q0 = U.i * 64;
      const int rows = min(64, P.s_q - q0);
      if (U.n == 0) {
        if constexpr (kEpi) continue;  // the epilogue warpgroup writes the empty row
        const size_t orow0 = (kPartial ? (size_t)U.split * P.plane : 0) + (size_t)U.bh_q * P.s_q + q0;
        if constexpr (kPartial) {
          float *o = P.opart + orow0 * D;
          for (int e = tid * 4; e < rows * D; e += kSoftmaxThreads * 4)
            *reinterpret_cast<float4 *>(o + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          uint16_t *o = static_cast<uint16_t *>(P.out) + orow0 * D;
          for (int e = tid * 8; e < rows * D; e += kSoftmaxThreads * 8)
            *reinterpret_cast<uint4 *>(o + e) = make_uint4(0, 0, 0, 0);
        }
        if (P.lse && tid < rows) P.lse[orow0 + tid] = -INFINITY;
        continue;
      }
      const int npairs = (U.n + 1) >> 1;
      const int qpos = q0 + row;
      const float qsl2 = kFp8 ? P.sl2 * __ldg(P.qscale + (size_t)U.bh_q * P.nq + U.i) : P.sl2;
      float m = -INFINITY;                 // running max of the row (log2 domain)
      float mt = -INFINITY;                // exact running max (PV-skip variant)
      uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};  // this thread's share of the row sum
      int j_next = half < U.n ? entry_of(U, half) : -1;
      for (int p = 0; p < npairs; ++p) {
        const int g = pc + p, ss = g % kSSlots, pb = g % kPBufs;
        const int j = j_next;
        {
          const int tn = 2 * (p + 1) + half;
          j_next = (p + 1 < npairs && tn < U.n) ? entry_of(U, tn) : -1;
        }
        const bool jvalid = j >= 0 && j < P.nk;
        const int kpos0 = (jvalid ? j : 0) * 64;
        // every key of this thread's block visible to its row
        const bool plain = jvalid && kpos0 + 64 <= P.s_k && (!P.causal || kpos0 + 63 <= qpos + P.koff);
        ok = mbar_wait_ok(ok, bar(B_SF + ss), (g / kSSlots) & 1, abort_flag, kWaitNs);
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld_rowhalf64(tl + kTS + ss * 128, sv);
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
        // row max over the pair (this thread's 64 keys, then the other half)
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
        // fp8: the two block scales fold into this thread's factor (its 64 keys
        // are one kv block); the pair max is then taken over scaled scores
        float fsc = P.sl2;
        if constexpr (kFp8) {
          fsc = qsl2 * (jvalid ? __ldg(P.kscale + (size_t)U.bh_k * P.nk + j) : 1.f);
          mx *= fsc;
        }
        uint32_t vote = 0;
        if constexpr (kPvSkip) {
          const float mx_other = __shfl_xor_sync(0xffffffffu, mx, 16);
          // block A (entry 2p) then block B (entry 2p + 1) against the exact
          // running max of the blocks visited before each; rows past the end
          // of the sequence do not veto
          const float a = (half == 0 ? mx : mx_other) * P.sl2;
          const float b = (half == 0 ? mx_other : mx) * P.sl2;
          const bool real = qpos < P.s_q;
          const bool sa = !real || a < mt - P.tau2;
          mt = fmaxf(mt, a);
          const bool sb = !real || b < mt - P.tau2;
          mt = fmaxf(mt, b);
          vote = (__all_sync(0xffffffffu, sa) ? 1u : 0u) | (__all_sync(0xffffffffu, sb) ? 2u : 0u);
          mx = fmaxf(mx, mx_other);
        } else {
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        }
        const float mxs = kFp8 ? mx : mx * P.sl2;
        const bool need = mxs > m + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
          // rare: some score of the warp's rows exceeds its running max by more
          // than 2^8 (always on the first pair): move the max, rescale l and O
          const float mn = need ? mxs : m;
          const float alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - mn);
          m = mn;
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 4; ++i) l2[i] = f2_mul(l2[i], a2);
          if (p > 0) {
            // O holds PV(0 .. p-1): wait for the last of them, then scale
            const int gp = g - 1;
            ok = mbar_wait_ok(ok, bar(B_PV + gp % kPBufs), (gp / kPBufs) & 1, abort_flag, kWaitNs);
            tc_fence_after();
            uint32_t o[D / 2];
            ld_o<D>(tl + kTO, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < D / 2; c += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[c]), __uint_as_float(o[c + 1])), a2);
              const float2 w2 = f2_unpack(v);
              o[c] = __float_as_uint(w2.x);
              o[c + 1] = __float_as_uint(w2.y);
            }
            st_o<D>(tl + kTO, o);
            tmem_wait_st();
          }
        }
        // P = exp2(s * scale * log2 e - m), packed to 16-bit pairs
        const float mu = (m == -INFINITY) ? 0.f : m;
        const uint64_t negm = f2_pack(-mu, -mu);
        const uint64_t fx2 = kFp8 ? f2_pack(fsc, fsc) : sl2x2;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                    fx2, negm);
          const float2 xv = f2_unpack(x);
          const float e0 = fast_exp2(xv.x), e1 = fast_exp2(xv.y);
          l2[i & 3] = f2_add(l2[i & 3], f2_pack(e0, e1));
          pk[i] = E::from_f2(e0, e1);
        }
        // P buffer pb was last read by PV(g - kPBufs): wait for the previous
        // completion of its barrier.  On a fresh barrier the phase before the
        // first counts as complete, so the first uses of a buffer pass at once
        // and the wait needs no branch around it (measured 4% faster).
        ok = mbar_wait_ok(ok, bar(B_PV + pb), ((g / kPBufs) & 1) ^ 1, abort_flag, kWaitNs);
        tc_fence_after();
        tmem_st_rowhalf32(tl + kTP + pb * 64, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (kPvSkip && lane == 0)  // read by the PV issuer once B_PF(pb) completes
          *reinterpret_cast<volatile uint8_t *>(smem + OFF_MISC + 8 + pb * 4 + sw) = (uint8_t)vote;
        mbar_arrive_lane0(bar(B_PF + pb), lane);
      }
      if constexpr (kEpi) {
        // the row's sum and max go to the epilogue warpgroup, which waits for
        // the row's last PV and stores O; this warp goes on to the next row
        float lt;
        {
          const float2 a = f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
          lt = a.x + a.y;
        }
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int rb = uc & 1;
        // slot rb was last read for row uc - 2 (on a fresh barrier the phase
        // before the first counts as complete)
        ok = mbar_wait_ok(ok, bar(B_STE + rb), ((uc >> 1) & 1) ^ 1, abort_flag, kWaitNs);
        if (half == 0) {
          stats[(rb * 64 + row) * 2] = m;
          stats[(rb * 64 + row) * 2 + 1] = lt;
        }
        __syncwarp();
        mbar_arrive_lane0(bar(B_STF + rb), lane);
        pc += npairs;
        uc += 1;
        continue;
      }
      // ---- fp32 partial (whole rows go to the epilogue warpgroup above):
      // O / l straight from registers, LSE = m ln 2 + ln l
      {
        const int gl = pc + npairs - 1;
        ok = mbar_wait_ok(ok, bar(B_PV + gl % kPBufs), (gl / kPBufs) & 1, abort_flag, kWaitNs);
        tc_fence_after();
        uint32_t o[D / 2];
        ld_o<D>(tl + kTO, o);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_lane0(bar(B_OF), lane);  // O may take the next row's first PV
        float lt;
        {
          const float2 a = f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])));
          lt = a.x + a.y;
        }
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const float inv = lt > 0.f ? 1.0f / lt : 0.f;
        const size_t orow0 = (size_t)U.split * P.plane + (size_t)U.bh_q * P.s_q + q0;
        if (P.lse && half == 0 && row < rows)
          P.lse[orow0 + row] = lt > 0.f ? m * 0.6931471805599453f + logf(lt) : -INFINITY;
        // this thread's D / 2 values of row `row`, d half `half`
        if (row < rows) {
          float4 *dst = reinterpret_cast<float4 *>(P.opart + (orow0 + row) * D + half * (D / 2));
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            dst[c] = make_float4(__uint_as_float(o[4 * c]) * inv, __uint_as_float(o[4 * c + 1]) * inv,
                                 __uint_as_float(o[4 * c + 2]) * inv,
                                 __uint_as_float(o[4 * c + 3]) * inv);
        }
      }
      pc += npairs;
    }
    if (!ok) fail(FBM_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpS) {
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

// [bh, s, d] 16-bit tensor (d = 64 or 128), box = 64 d x 64 rows x 1 head,
// 128B swizzle
bool make_map(CUtensorMap *m, const void *base, int bh, int s, int d, bool bf16) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)s * d * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// e4m3 codes [bh, s, 128]: one 128-byte-wide box of 64 rows, 128-byte swizzle
bool make_map8(CUtensorMap *m, const void *base, int bh, int s) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)s, (cuuint64_t)bh};
  cuuint64_t strides[2] = {128, (cuuint64_t)s * 128};
  cuuint32_t box[3] = {128, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;

int sm_count() {
  static int n[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

template <int D, bool BF16, bool PARTIAL, bool PVSKIP, bool FP8 = false>
cudaError_t launch_t(const FmhaLaunch &L, cudaStream_t st) {
  constexpr int SMEM_ALLOC = Lay<D>::SMEM_ALLOC;
  static_assert(!(PARTIAL && PVSKIP), "the PV skip runs on whole rows only");
  // the shared-memory attribute is per device: set it once on each
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_fmha_tc<D, BF16, PARTIAL, PVSKIP, FP8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev].store(true, std::memory_order_release);
  }
  TcParams P;
  memset(&P, 0, sizeof(P));
  const bool qk_ok = FP8 ? (make_map8(&P.tq, L.q, L.b * L.hq, L.s_q) &&
                            make_map8(&P.tk, L.k, L.b * L.hk, L.s_k))
                         : (make_map(&P.tq, L.q, L.b * L.hq, L.s_q, D, BF16) &&
                            make_map(&P.tk, L.k, L.b * L.hk, L.s_k, D, BF16));
  if (!qk_ok || !make_map(&P.tv, L.v, L.b * L.hk, L.s_k, D, BF16) ||
      (L.out && !make_map(&P.to, L.out, L.b * L.hq, L.s_q, D, BF16)))
    return cudaErrorInvalidValue;
  P.lut = L.lut;
  P.cnt = L.cnt;
  P.out = L.out;
  P.opart = PARTIAL ? L.o_part : nullptr;
  P.lse = PARTIAL ? L.lse_part : L.lse;
  P.splits = L.num_splits;
  P.plane = (size_t)L.b * L.hq * L.s_q;
  P.err = L.err;
  P.b = L.b; P.hq = L.hq; P.hk = L.hk; P.s_q = L.s_q; P.s_k = L.s_k; P.nq = L.nq; P.nk = L.nk;
  P.lut_stride = L.lut_stride;
  P.causal = L.causal;
  P.koff = L.key_offset;
  P.units = L.b * L.hq * L.nq * L.num_splits;
  P.sl2 = L.scale * 1.4426950408889634f;
  P.tau2 = L.pv_threshold * 1.4426950408889634f;
  P.qscale = L.q_scale;
  P.kscale = L.k_scale;
  const int grid = std::min(P.units, sm_count());
  k_fmha_tc<D, BF16, PARTIAL, PVSKIP, FP8><<<grid, PARTIAL ? kThreads : kThreadsEp, SMEM_ALLOC, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() { return get_encode(); }
int device_sm_count() { return sm_count(); }

bool fmha_tc_supported(int d, int dv, int num_splits, int s_q, int s_k) {
  return (d == 64 || d == 128) && dv == d && num_splits >= 1 && s_q > 0 && s_k > 0;
}

namespace {
template <int D>
cudaError_t launch_d(const FmhaLaunch &L, cudaStream_t st) {
  // whole rows in dtype, or fp32 partials (split chunks, or rows for a combine)
  if (L.out == nullptr)
    return L.bf16 ? launch_t<D, true, true, false>(L, st) : launch_t<D, false, true, false>(L, st);
  if (L.pv_threshold < INFINITY)
    return L.bf16 ? launch_t<D, true, false, true>(L, st) : launch_t<D, false, false, true>(L, st);
  return L.bf16 ? launch_t<D, true, false, false>(L, st) : launch_t<D, false, false, false>(L, st);
}
}  // namespace

cudaError_t launch_fmha_tc(const FmhaLaunch &L, cudaStream_t st) {
  if (L.q_scale)  // e4m3 Q and K, d = 128 (whole rows; the caller has checked)
    return L.bf16 ? launch_t<128, true, false, false, true>(L, st)
                  : launch_t<128, false, false, false, true>(L, st);
  return L.d == 128 ? launch_d<128>(L, st) : launch_d<64>(L, st);
}

}  // namespace fbm
