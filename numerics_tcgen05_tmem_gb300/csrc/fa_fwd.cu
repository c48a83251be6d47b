// Attention forward for sm_103a: tcgen05 MMAs into tensor memory, TMA-fed
// K/V ring, per-row online softmax with the stabilised shift.
//
// Method (ijyty.com/news/896914, §2.1): for each key block j of a query tile,
//   S = Q K_j^T (raw, FP32),  m = shift(running stats),  P~ = exp(scale (S - m)),
//   l = exp(scale (m_prev - m)) l + rowsum(P~),
//   O = exp(scale (m_prev - m)) O + P~ V_j,   finally O = O / l,
//   lse = scale m + ln l.
// Stabilised shift (same page, §4.1/§4.2; web578.cn "mechanism 2"): each row
// keeps its running raw maximum rm and how often it occurred, rs; the shift is
//   m = beta rm if rm > 0 and rs > 1;  m = 0 if rm < 0 and rs > 1;  else m = rm,
// evaluated with selects (no divergent branch) after every block.
// Precision (jsqmd.com "Flash Attention低精度训练稳定性优化实践" §3.2): QK^T and
// P~V accumulate in FP32 (TMEM), the softmax runs in FP32, P~ is rounded to BF16
// (round-to-nearest-even) for the P~V product; l is summed with Kahan compensation
// across key blocks (ijyty.com §7.2).
// FP8 variant (ijyty.com §6.1, FP8 with dynamic scaling): E4M3 Q, K, V with per-tensor
// scales folded into the exponent's factor, kind::f8f6f4 MMAs, P~ * 2^8 rounded to E4M3.
//
// CTA organisation (one CTA = two 128-row query tiles of one (b, h)), 512 threads:
//   warps 0-3   softmax warpgroup for tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7   softmax warpgroup for tile 1
//   warps 8-11  correction warpgroup: O <- alpha O between P~V products, then O / l
//   warp  12    MMA issuer (one elected thread)
//   warp  13    TMA producer (one elected thread)
// Registers are rebalanced after the launch (setmaxnreg): softmax threads hold a whole
// 128-column row of S, the others need few.
// Tensor memory (512 columns): S0 | S1 | O0 | O1; the BF16 P~ of a tile is written
// over the first 64 columns of its S (32 for E4M3; each thread has read its own S row
// first) and fed to the P~V MMA straight from TMEM.  At d = 128 P~ goes to TMEM in two
// halves, and the MMA warp starts the first half's P~V while the second is computed.
// The row's block maximum comes with the TMEM load of S (tcgen05.ld.red.max) whenever
// the block has no masked column.
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "fa_host.h"
#include "sm103.cuh"

namespace fa {
namespace fwd {

constexpr int kBlockM = 128;   // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;   // keys per block
constexpr int kPScaleLog2 = 8;  // FP8 path: P~ is scaled by 2^8 before its E4M3 rounding

// CTA shape for kT query tiles of 128 rows.
//   kT = 2: warps 0-7 softmax (one warpgroup per tile), 8-11 correction, 12 MMA, 13 TMA,
//           14-15 set-up and teardown only; 512 threads, all 512 TMEM columns, one CTA per SM.
//   kT = 1: warps 0-3 softmax, 4-7 correction, 8 MMA, 9 TMA, 10-11 set-up and teardown only;
//           384 threads, 256 TMEM columns and under 100 KB of shared memory at d = 64, so two
//           CTAs share an SM and one's pipeline fill and drain overlap the other's work (short
//           rows, small grids).
// setmaxnreg acts on whole warpgroups, hence the idle warps that complete the last one.
// Registers are rebalanced after the launch (setmaxnreg): softmax threads hold a whole
// 128-column row of S, the others need few; the split must not exceed the launch allocation.
template <int kT>
struct Shape {
  static constexpr int kTiles = kT;
  static constexpr int kSoftmaxWarps = 4 * kT;
  static constexpr int kMmaWarp = 4 * kT + 4;
  static constexpr int kLoadWarp = 4 * kT + 5;
  static constexpr int kThreads = (kT == 2) ? 512 : 384;
  static constexpr int kCtasPerSm = (kT == 2) ? 1 : 2;
  static constexpr uint32_t kTmemCols = (kT == 2) ? 512 : 256;
  static constexpr int kRegLaunch = (kT == 2) ? 128 : 80;
  static constexpr int kRegSoftmax = (kT == 2) ? 176 : 168, kRegCorr = (kT == 2) ? 96 : 40,
                       kRegOther = (kT == 2) ? 56 : 32;
  static constexpr int kSplit = 128 * kT * kRegSoftmax + 128 * kRegCorr + (kThreads - 128 * kT - 128) * kRegOther;
  static_assert(kSplit <= kThreads * kRegLaunch, "register split exceeds the launch allocation");
  static_assert(kRegLaunch * kThreads * kCtasPerSm <= 65536, "launch registers exceed the SM's file");
};

// kFp8: Q, K, V (and P~ for the P~V product) are E4M3 instead of BF16.  Every operand row
// is then D bytes, so a 128-byte swizzle atom spans 128 elements instead of 64, and one MMA
// instruction consumes 32 elements of K instead of 16 -- always 32 bytes per k-step.
template <int D, bool kFp8 = false, int kT = 2>
struct Cfg {
  static constexpr int kTiles = kT;
  static constexpr int kElem = kFp8 ? 1 : 2;                // bytes per Q/K/V element
  // K/V ring depth: what fits beside the Q tiles (two CTAs per SM for kT = 1)
  static constexpr int kStages = kFp8 ? 4 : ((kT == 1 || D == 128) ? 2 : 4);
  static constexpr int kTileBytes = kBlockM * D * kElem;    // one 128 x D tile (Q, K or V)
  // Swizzle atom: 128-byte rows, or 64-byte rows when a tile row is only 64 bytes (E4M3, d = 64)
  static constexpr int kAtomBytes = (D * kElem >= 128) ? 128 : 64;
  static constexpr int kAtoms = D * kElem / kAtomBytes;     // atom column blocks of a tile
  static constexpr int kAtomElems = kAtomBytes / kElem;     // elements per atom row
  static constexpr int kAtomBlock = kBlockM * kAtomBytes;   // bytes of one atom column block (128 rows)
  static constexpr int kStepsPerAtom = kAtomBytes / 32;     // 32-byte k-steps per atom row
  static constexpr int kKStepsS = D * kElem / 32;           // Q K^T k-steps (32 bytes each)
  static constexpr int kKStepsO = kBlockN * kElem / 32;     // P~ V k-steps over the keys
  static constexpr int kPCols = kBlockN * kElem / 4;        // TMEM columns of a packed P~ row
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTiles * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kVOff + kStages * kTileBytes + 1024;  // +1024 for alignment
  // d = 64 with two tiles leaves 128 TMEM columns beside S0 | S1 | O0 | O1: a third S
  // buffer.  The S of (tile t, block j) then goes to buffer (2j + t) mod 3, so a tile's next S
  // can be computed while its softmax still works on the current one.  One tile: S0 | O0.
  static constexpr bool kRing = (D == 64 && kT == 2);
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128;
  static constexpr uint32_t kTmemO0 = kRing ? 384 : 128 * kT, kTmemO1 = kTmemO0 + D;
  __device__ static uint32_t s_col(int t, int j) {
    return kRing ? (uint32_t)(((2 * j + t) % 3) * 128) : (t == 0 ? kTmemS0 : kTmemS1);
  }
  // Q K^T with both operands K-major; P~ (TMEM) x V with V MN-major
  static constexpr uint32_t kIdescS = kFp8 ? idesc_e4m3(128, kBlockN, false, false) : idesc_bf16(128, kBlockN, false, false);
  static constexpr uint32_t kIdescO = kFp8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
  static_assert(kAtoms >= 1 && kAtoms * kAtomBytes == D * kElem, "tile rows must be whole swizzle atoms");
  static_assert((kRing ? 3 : kT) * 128 <= kTmemO0 && kTmemO0 + kT * D <= Shape<kT>::kTmemCols,
                "TMEM plan exceeds the allocation");
  static_assert(kT == 2 || 2 * (kSmemBytes + 4096) <= 228 * 1024, "two CTAs must fit one SM's shared memory");
  // shared-memory descriptor of an operand in this tile layout (8-row groups kAtomBytes * 8 apart)
  __device__ static uint64_t sdesc(uint32_t saddr, uint32_t lbo) {
    return kAtomBytes == 128 ? sdesc_sw128(saddr, lbo, 8 * kAtomBytes) : sdesc_sw64(saddr, lbo, 8 * kAtomBytes);
  }
};

// Barrier slot and wait parity of hand-off event e (see Shared): two alternating barriers
// with the d = 64 ring, one barrier otherwise.
template <bool kTwo>
__device__ __forceinline__ int ev_slot(int e) { return kTwo ? (e & 1) : 0; }
template <bool kTwo>
__device__ __forceinline__ uint32_t ev_parity(int e) { return kTwo ? (uint32_t)((e >> 1) & 1) : (uint32_t)(e & 1); }

struct Params {
  __nv_bfloat16* o;
  float* lse;
  float* stat_rm;
  int32_t* stat_rs;
  int8_t* stat_branch;
  int32_t* stat_ones;
  float* stat_min;
  DevStatus* status;
  int N;
  int BH;
  int n_qblocks;   // ceil(N / (128 kT))
  int causal;
  float scale;
  float scale_log2;  // scale * log2(e)
  const float* descale;  // FP8 inputs: device [3] = per-tensor scales of Q, K, V
  float beta;
  int inject_stall;  // test builds only (FA_TEST_HOOKS): make the MMA warp's first wait run out
};

template <int kTiles>
struct Shared {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  // Hand-offs that can run two events ahead of their waiter (with the d = 64 ring a tile's
  // softmax may finish two blocks before the MMA warp takes the first) use two barriers
  // per tile: event e lands on [e & 1] and is awaited with parity (e >> 1) & 1, so neither
  // barrier runs more than one phase ahead.  Without the ring only [0] is used, with
  // parity e & 1.  Events: S and P~ of block j (e = j); alpha and the corrected O of
  // block j >= 1 (e = j - 1).  Without the ring p_ready[t][1] carries the first half of
  // P~ (keys 0-63 of the block), handed over before the second half is computed.
  uint64_t s_full[kTiles][2], p_ready[kTiles][2], pv_done[kTiles];
  // o_done[t]: the last P~V of tile t has completed (committed once, after it).  The epilogue
  // waits on it rather than on pv_done's parity, which could alias if it ran two products
  // behind.
  uint64_t o_done[kTiles];
  uint64_t alpha_ready[kTiles][2], o_ready[kTiles][2], l_ready[kTiles];
  uint64_t mma_done;
  uint64_t never;  // test builds only: a barrier nothing arrives on
  // correction factor of each row, by alpha event parity: a softmax can hand over the next
  // block's factor before the correction warpgroup has read the current one only with the
  // d = 64 ring, and never two ahead (the P~V that gates its next S waits for that read)
  float alpha[kTiles][2][kBlockM];
  float lfin[kTiles][kBlockM];   // final row sums for the epilogue
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// Which key blocks tile t of query block qb (kTiles tiles of 128 rows) attends: [0, nb).
// 0 if the tile is entirely past N.
template <int kTiles>
__device__ __forceinline__ int tile_blocks(const Params& p, int qb, int t) {
  const int row0 = qb * (kTiles * kBlockM) + t * kBlockM;
  if (row0 >= p.N) return 0;
  const int nk = (p.N + kBlockN - 1) / kBlockN;
  if (!p.causal) return nk;
  const int last = (row0 + kBlockM - 1) / kBlockN;  // diagonal block of the tile
  return min(nk, last + 1);
}

// kStable: 0 = plain shift (running max); 1 = stabilised shift on the running (max, count)
// of the row; 2 = block-local reading: each key block's own (max, count) picks a shift by
// the same rule and the row keeps the largest shift seen so far.
template <int D, int kStable, bool kStats, bool kFp8, int kT>
__global__ void __launch_bounds__(Shape<kT>::kThreads, Shape<kT>::kCtasPerSm)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<D, kFp8, kT>;
  using L = Shape<kT>;
  constexpr int kTiles = kT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Shared<kT> sh;
  volatile uint32_t* abort_flag = &sh.abort_flag;

  const int warp = threadIdx.x / 32;
  // heaviest (largest causal) query blocks first
  const int qb = p.causal ? (p.n_qblocks - 1 - (int)(blockIdx.x / p.BH)) : (int)(blockIdx.x / p.BH);
  const int bh = blockIdx.x % p.BH;
  const int nb0 = tile_blocks<kT>(p, qb, 0), nb1 = (kT > 1) ? tile_blocks<kT>(p, qb, 1) : 0;
  const int nbmax = max(nb0, nb1);

  if (threadIdx.x == 0) {
    sh.abort_flag = 0;
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&sh.s_full[t][0], 1);
      mbar_init(&sh.s_full[t][1], 1);
      mbar_init(&sh.p_ready[t][0], kBlockM);
      mbar_init(&sh.p_ready[t][1], kBlockM);
      mbar_init(&sh.pv_done[t], 1);
      mbar_init(&sh.o_done[t], 1);
      mbar_init(&sh.alpha_ready[t][0], kBlockM);
      mbar_init(&sh.alpha_ready[t][1], kBlockM);
      mbar_init(&sh.o_ready[t][0], kBlockM);
      mbar_init(&sh.o_ready[t][1], kBlockM);
      mbar_init(&sh.l_ready[t], kBlockM);
    }
    mbar_init(&sh.mma_done, 1);
    mbar_init(&sh.never, 1);
    fence_barrier_init();
    FA_BOUNDS_OK((uint32_t)(smem - smem_raw) + C::kVOff + C::kStages * C::kTileBytes <= dynamic_smem_bytes(),
                 p.status, kSiteFwdSmemSize, dynamic_smem_bytes());
  }
  if (warp == L::kMmaWarp) {
    tmem_alloc(&sh.tmem_base, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  // Roles by warpgroup; each branch first rebalances its registers (setmaxnreg) so the
  // softmax warpgroups can hold a 128-column row of S each.
  if (warp >= L::kMmaWarp) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kRegOther));
  if (warp == L::kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int ntiles = (kT > 1 && nb1 > 0) ? 2 : 1;
      mbar_arrive_expect_tx(&sh.q_full, ntiles * C::kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        if (FA_BOUNDS_OK(qb * (kTiles * kBlockM) + t * kBlockM < p.N, p.status, kSiteFwdQRow,
                         qb * (kTiles * kBlockM) + t * kBlockM))
          for (int c = 0; c < C::kAtoms; ++c)
            tma_load_3d(smem + C::kQOff + t * C::kTileBytes + c * C::kAtomBlock, &tmQ, &sh.q_full,
                        c * C::kAtomElems, qb * (kTiles * kBlockM) + t * kBlockM, bh);
      int nk_issued = 0, nv_issued = 0;
      for (int j = 0; j < nbmax; ++j) {
        const int s = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        if (!mbar_wait(&sh.k_empty[s], ph ^ 1, abort_flag, p.status)) break;
        if (!FA_BOUNDS_OK(j * kBlockN < p.N, p.status, kSiteFwdKVRow, j * kBlockN)) break;
        mbar_arrive_expect_tx(&sh.k_full[s], C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(smem + C::kKOff + s * C::kTileBytes + c * C::kAtomBlock, &tmK, &sh.k_full[s], c * C::kAtomElems,
                      j * kBlockN, bh);
        nk_issued = j + 1;
        if (!mbar_wait(&sh.v_empty[s], ph ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&sh.v_full[s], C::kTileBytes);
        for (int c = 0; c < C::kAtoms; ++c)
          tma_load_3d(smem + C::kVOff + s * C::kTileBytes + c * C::kAtomBlock, &tmV, &sh.v_full[s], c * C::kAtomElems,
                      j * kBlockN, bh);
        nv_issued = j + 1;
      }
      if (*abort_flag) {
        // let copies still in flight land before the CTA's shared memory goes away
        volatile uint32_t ignore_abort = 0;
        mbar_wait(&sh.q_full, 0, &ignore_abort, p.status);
        for (int j = max(0, nk_issued - C::kStages); j < nk_issued; ++j)
          mbar_wait(&sh.k_full[j % C::kStages], (j / C::kStages) & 1, &ignore_abort, p.status);
        for (int j = max(0, nv_issued - C::kStages); j < nv_issued; ++j)
          mbar_wait(&sh.v_full[j % C::kStages], (j / C::kStages) & 1, &ignore_abort, p.status);
      }
    }
  } else if (warp == L::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t sQ = smem_u32(smem + C::kQOff);
      const uint32_t sK = smem_u32(smem + C::kKOff);
      const uint32_t sV = smem_u32(smem + C::kVOff);
      const int nb[2] = {nb0, nb1};
      bool ok = mbar_wait(&sh.q_full, 0, abort_flag, p.status);
#ifdef FA_TEST_HOOKS
      // failure-detection test: wait on a barrier nothing arrives on; the bounded wait runs
      // out, raises the CTA's abort flag and records a timeout, and every warp unwinds
      if (p.inject_stall) ok = ok && mbar_wait(&sh.never, 0, abort_flag, p.status);
#endif
      tc_fence_after();
      // S_t = Q_t K_j^T over 32-byte k-steps (K-major swizzled operands, one atom column
      // block of 128 rows per kAtomBytes of each row)
      auto issue_s = [&](int t, int s, int j) {
        const uint32_t a0 = sQ + t * C::kTileBytes, b0 = sK + s * C::kTileBytes;
        const uint32_t d = tmem + C::s_col(t, j);
#pragma unroll
        for (int kk = 0; kk < C::kKStepsS; ++kk) {
          const uint32_t off = (kk / C::kStepsPerAtom) * C::kAtomBlock + (kk % C::kStepsPerAtom) * 32;
          if constexpr (kFp8)
            mma_ss_f8(d, C::sdesc(a0 + off, 16), C::sdesc(b0 + off, 16), C::kIdescS, kk > 0);
          else
            mma_ss(d, C::sdesc(a0 + off, 16), C::sdesc(b0 + off, 16), C::kIdescS, kk > 0);
        }
        tc_commit(&sh.s_full[t][ev_slot<C::kRing>(j)]);
      };
      // O_t += P~_t V_j: P~ from TMEM (K = 128 keys, 8 columns = 32 bytes per k-step), V MN-major
      // (a k-step covers 32 / kElem keys of 128-byte rows)
      auto issue_pv = [&](int t, int s, int j, int k_lo = 0, int k_hi = C::kKStepsO) {
        const uint32_t b0 = sV + s * C::kTileBytes;
        const uint32_t d = tmem + (t == 0 ? C::kTmemO0 : C::kTmemO1);
        const uint32_t a = tmem + C::s_col(t, j);
#pragma unroll
        for (int kk = k_lo; kk < k_hi; ++kk) {
          // a k-step covers 32 / kElem keys, one atom row (kAtomBytes) each; LBO = the next
          // atom column block along d (only with two or more)
          FA_BOUNDS_OK((kk + 1) * (32 / C::kElem) * C::kAtomBytes <= C::kAtomBlock && s < C::kStages, p.status,
                       kSiteFwdVDesc, kk);
          const uint64_t bd = C::sdesc(b0 + kk * (32 / C::kElem) * C::kAtomBytes, C::kAtomBlock);
          if constexpr (kFp8)
            mma_ts_f8(d, a + kk * 8, bd, C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
          else
            mma_ts(d, a + kk * 8, bd, C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (k_hi == C::kKStepsO) {
          tc_commit(&sh.pv_done[t]);
          if (j == nb[t] - 1) tc_commit(&sh.o_done[t]);
        }
      };
      if constexpr (C::kRing) {
        // Order: S0_0 S1_0 S0_1 | PV0_0 S1_1 PV1_0 S0_2 | PV0_1 S1_2 PV1_1 S0_3 | ...
        // S(t, j) writes buffer (2j + t) mod 3, whose previous user's P~V is always issued
        // before it (same-thread MMAs run in order), and each P~V follows its softmax.
        int k_ready = -1;  // K blocks up to this one have landed
        auto need_k = [&](int b) {
          if (b <= k_ready) return true;
          if (!(ok = mbar_wait(&sh.k_full[b % C::kStages], (b / C::kStages) & 1, abort_flag, p.status))) return false;
          tc_fence_after();
          k_ready = b;
          return true;
        };
        auto pv_when_ready = [&](int t, int b) {  // P~V of (tile t, block b) once P~ and O are ready
          if (!(ok = mbar_wait(&sh.p_ready[t][ev_slot<true>(b)], ev_parity<true>(b), abort_flag, p.status))) return;
          if (b > 0 &&
              !(ok = mbar_wait(&sh.o_ready[t][ev_slot<true>(b - 1)], ev_parity<true>(b - 1), abort_flag, p.status)))
            return;
          tc_fence_after();
          issue_pv(t, b % C::kStages, b);
        };
        if (nbmax > 0 && need_k(0)) {
          for (int t = 0; t < kTiles; ++t)
            if (nb[t] > 0) issue_s(t, 0, 0);
          tc_commit(&sh.k_empty[0]);
          if (nb[0] > 1 && need_k(1)) issue_s(0, 1, 1);
        }
        for (int j = 1; ok && j <= nbmax; ++j) {
          const int sp = (j - 1) % C::kStages;  // stage of block j-1
          if (!(ok = mbar_wait(&sh.v_full[sp], ((j - 1) / C::kStages) & 1, abort_flag, p.status))) break;
          tc_fence_after();
          if (j - 1 < nb[0]) {
            pv_when_ready(0, j - 1);
            if (!ok) break;
          }
          if (j < nb[1]) {
            if (!need_k(j)) break;
            issue_s(1, j % C::kStages, j);
          }
          if (j < nbmax) tc_commit(&sh.k_empty[j % C::kStages]);  // S(0, j) and S(1, j) issued
          if (j - 1 < nb[1]) {
            pv_when_ready(1, j - 1);
            if (!ok) break;
          }
          tc_commit(&sh.v_empty[sp]);
          if (j + 1 < nb[0]) {
            if (!need_k(j + 1)) break;
            issue_s(0, (j + 1) % C::kStages, j + 1);
          }
        }
      } else {
        // Order: S0_0 S1_0 | PV0_0 S0_1 PV1_0 S1_1 | PV0_1 S0_2 PV1_1 S1_2 | ... | PV0_last PV1_last
        // Each P~V runs in two halves over the keys, the first as soon as the softmax has
        // stored the first half of P~ (2-3 % faster than waiting for all of it; four or
        // eight parts measured slower: the single issuer then waits on one tile too often).
        for (int j = 0; ok && j <= nbmax; ++j) {
          const int s = j % C::kStages;
          const uint32_t ph = (j / C::kStages) & 1;
          const int sp = (j + C::kStages - 1) % C::kStages;  // stage of block j-1
          if (j < nbmax) {
            if (!(ok = mbar_wait(&sh.k_full[s], ph, abort_flag, p.status))) break;
            tc_fence_after();
          }
          if (j > 0) {
            if (!(ok = mbar_wait(&sh.v_full[sp], ((j - 1) / C::kStages) & 1, abort_flag, p.status))) break;
            tc_fence_after();
          }
          for (int t = 0; t < kTiles; ++t) {
            if (j > 0 && j - 1 < nb[t]) {
              // the first half of P~ (keys 0-63) is handed over before the second is computed
              if (!(ok = mbar_wait(&sh.p_ready[t][1], ev_parity<false>(j - 1), abort_flag, p.status))) break;
              // O_t must carry block j-1's correction (applied by the correction warpgroup)
              if (j - 1 > 0 && !(ok = mbar_wait(&sh.o_ready[t][0], ev_parity<false>(j - 2), abort_flag, p.status)))
                break;
              tc_fence_after();
              issue_pv(t, sp, j - 1, 0, C::kKStepsO / 2);
              if (!(ok = mbar_wait(&sh.p_ready[t][0], ev_parity<false>(j - 1), abort_flag, p.status))) break;
              tc_fence_after();
              issue_pv(t, sp, j - 1, C::kKStepsO / 2, C::kKStepsO);
            }
            if (j < nb[t]) issue_s(t, s, j);
          }
          if (!ok) break;
          if (j < nbmax) tc_commit(&sh.k_empty[s]);
          if (j > 0) tc_commit(&sh.v_empty[sp]);
        }
      }
      // every MMA issued above has completed before TMEM is released
      tc_commit(&sh.mma_done);
      {
        // MMAs still in flight must finish before TMEM is released, even after an abort
        volatile uint32_t ignore_abort = 0;
        mbar_wait(&sh.mma_done, 0, &ignore_abort, p.status);
      }
    }
  }
  } else if (warp < L::kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kRegSoftmax));
    const int t = warp / 4;                      // tile
    const int lane_base = (warp % 4) * 32;       // TMEM lane quarter of this warp
    const int r = lane_base + (threadIdx.x % 32);  // row within the tile
    const int nb = (t == 0) ? nb0 : nb1;
    const int row = qb * (kTiles * kBlockM) + t * kBlockM + r;
    const uint32_t lane_off = (uint32_t)lane_base << 16;
    const uint32_t tS_fixed = tmem + C::s_col(t, 0) + lane_off;  // without the ring: S0 or S1
    // FP8: raw scores are in units of dq * dk (the Q and K scales); fold both into the
    // exponent's scale.  rm, m and the tie count stay in accumulator units, which is the same
    // rule on the dequantised scores (a positive factor keeps order, equality and sign).
    float dqk = 1.f;
    if constexpr (kFp8) dqk = __ldg(p.descale) * __ldg(p.descale + 1);
    const float c = p.scale_log2 * dqk;
    float rm = -INFINITY, m = -INFINITY, l = 0.f;
    float lc = 0.f;         // compensation of l: the row sum is l - lc (Kahan)
    float rmin = INFINITY;  // smallest visible raw score (statistics only)
    int rs = 0, ones = 0;
    int branch = 0;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!(ok = mbar_wait(&sh.s_full[t][ev_slot<C::kRing>(j)], ev_parity<C::kRing>(j), abort_flag, p.status))) break;
      tc_fence_after();
      const uint32_t tS = C::kRing ? tmem + C::s_col(t, j) + lane_off : tS_fixed;  // this block's S, then P~
      FA_BOUNDS_OK(C::s_col(t, j) + kBlockN <= C::kTmemO0, p.status, kSiteFwdTmemS, C::s_col(t, j));
      // the whole 128-column row in one round trip: four loads, one wait; each load also
      // returns the largest of its 32 raw scores
      uint32_t raw[kBlockN];
      float pmax[kBlockN / 32];
#pragma unroll
      for (int c0 = 0; c0 < kBlockN; c0 += 32)
        tmem_ld32_max(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(raw + c0), pmax[c0 / 32]);
      tmem_ld_wait();
      reg_fence(raw);
      reg_fence(pmax);
      float sv[kBlockN];
#pragma unroll
      for (int i = 0; i < kBlockN; ++i) sv[i] = __uint_as_float(raw[i]);
      // mask: keys past N, and keys after the query on the causal diagonal
      const int col0 = j * kBlockN;
      const int lim = p.causal ? min(p.N - col0, row - col0 + 1) : (p.N - col0);
      if (lim < kBlockN) {
#pragma unroll
        for (int i = 0; i < kBlockN; ++i) sv[i] = (i < lim) ? sv[i] : -INFINITY;
      }
      // block max and each 32-column chunk's maximum: from the loads' reductions when no row
      // of the warp has a masked column, else over the masked values (3-input max, one
      // independent chain per chunk)
      float pm[kBlockN / 32];
      const bool unmasked = __all_sync(0xffffffffu, lim >= kBlockN);
      if (unmasked) {
#pragma unroll
        for (int c0 = 0; c0 < kBlockN / 32; ++c0) pm[c0] = pmax[c0];
      } else {
#pragma unroll
        for (int c0 = 0; c0 < kBlockN / 32; ++c0) {
          float mx = max3f(sv[32 * c0], sv[32 * c0 + 1], sv[32 * c0 + 2]);
#pragma unroll
          for (int i = 32 * c0 + 3; i < 32 * c0 + 31; i += 2) mx = max3f(mx, sv[i], sv[i + 1]);
          pm[c0] = fmaxf(mx, sv[32 * c0 + 31]);
        }
      }
      const float bm = fmaxf(max3f(pm[0], pm[1], pm[2]), pm[3]);
      if constexpr (kStats) {
        // masked entries hold -inf; they never count as the row's minimum
        float mn0 = INFINITY, mn1 = INFINITY;
#pragma unroll
        for (int i = 0; i < kBlockN; i += 4) {
          mn0 = min3f(mn0, sv[i] == -INFINITY ? INFINITY : sv[i], sv[i + 1] == -INFINITY ? INFINITY : sv[i + 1]);
          mn1 = min3f(mn1, sv[i + 2] == -INFINITY ? INFINITY : sv[i + 2], sv[i + 3] == -INFINITY ? INFINITY : sv[i + 3]);
        }
        rmin = fminf(rmin, fminf(mn0, mn1));
      }
      float m_new;
      int bc = 0;
      if constexpr (kStable != 0 || kStats) {
        // running (max, count) merge: rs' = [rm == rm'] rs + [bm == rm'] bc.  The block's
        // count only matters when bm reaches the running max (or, block-locally, always).
        // Only a chunk whose maximum equals the block maximum can hold it, so the warp counts
        // just the chunks one of the rows that need the count needs (exact -- a skipped chunk
        // has no entry equal to bm in any row that uses bc); a warp whose rows all have
        // bm < rm counts nothing.  Each equality gives 1.0, summed in FP32 pairs (exact).
        const bool need = (kStable == 2) || (bm >= rm);
        float c0s = 0.f, c1s = 0.f, c2s = 0.f, c3s = 0.f;  // two independent pair sums
#pragma unroll
        for (int c0 = 0; c0 < kBlockN / 32; ++c0) {
          if (__any_sync(0xffffffffu, need && pm[c0] == bm)) {
#pragma unroll
            for (int i = c0 * 32; i < c0 * 32 + 32; i += 4) {
              add2(c0s, c1s, c0s, c1s, eq_one(sv[i], bm), eq_one(sv[i + 1], bm));
              add2(c2s, c3s, c2s, c3s, eq_one(sv[i + 2], bm), eq_one(sv[i + 3], bm));
            }
          }
        }
        bc = (bm == -INFINITY) ? 0 : (int)((c0s + c1s) + (c2s + c3s));
        const float rm_new = fmaxf(rm, bm);
        rs = ((rm == rm_new) ? rs : 0) + ((bm == rm_new) ? bc : 0);
        rm = rm_new;
      } else {
        rm = fmaxf(rm, bm);
      }
      if constexpr (kStable == 1) {
        const bool rep = rs > 1;
        const bool pos = rep && (rm > 0.f), neg = rep && (rm < 0.f);
        m_new = pos ? p.beta * rm : (neg ? 0.f : rm);
        branch = pos ? 1 : (neg ? 2 : 0);
      } else if constexpr (kStable == 2) {
        const bool rep = bc > 1;
        const bool pos = rep && (bm > 0.f), neg = rep && (bm < 0.f);
        const float mb = pos ? p.beta * bm : (neg ? 0.f : bm);
        const int brb = pos ? 1 : (neg ? 2 : 0);
        branch = (mb >= m) ? brb : branch;   // branch of the block that set the shift
        m_new = fmaxf(m, mb);
      } else {
        m_new = rm;
      }
      const float alpha = ex2_approx((m - m_new) * c);  // 0 on the first block (m = -inf)
      if (j > 0) {
        // hand the row's correction factor to the correction warpgroup right away
        sh.alpha[t][(j - 1) & 1][r] = alpha;
        mbar_arrive(&sh.alpha_ready[t][ev_slot<C::kRing>(j - 1)]);
      }
      // FP8: P~ * 2^8 (added to the exponent) uses the E4M3 range below 448 instead of <= 1
      const float nmc = kFp8 ? fmaf(-m_new, c, (float)kPScaleLog2) : -m_new * c;
      float sum0 = 0.f, sum1 = 0.f;
      if constexpr (kFp8) {
        uint32_t pk[kBlockN / 4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = h * 64; i < h * 64 + 64; i += 4) {
            float x0, x1, x2, x3;
            fma2(x0, x1, sv[i], sv[i + 1], c, c, nmc, nmc);       // scale*log2(e)*dq*dk * (S - m) + 8
            fma2(x2, x3, sv[i + 2], sv[i + 3], c, c, nmc, nmc);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            add2(sum0, sum1, sum0, sum1, p0, p1);
            add2(sum0, sum1, sum0, sum1, p2, p3);
            pk[i / 4] = pack_e4m3x4(p0, p1, p2, p3);
          }
          if constexpr (!C::kRing) {
            __syncwarp();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pk[h * 16 + i];
            tmem_st16(tS + h * 16, w);
            if (h == 0) {
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(&sh.p_ready[t][1]);
            }
          }
        }
        if constexpr (kStats) {
          // an entry of exactly 1.0 is 2^8 = E4M3 code 0x78 after the scaling
#pragma unroll
          for (int i = 0; i < kBlockN / 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) ones += (((pk[i] >> (8 * b)) & 0xFFu) == 0x78u) ? 1 : 0;
        }
        if constexpr (C::kRing) {
          __syncwarp();
          tmem_st32(tS, pk);
        }
      } else {
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = h * 64; i < h * 64 + 64; i += 2) {
            float x0, x1;
            fma2(x0, x1, sv[i], sv[i + 1], c, c, nmc, nmc);   // scale*log2(e) * (S - m)
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            add2(sum0, sum1, sum0, sum1, p0, p1);
            pk[i / 2] = pack_bf16x2(p0, p1);
          }
          __syncwarp();
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = pk[h * 32 + i];
          tmem_st32(tS + h * 32, w);
          if constexpr (!C::kRing) {
            if (h == 0) {
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(&sh.p_ready[t][1]);
            }
          }
        }
        if constexpr (kStats) {
#pragma unroll
          for (int i = 0; i < kBlockN / 2; ++i)
            ones += ((pk[i] & 0xFFFFu) == 0x3F80u ? 1 : 0) + ((pk[i] >> 16) == 0x3F80u ? 1 : 0);
        }
      }
      {
        // l <- alpha l + rowsum(P~) with compensated (Kahan) summation across blocks; the
        // rounding error of alpha * l is captured exactly by an FMA and folded in too
        const float bsum = sum0 + sum1;
        const float ls = alpha * l;
        const float e = fmaf(alpha, l, -ls);
        const float y = bsum - (alpha * lc - e);
        const float tsum = ls + y;
        lc = (tsum - ls) - y;
        l = tsum;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sh.p_ready[t][ev_slot<C::kRing>(j)]);
      m = m_new;
    }
    // ------------------------------------------------------------ row results
    if (ok && nb > 0) {
      l -= lc;  // fold the compensation in
      sh.lfin[t][r] = l;
      mbar_arrive(&sh.l_ready[t]);
      // FP8: l sums P~ * 2^8
      const float lse_row = kFp8 ? m * (p.scale * dqk) + (logf(l) - (float)kPScaleLog2 * 0.6931471805599453f)
                                 : m * p.scale + logf(l);
      report_nonfinite((row < p.N && !(fabsf(lse_row) < INFINITY)) ? 1u : 0u, p.status, kOutLse);
      if (row < p.N &&
          FA_BOUNDS_OK((long long)bh * p.N + row < (long long)p.BH * p.N, p.status, kSiteFwdLseRow, row)) {
        const size_t srow = (size_t)bh * p.N + row;
        p.lse[srow] = lse_row;
        if constexpr (kStats) {
          if (p.stat_rm) p.stat_rm[srow] = rm * dqk;
          if (p.stat_rs) p.stat_rs[srow] = rs;
          if (p.stat_branch) p.stat_branch[srow] = (int8_t)branch;
          if (p.stat_ones) p.stat_ones[srow] = ones;
          if (p.stat_min) p.stat_min[srow] = rmin * dqk;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ correction warpgroup
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kRegCorr));
    // O_t <- alpha O_t between P~V products (ijyty.com §2.1, O = diag(exp(m_prev - m)) O_prev + P~V),
    // then the epilogue O = O / l.  Thread = row of the lane quarter, for both tiles.
    const int lane_base = (warp % 4) * 32;
    const int r = lane_base + (threadIdx.x % 32);
    const int nb[2] = {nb0, nb1};
    bool ok = true;
    for (int j = 1; ok && j < nbmax; ++j) {
      for (int t = 0; t < kTiles; ++t) {
        if (j >= nb[t]) continue;
        if (!(ok = mbar_wait(&sh.alpha_ready[t][ev_slot<C::kRing>(j - 1)], ev_parity<C::kRing>(j - 1), abort_flag,
                             p.status)))
          break;
        const float alpha = sh.alpha[t][(j - 1) & 1][r];
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // the previous P~V of this tile has landed (its S_j commit already implies it)
          if (!(ok = mbar_wait(&sh.pv_done[t], (j - 1) & 1, abort_flag, p.status))) break;
          tc_fence_after();
          const uint32_t tO = tmem + (t == 0 ? C::kTmemO0 : C::kTmemO1) + ((uint32_t)lane_base << 16);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t w[32];
            tmem_ld32(tO + c0, w);
            tmem_ld_wait();
            reg_fence(w);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float a0, a1;
              mul2(a0, a1, __uint_as_float(w[i]), __uint_as_float(w[i + 1]), alpha, alpha);
              w[i] = __float_as_uint(a0);
              w[i + 1] = __float_as_uint(a1);
            }
            tmem_st32(tO + c0, w);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&sh.o_ready[t][ev_slot<C::kRing>(j - 1)]);
      }
    }
    // ------------------------------------------------------------ epilogue: O = O / l -> BF16
    for (int t = 0; ok && t < kTiles; ++t) {
      if (nb[t] == 0) continue;
      if (!(ok = mbar_wait(&sh.o_done[t], 0, abort_flag, p.status))) break;
      if (!(ok = mbar_wait(&sh.l_ready[t], 0, abort_flag, p.status))) break;
      tc_fence_after();
      // FP8: O = (P~ 2^8)_E4M3 V8 * dv / (l 2^8); the 2^8 is in both sums
      const float inv_l = (kFp8 ? __ldg(p.descale + 2) : 1.f) / sh.lfin[t][r];
      const int row = qb * (kTiles * kBlockM) + t * kBlockM + r;
      const bool valid = row < p.N;
      const size_t orow = ((size_t)bh * p.N + (valid ? row : 0)) * D;
      const uint32_t tO = tmem + (t == 0 ? C::kTmemO0 : C::kTmemO1) + ((uint32_t)lane_base << 16);
      uint32_t bad = 0;  // NaN/Inf entries of this row of O, as stored
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(tO + c0, w);
        tmem_ld_wait();
        reg_fence(w);
        uint4 pkd[4];
        uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float o0 = __uint_as_float(w[2 * i]) * inv_l, o1 = __uint_as_float(w[2 * i + 1]) * inv_l;
          pw[i] = pack_bf16x2(o0, o1);
          bad += nonfinite_bf16x2(pw[i]);
        }
        if (valid && FA_BOUNDS_OK(orow + c0 + 32 <= (size_t)p.BH * p.N * D, p.status, kSiteFwdORow, row)) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + orow + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = pkd[i];
        }
      }
      report_nonfinite(valid ? bad : 0u, p.status, kOutO);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace fwd
}  // namespace fa

namespace {

template <int D, int kStable, bool kStats, bool kFp8, int kT>
int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const fa::fwd::Params& p0,
               cudaStream_t stream) {
  using C = fa::fwd::Cfg<D, kFp8, kT>;
  using L = fa::fwd::Shape<kT>;
  auto kern = fa::fwd::fa_fwd_kernel<D, kStable, kStats, kFp8, kT>;
  fa::fwd::Params p = p0;
  p.n_qblocks = (p.N + kT * fa::fwd::kBlockM - 1) / (kT * fa::fwd::kBlockM);
  // setmaxnreg.inc waits until the block's launch registers can cover the new split: refuse
  // to launch a build whose launch allocation is smaller than the split needs
  static std::atomic<uint64_t> prepared{0};
  int rc = fa::prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, L::kThreads, L::kSplit,
                              "forward kernel", &prepared);
  if (rc) return rc;
  const dim3 grid((unsigned)(p.n_qblocks * p.BH));
  kern<<<grid, L::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return fa::check_cuda(cudaGetLastError(), "launch fa_fwd_kernel");
}

template <int D, bool kFp8, int kT>
int dispatch_fwd_tiles(int stable, bool stats, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const fa::fwd::Params& p, cudaStream_t s) {
  if (stable == 2)
    return stats ? launch_fwd<D, 2, true, kFp8, kT>(tq, tk, tv, p, s) : launch_fwd<D, 2, false, kFp8, kT>(tq, tk, tv, p, s);
  if (stable == 1)
    return stats ? launch_fwd<D, 1, true, kFp8, kT>(tq, tk, tv, p, s) : launch_fwd<D, 1, false, kFp8, kT>(tq, tk, tv, p, s);
  return stats ? launch_fwd<D, 0, true, kFp8, kT>(tq, tk, tv, p, s) : launch_fwd<D, 0, false, kFp8, kT>(tq, tk, tv, p, s);
}

// At d = 64 and up to kShortRows keys, one query tile per CTA with two CTAs per SM: rows of
// at most 16 key blocks spend much of a CTA's life filling and draining its pipeline, and a
// second CTA on the SM covers that (GPT-2-shaped problems, 1024 tokens: +5-13 %).  Longer rows
// keep two tiles per CTA, whose third S buffer in TMEM is worth more there (16k tokens: the
// single-tile CTA is 5-12 % slower).  d = 128 always takes two tiles (two CTAs' shared memory
// would not fit an SM).
constexpr int kShortRows = 2048;

template <int D, bool kFp8>
int dispatch_fwd(int stable, bool stats, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const fa::fwd::Params& p, cudaStream_t s) {
  if constexpr (D == 64) {
    if (p.N <= kShortRows) return dispatch_fwd_tiles<D, kFp8, 1>(stable, stats, tq, tk, tv, p, s);
  }
  return dispatch_fwd_tiles<D, kFp8, 2>(stable, stats, tq, tk, tv, p, s);
}

// Argument checks and kernel parameters shared by the BF16 and FP8 entry points.
int prepare_fwd(fa::fwd::Params& p, bool& want_stats, const void* q, const void* k, const void* v, void* o,
                float* lse, int B, int H, int N, int d, int causal, float scale, int stable, float beta,
                const fa_row_stats* stats) {
  using namespace fa;
  int rc;
  if ((rc = check_shape(B, H, N, d))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) || (rc = check_ptr(o, "o")))
    return rc;
  if (!lse) return set_error(FA_ERR_INVALID_ARG, "lse is NULL");
  if (!(scale > 0.f) || !isfinite(scale)) return set_error(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (stable < 0 || stable > 2) return set_error(FA_ERR_INVALID_ARG, "stable must be 0, 1 or 2 (got %d)", stable);
  if (stable && (!isfinite(beta) || beta < 1.f)) return set_error(FA_ERR_INVALID_ARG, "beta must be finite and >= 1");
  p = fwd::Params{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  want_stats = false;
  if (stats) {
    p.stat_rm = stats->row_max_raw;
    p.stat_rs = stats->row_ties;
    p.stat_branch = stats->row_branch;
    p.stat_ones = stats->row_ones;
    p.stat_min = stats->row_min_raw;
    want_stats = p.stat_rm || p.stat_rs || p.stat_branch || p.stat_ones || p.stat_min;
  }
  p.status = device_status_word();
  if (!p.status) return set_error(FA_ERR_CUDA, "could not allocate the device status record");
  p.N = N;
  p.BH = B * H;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.beta = beta;
#ifdef FA_TEST_HOOKS
  const char* inject = getenv("FA_TEST_INJECT_STALL");
  p.inject_stall = (inject && inject[0] == '1') ? 1 : 0;
#endif
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                      int causal, float scale, int stable, float beta, const fa_row_stats* stats, void* stream) {
  fa::NvtxRange nvtx_range("fa_fwd");
  using namespace fa;
  clear_error();
  fwd::Params p;
  bool want_stats;
  int rc = prepare_fwd(p, want_stats, q, k, v, o, lse, B, H, N, d, causal, scale, stable, beta, stats);
  if (rc) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_tmap_bhnd(&tq, q, B * H, N, d, fwd::kBlockM)) || (rc = make_tmap_bhnd(&tk, k, B * H, N, d, fwd::kBlockN)) ||
      (rc = make_tmap_bhnd(&tv, v, B * H, N, d, fwd::kBlockN)))
    return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? dispatch_fwd<64, false>(stable, want_stats, tq, tk, tv, p, s)
                 : dispatch_fwd<128, false>(stable, want_stats, tq, tk, tv, p, s);
}

extern "C" int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* descale, void* o, float* lse,
                          int B, int H, int N, int d, int causal, float scale, int stable, float beta,
                          const fa_row_stats* stats, void* stream) {
  fa::NvtxRange nvtx_range("fa_fwd_fp8");
  using namespace fa;
  clear_error();
  if (d != 64 && d != 128) return set_error(FA_ERR_UNSUPPORTED, "head dim d=%d not supported (64 or 128)", d);
  if (!descale) return set_error(FA_ERR_INVALID_ARG, "descale is NULL");
  if (reinterpret_cast<uintptr_t>(descale) & 3) return set_error(FA_ERR_INVALID_ARG, "descale is not 4-byte aligned");
  fwd::Params p;
  bool want_stats;
  int rc = prepare_fwd(p, want_stats, q8, k8, v8, o, lse, B, H, N, d, causal, scale, stable, beta, stats);
  if (rc) return rc;
  p.descale = descale;
  CUtensorMap tq, tk, tv;
  if ((rc = make_tmap_u8_bhnd(&tq, q8, B * H, N, d, fwd::kBlockM)) ||
      (rc = make_tmap_u8_bhnd(&tk, k8, B * H, N, d, fwd::kBlockN)) ||
      (rc = make_tmap_u8_bhnd(&tv, v8, B * H, N, d, fwd::kBlockN)))
    return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? dispatch_fwd<64, true>(stable, want_stats, tq, tk, tv, p, s)
                 : dispatch_fwd<128, true>(stable, want_stats, tq, tk, tv, p, s);
}
