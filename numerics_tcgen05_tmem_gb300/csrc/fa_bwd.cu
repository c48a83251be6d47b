// Attention backward for sm_103a by recomputation.
//
// The backward re-derives the attention probabilities from Q, K and the saved
// log-sum-exp instead of storing them ("FlashAttention 训练时为什么会梯度爆炸？",
// §2), and uses delta = rowsum(dO o O) (ijyty.com/news/896914, §3.1).  The
// gradient formulas, which the pages do not print, are the calculus of
// O = softmax(scale Q K^T) V:
//   P = exp(scale S - lse),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - delta),   dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels on the caller's stream:
//   fa_bwd_preprocess: delta_i = sum_c dO_ic O_ic (FP32), lse_i log2(e), both padded per
//                      head to a multiple of 128 rows, and dQ_acc = 0
//   fa_bwd_main:       work items are (b, h, 128-key tile); a CTA takes one or more items
//                      and loops over each item's query tiles
//   fa_bwd_dq_convert: dq = bf16(scale * dQ_acc)
//
// fa_bwd_main CTA organisation (512 threads, registers rebalanced per warpgroup):
//   warps 0-7  two "softmax" warpgroups; thread = key row (TMEM lane) of the tile,
//              warpgroup h takes query columns [64h, 64h+64):
//              P^T = exp2(S^T c - lse_q log2 e) into TMEM (BF16) for the dV MMA,
//              dS^T = P^T o (dP^T - delta_q) as BF16 into its dP^T columns of TMEM (the A
//              operand of the dK MMA) and into shared memory (128B swizzle; the MN-major
//              A operand of the dQ MMA); finally warpgroup 0 writes dK, 1 writes dV.
//   warps 8-11 dQ warpgroup: thread = query row; loads each dQ tile from TMEM in one
//              round trip, hands the columns back, then reduces it into the FP32 dQ
//              accumulator through shared-memory staging and TMA reduce-adds.
//   warp  12   MMA issuer;  warp 13  TMA producer (K, V per item; Q, dO tiles and the
//              per-tile lse / delta vectors per step);  warps 14-15 set-up/teardown only.
// At d = 64 with up to 4096 keys the grid is one CTA per SM and each CTA walks several items
// (fa_bwd_main<64, true>): the next item's K and V load into a second buffer during the
// current item's last steps, and its first S^T and dP^T products run while the P/dS
// warpgroups write the current item's dK and dV.  Longer rows, and d = 128 (whose shared
// memory has no room for a second K/V buffer), take one CTA per item.
// Tensor memory (512 columns): S^T | dP^T (the dQ tile reuses these columns) | dK | dV, and
// at d = 64 a second S^T buffer in the last 128 columns (S^T of odd query steps).
#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>

#include <mutex>

#include "fa_host.h"
#include "sm103.cuh"

namespace fa {
namespace bwd {

constexpr int kBlock = 128;     // keys per CTA tile and queries per step
constexpr int kThreads = 512;   // 16 warps; warps 14-15 only take part in set-up and teardown
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;
// Per-thread register budgets after the launch (setmaxnreg): the dQ warpgroup holds a whole
// dQ row (D FP32) so it can hand the TMEM columns back in one round trip, the P/dS
// warpgroups hold a 64-column row of P and dP, the MMA/TMA warpgroup needs few.
constexpr int kRegLaunch = 128;
constexpr int kRegPdS = 144, kRegDQ = 152, kRegOther = 72;
static_assert(2 * 128 * kRegPdS + 128 * kRegDQ + 128 * kRegOther <= kThreads * kRegLaunch,
              "register split exceeds the launch allocation");
constexpr int kMaxStages = 3;   // deepest Q-tile ring (dO is single-buffered)
constexpr int kMaxKVBufs = 2;   // most K/V buffers

template <int D, bool kWalk>
struct Cfg {
  // d = 64 has room for a third Q stage and a second S^T buffer in TMEM: S_{i+2} is computed
  // into the other buffer while the P/dS warpgroups still work on step i+1
  static constexpr int kStages = (D == 64) ? 3 : 2;   // Q-tile ring depth
  static constexpr bool kDoubleS = (D == 64);
  static_assert(kStages <= kMaxStages, "Q ring deeper than the barrier arrays");
  static constexpr int kTileBytes = kBlock * D * 2;
  // kWalk: a CTA walks several work items, with two K/V buffers so the next item's K and V
  // load while it still works on the current one (K of buffer b at kKOff + b kKVBytes, V
  // after it).  Without it a CTA takes one item and the item loops fold away.
  static constexpr bool kMultiItem = kWalk;
  static constexpr int kKVBufs = kWalk ? 2 : 1;
  static_assert(kKVBufs <= kMaxKVBufs, "more K/V buffers than barriers");
  static constexpr int kKVBytes = 2 * kTileBytes;
  static constexpr int kKOff = 0;
  static constexpr int kQOff = kKOff + kKVBufs * kKVBytes;
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;
  static constexpr int kDSOff = kDOOff + kTileBytes;                // dS^T, 128 x 128 BF16
  // dQ staging: a ring of four 128B-swizzled slots of 32 FP32 columns x 64 rows (8 KB), the
  // sources of the TMA reduce-adds into the accumulator; a 32-column group of a dQ tile
  // takes two slots (rows 0-63, 64-127)
  static constexpr int kDQSlot = 64 * 128;
  static constexpr int kDQOff = kDSOff + kBlock * kBlock * 2;
  static constexpr int kLseOff = kDQOff + 4 * kDQSlot;               // lse*log2(e), per stage
  static constexpr int kDeltaOff = kLseOff + kStages * kBlock * 4;   // delta, per stage
  static constexpr int kBarOff = kDeltaOff + kStages * kBlock * 4;
  static constexpr int kSmemBytes = kBarOff + 256;
  static_assert(kSmemBytes <= 227 * 1024, "backward shared-memory layout exceeds 227 KB");
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDQ = 128, kTmemDK = 256, kTmemDV = 256 + D;
  static constexpr uint32_t kTmemS1 = kTmemDV + D;  // second S^T buffer (d = 64)
  static_assert(kTmemDV + D <= 512 && kTmemDQ + D <= kTmemDK && (!kDoubleS || kTmemS1 + 128 <= 512),
                "TMEM plan exceeds 512 columns");
  // S^T (then P^T) of query step `it`, and the barrier slot / parity of its s_full event
  __device__ static uint32_t s_col(int it) { return (kDoubleS && (it & 1)) ? kTmemS1 : kTmemS; }
  __device__ static int s_slot(int it) { return kDoubleS ? (it & 1) : 0; }
  __device__ static uint32_t s_parity(int it) { return kDoubleS ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1); }
  static constexpr uint32_t kIdescSq = idesc_bf16(128, kBlock, false, false);  // S^T, dP^T
  static constexpr uint32_t kIdescKV = idesc_bf16(128, D, false, true);        // dV (TMEM A), dK
  static constexpr uint32_t kIdescQ = idesc_bf16(128, D, true, true);          // dQ: A = dS (MN-major)
};

struct Bars {
  uint64_t kv_full[kMaxKVBufs], kv_empty[kMaxKVBufs];
  uint64_t q_full[kMaxStages], q_empty[kMaxStages], do_full, do_empty;
  uint64_t s_full[2], p_ready, dp_full, ds_ready, ds_empty, dq_full, dq_empty;
  uint64_t acc_full, acc_empty;  // an item's dK, dV complete in TMEM / read out by the epilogue
  uint64_t mma_done;
  uint64_t never;  // test builds only: a barrier nothing arrives on
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barriers exceed their 256-byte slot in shared memory");

struct Params {
  const float* lse2;    // [BH, N_pad] lse * log2(e), +inf past N
  const float* delta;   // [BH, N_pad] delta, 0 past N
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  DevStatus* status;
  int N;
  int BH;
  int N_pad;        // N rounded up to 128
  int n_tiles;      // N_pad / 128
  int causal;
  float scale;
  float scale_log2;
  int inject_stall;  // test builds only (FA_TEST_HOOKS): make the MMA warp's first wait run out
};

// --------------------------------------------------------------------------- preprocess
// Over the padded rows (bh, q < N_pad): delta = rowsum(dO o O) in FP32, lse2 = lse log2(e)
// and dQ_acc = 0 for q < N; delta = 0 and lse2 = +inf (so P = 0) for the padding.
// d/8 lanes per row, 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ delta,
                                                         float* __restrict__ lse2, float* __restrict__ delta_out,
                                                         float* __restrict__ dq_acc, long long rows_pad, int N,
                                                         int N_pad) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x % 32;
  const long long warp_global = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const long long prow = warp_global * kRowsPerWarp + lane / kLanesPerRow;
  const long long bh = prow / N_pad;
  const int q = (int)(prow - bh * N_pad);
  const bool valid = prow < rows_pad && q < N;
  const long long row = bh * N + q;
  const int c = (lane % kLanesPerRow) * 8;
  float acc = 0.f;
  if (valid) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + c);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + row * D + c);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa2 = __bfloat1622float2(pa[i]);
      const float2 fb2 = __bfloat1622float2(pb[i]);
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D + c);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (prow < rows_pad && (lane % kLanesPerRow) == 0) {
    delta[prow] = acc;
    lse2[prow] = valid ? lse[row] * 1.4426950408889634f : INFINITY;
    if (valid && delta_out) delta_out[row] = acc;
  }
}

// --------------------------------------------------------------------------- dQ convert
__global__ void __launch_bounds__(256) fa_bwd_dq_convert(const float* __restrict__ dq_acc,
                                                         __nv_bfloat16* __restrict__ dq, float scale,
                                                         long long n8, DevStatus* status) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = i < n8;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (in) {
    a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
    b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  }
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  report_nonfinite(nonfinite_bf16x2(out.x) + nonfinite_bf16x2(out.y) + nonfinite_bf16x2(out.z) +
                       nonfinite_bf16x2(out.w),
                   status, kOutDq);
  if (!in) return;
  reinterpret_cast<uint4*>(dq)[i] = out;
}

// --------------------------------------------------------------------------- main kernel
// Work item n of this CTA.  Items are the (key tile, head) pairs in key-tile order, so the
// items with the most query tiles come first when causal; they are dealt to the CTAs in rounds
// of gridDim.x, every other round in reverse CTA order, which evens out each CTA's total.
// With one CTA per item (gridDim.x = items) every CTA gets exactly one.
__device__ __forceinline__ bool work_item(const Params& p, int n, int& jt, int& bh) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long pos = (long long)n * G + ((n & 1) ? (G - 1 - c) : c);
  if (pos >= (long long)p.n_tiles * p.BH) return false;
  jt = (int)(pos / p.BH);
  bh = (int)(pos % p.BH);
  return true;
}

template <int D, bool kWalk>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const __grid_constant__ CUtensorMap tmDQ, const Params p) {
  using C = Cfg<D, kWalk>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The swizzled operand layouts need a 1024-byte aligned base; there is no slack
  // for re-alignment at d = 128, so refuse to run rather than compute garbage.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) report_bounds(p.status, kSiteSmemAlign, (long long)smem_u32(smem));
    return;
  }
  Bars& sh = *reinterpret_cast<Bars*>(smem + C::kBarOff);
  volatile uint32_t* abort_flag = &sh.abort_flag;
  const int warp = threadIdx.x / 32;
  // Per-step barriers alternate phases over the CTA's query steps counted across its items
  // (g below); per-item barriers over its items (n).

  if (threadIdx.x == 0) {
    sh.abort_flag = 0;
    for (int b = 0; b < C::kKVBufs; ++b) {
      mbar_init(&sh.kv_full[b], 1);
      mbar_init(&sh.kv_empty[b], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.q_empty[s], 1);
    }
    mbar_init(&sh.do_full, 1);
    mbar_init(&sh.do_empty, 1);
    mbar_init(&sh.s_full[0], 1);
    mbar_init(&sh.s_full[1], 1);
    mbar_init(&sh.p_ready, 2 * kBlock);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.ds_ready, 2 * kBlock);
    mbar_init(&sh.ds_empty, 1);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_empty, kBlock);
    mbar_init(&sh.acc_full, 1);
    mbar_init(&sh.acc_empty, 2 * kBlock);
    mbar_init(&sh.mma_done, 1);
    mbar_init(&sh.never, 1);
    fence_barrier_init();
    FA_BOUNDS_OK(C::kBarOff + sizeof(Bars) <= dynamic_smem_bytes(), p.status, kSiteBwdSmemSize,
                 dynamic_smem_bytes());
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp >= 12) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegOther));
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      int g = 0;                     // query steps so far, over all items
      int nq = 0, ndo = 0, nkv = 0;  // loads issued: Q tiles, dO tiles, K/V pairs
      bool ok = true;
      for (int n = 0; ok && (C::kMultiItem || n == 0); ++n) {
        int jt, bh;
        if (!work_item(p, n, jt, bh)) break;
        const int b = n % C::kKVBufs;
        // the buffer's previous item has issued its last MMA reading K or V
        if (!(ok = mbar_wait(&sh.kv_empty[b], ((n / C::kKVBufs) & 1) ^ 1, abort_flag, p.status))) break;
        mbar_arrive_expect_tx(&sh.kv_full[b], 2 * C::kTileBytes);
        uint8_t* kv = smem + C::kKOff + b * C::kKVBytes;
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(kv + c * 16384, &tmK, &sh.kv_full[b], c * 64, jt * kBlock, bh);
          tma_load_3d(kv + C::kTileBytes + c * 16384, &tmV, &sh.kv_full[b], c * 64, jt * kBlock, bh);
        }
        nkv = n + 1;
        const int i0 = p.causal ? jt : 0;  // first query tile that sees this key tile
        const int n_it = p.n_tiles - i0;
        const size_t stat_base = (size_t)bh * p.N_pad;
        for (int it = 0; it < n_it; ++it, ++g) {
          const int s = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          const int row0 = (i0 + it) * kBlock;
          if (!(ok = mbar_wait(&sh.q_empty[s], ph ^ 1, abort_flag, p.status))) break;
          if (!FA_BOUNDS_OK(row0 < p.N_pad && (long long)stat_base + row0 + kBlock <= (long long)p.BH * p.N_pad,
                            p.status, kSiteBwdQRow, row0)) {
            ok = false;
            break;
          }
          // Q tile plus the tile's 128 padded lse*log2(e) and delta values (512 B each)
          mbar_arrive_expect_tx(&sh.q_full[s], C::kTileBytes + 2 * kBlock * 4);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::kQOff + s * C::kTileBytes + c * 16384, &tmQ, &sh.q_full[s], c * 64, row0, bh);
          bulk_load(smem + C::kLseOff + s * kBlock * 4, p.lse2 + stat_base + row0, kBlock * 4, &sh.q_full[s]);
          bulk_load(smem + C::kDeltaOff + s * kBlock * 4, p.delta + stat_base + row0, kBlock * 4, &sh.q_full[s]);
          nq = g + 1;
          if (!(ok = mbar_wait(&sh.do_empty, (g & 1) ^ 1, abort_flag, p.status))) break;
          mbar_arrive_expect_tx(&sh.do_full, C::kTileBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + C::kDOOff + c * 16384, &tmDO, &sh.do_full, c * 64, row0, bh);
          ndo = g + 1;
        }
      }
      if (*abort_flag) {
        // let copies still in flight land before the CTA's shared memory goes away
        volatile uint32_t ignore_abort = 0;
        for (int n = max(0, nkv - C::kKVBufs); n < nkv; ++n)
          mbar_wait(&sh.kv_full[n % C::kKVBufs], (n / C::kKVBufs) & 1, &ignore_abort, p.status);
        for (int i = max(0, nq - C::kStages); i < nq; ++i)
          mbar_wait(&sh.q_full[i % C::kStages], (i / C::kStages) & 1, &ignore_abort, p.status);
        if (ndo > 0) mbar_wait(&sh.do_full, (ndo - 1) & 1, &ignore_abort, p.status);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t sQ = smem_u32(smem + C::kQOff), sDO = smem_u32(smem + C::kDOOff);
      const uint32_t sDS = smem_u32(smem + C::kDSOff);
      // K-major operand with D (or 128) columns: 16 KB per 64 columns, 32 B per k-step
      auto kmaj = [](uint32_t base, int kk) { return sdesc_sw128(base + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024); };
      // MN-major operand with 128 K rows: 2 KB per k-step, 16 KB between 64-column blocks
      auto mnmaj = [](uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 16384, 1024); };
      bool ok = true;
#ifdef FA_TEST_HOOKS
      // failure-detection test: wait on a barrier nothing arrives on; the bounded wait runs
      // out, raises the CTA's abort flag and records a timeout, and every warp unwinds
      if (p.inject_stall) ok = mbar_wait(&sh.never, 0, abort_flag, p.status);
#endif
      int g0 = 0;  // query steps before the current item, over all items
      for (int n = 0; ok && (C::kMultiItem || n == 0); ++n) {
        int jt, bh;
        if (!work_item(p, n, jt, bh)) break;
        const int b = n % C::kKVBufs;
        const uint32_t sK = smem_u32(smem + C::kKOff + b * C::kKVBytes), sV = sK + C::kTileBytes;
        const int n_it = p.n_tiles - (p.causal ? jt : 0);
        if (!(ok = mbar_wait(&sh.kv_full[b], (n / C::kKVBufs) & 1, abort_flag, p.status))) break;
        // the lambdas take the item's step `it`; barriers and buffers go by the CTA's step g0 + it
        auto issue_s = [&](int it) {  // S^T = K_j Q_i^T
          const int g = g0 + it;
          const int s = g % C::kStages;
          if (!(ok = mbar_wait(&sh.q_full[s], (g / C::kStages) & 1, abort_flag, p.status))) return;
          tc_fence_after();
          const uint32_t q = sQ + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::s_col(g), kmaj(sK, kk), kmaj(q, kk), C::kIdescSq, kk > 0);
          tc_commit(&sh.s_full[C::s_slot(g)]);
        };
        // dP^T = V_j dO_i^T into dP^T's columns (which held dQ of the step before: wait until drained)
        auto issue_dp = [&](int it) {
          const int g = g0 + it;
          if (!(ok = mbar_wait(&sh.do_full, g & 1, abort_flag, p.status))) return;
          if (g > 0 && !(ok = mbar_wait(&sh.dq_empty, (g - 1) & 1, abort_flag, p.status))) return;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + C::kTmemDP, kmaj(sV, kk), kmaj(sDO, kk), C::kIdescSq, kk > 0);
          tc_commit(&sh.dp_full);
        };
        // dV += P^T dO_i: P^T (BF16) sits in S^T's columns 0-31 (queries 0-63) and
        // 64-95 (queries 64-127); 8 columns per k-step of 16 queries.  An item's first dV
        // product overwrites the accumulator: the previous item's dK and dV must be read out.
        auto issue_dv = [&](int it) {
          const int g = g0 + it;
          if (!(ok = mbar_wait(&sh.do_full, g & 1, abort_flag, p.status))) return;
          if (!(ok = mbar_wait(&sh.p_ready, g & 1, abort_flag, p.status))) return;
          if (it == 0 && n > 0 && !(ok = mbar_wait(&sh.acc_empty, (n - 1) & 1, abort_flag, p.status))) return;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk)
            mma_ts(tmem + C::kTmemDV, tmem + C::s_col(g) + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8), mnmaj(sDO, kk),
                   C::kIdescKV, (it > 0 || kk > 0) ? 1u : 0u);
        };
        // Issue order (same-thread MMAs execute in order):
        //   S_0 dP_0 dV_0 S_1 | dK_0 dQ_0 dP_1 dV_1 S_2 | dK_1 dQ_1 dP_2 dV_2 S_3 | ...
        // dP_{i+1} needs only dO and the drained dQ_i columns, so it runs while the softmax
        // warpgroups compute P_{i+1}; dV_{i+1} follows once P_{i+1} is in TMEM.  With two S^T
        // buffers (d = 64) S_{i+2} goes before dV_{i+1}: its buffer's last reader, dV_i, was
        // issued a round earlier.  The next item's S_0, dP_0 (and S_1) need none of this item's
        // accumulators, so they run while its dK and dV are written out.
        tc_fence_after();
        issue_s(0);
        if (ok) issue_dp(0);
        if (C::kDoubleS && ok && n_it > 1) issue_s(1);
        if (ok) issue_dv(0);
        if (ok) tc_commit(&sh.do_empty);
        if (!C::kDoubleS && ok && n_it > 1) issue_s(1);
        for (int it = 0; ok && it < n_it; ++it) {
          const int g = g0 + it;
          const int s = g % C::kStages;
          const uint32_t q = sQ + s * C::kTileBytes;
          // dK += dS^T Q_i ;  dQ_i = dS K_j
          if (!(ok = mbar_wait(&sh.ds_ready, g & 1, abort_flag, p.status))) break;
          tc_fence_after();
          // dS^T (BF16) sits in dP^T's columns 0-31 (queries 0-63) and 64-95 (queries 64-127);
          // reading it from TMEM spares shared-memory bandwidth (dQ, issued next, overwrites
          // those columns only after this MMA has read them: same-thread MMAs run in order)
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk)
            mma_ts(tmem + C::kTmemDK, tmem + C::kTmemDP + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8), mnmaj(q, kk),
                   C::kIdescKV, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk)
            mma_ss(tmem + C::kTmemDQ, mnmaj(sDS, kk), mnmaj(sK, kk), C::kIdescQ, kk > 0);
          tc_commit(&sh.q_empty[s]);
          tc_commit(&sh.ds_empty);
          tc_commit(&sh.dq_full);
          if (it + 1 < n_it) {
            issue_dp(it + 1);
            if (!ok) break;
            if (C::kDoubleS && it + 2 < n_it) {
              issue_s(it + 2);
              if (!ok) break;
            }
            issue_dv(it + 1);
            if (!ok) break;
            tc_commit(&sh.do_empty);
            if (!C::kDoubleS && it + 2 < n_it) {
              issue_s(it + 2);
              if (!ok) break;
            }
          }
        }
        if (!ok) break;
        // the item's dK and dV are complete once its last products finish; so are its K and V reads
        tc_commit(&sh.acc_full);
        tc_commit(&sh.kv_empty[b]);
        g0 += n_it;
      }
      tc_commit(&sh.mma_done);
      {
        // MMAs still in flight must finish before TMEM is released, even after an abort
        volatile uint32_t ignore_abort = 0;
        mbar_wait(&sh.mma_done, 0, &ignore_abort, p.status);
      }
    }
  }
  } else if (warp < 8) {
    // ------------------------------------------------------------------ P^T / dS^T warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegPdS));
    // warpgroup h handles query columns [64h, 64h + 64) of every key row
    const int h = warp / 4;
    const int lane_base = (warp % 4) * 32;
    const int r = lane_base + (threadIdx.x % 32);  // key row within the tile (= TMEM lane)
    const uint32_t lane_off = (uint32_t)lane_base << 16;
    const uint32_t tS0 = tmem + lane_off + 64 * h;  // + the step's S^T buffer column
    const uint32_t tDP = tmem + C::kTmemDP + lane_off + 64 * h;
    const float c = p.scale_log2;
    uint8_t* ds_row = smem + C::kDSOff + h * 16384 + r * 128;
    const uint32_t sw = (uint32_t)(r & 7);
    bool ok = true;
    int g0 = 0;  // query steps before the current item, over all items
    for (int n = 0; ok && (C::kMultiItem || n == 0); ++n) {
    int jt, bh;
    if (!work_item(p, n, jt, bh)) break;
    const int n_it = p.n_tiles - (p.causal ? jt : 0);
    for (int it = 0; it < n_it; ++it) {
      const int g = g0 + it;
      const int s = g % C::kStages;
      const bool diag = p.causal && it == 0;  // query tile i0 == key tile jt: mask q < key
      const uint32_t tS = tS0 + C::s_col(g);
      const float4* lse4 = reinterpret_cast<const float4*>(smem + C::kLseOff + s * kBlock * 4) + 16 * h;
      const float4* dl4 = reinterpret_cast<const float4*>(smem + C::kDeltaOff + s * kBlock * 4) + 16 * h;
      if (!(ok = mbar_wait(&sh.q_full[s], (g / C::kStages) & 1, abort_flag, p.status))) break;
      if (!(ok = mbar_wait(&sh.s_full[C::s_slot(g)], C::s_parity(g), abort_flag, p.status))) break;
      tc_fence_after();
      // P^T = exp2(S^T c - lse_q log2 e); padded queries carry lse = +inf -> 0
      // this warpgroup's 64 columns of the row in one round trip
      uint32_t w[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(w));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(w + 32));
      tmem_ld_wait();
      reg_fence(w);
      float pr[64];
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 l4 = lse4[i / 4];
        float x0, x1, x2, x3;
        fma2(x0, x1, __uint_as_float(w[i + 0]), __uint_as_float(w[i + 1]), c, c, -l4.x, -l4.y);
        fma2(x2, x3, __uint_as_float(w[i + 2]), __uint_as_float(w[i + 3]), c, c, -l4.z, -l4.w);
        pr[i + 0] = ex2_approx(x0);
        pr[i + 1] = ex2_approx(x1);
        pr[i + 2] = ex2_approx(x2);
        pr[i + 3] = ex2_approx(x3);
      }
      if (diag) {
        // query column 64h + j is visible to key row r iff 64h + j >= r
#pragma unroll
        for (int j = 0; j < 64; ++j) pr[j] = (64 * h + j >= r) ? pr[j] : 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pr[2 * i], pr[2 * i + 1]);
        __syncwarp();
        tmem_st32(tS, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sh.p_ready);
      // dS^T = P^T o (dP^T - delta_q), written 32 queries at a time into the swizzled
      // dS^T tile once the previous step's dK / dQ MMAs have finished reading it
      if (!(ok = mbar_wait(&sh.dp_full, g & 1, abort_flag, p.status))) break;
      if (g > 0 && !(ok = mbar_wait(&sh.ds_empty, (g - 1) & 1, abort_flag, p.status))) break;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(tDP + c0, w);
        tmem_ld_wait();
        reg_fence(w);
        uint32_t dsk[16];  // this chunk's dS^T as BF16 pairs, also kept in TMEM for the dK MMA
        // row r of dS^T, 16-byte chunk g (8 queries) of this 64-query block, swizzled (g ^ r%8)
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int i = gg * 8;
          const float4 da = dl4[(c0 + i) / 4], db = dl4[(c0 + i) / 4 + 1];
          const float* pp = pr + c0 + i;
          float g[8];
          // g = P * (dP - delta), two lanes per instruction
          add2(g[0], g[1], __uint_as_float(w[i + 0]), __uint_as_float(w[i + 1]), -da.x, -da.y);
          add2(g[2], g[3], __uint_as_float(w[i + 2]), __uint_as_float(w[i + 3]), -da.z, -da.w);
          add2(g[4], g[5], __uint_as_float(w[i + 4]), __uint_as_float(w[i + 5]), -db.x, -db.y);
          add2(g[6], g[7], __uint_as_float(w[i + 6]), __uint_as_float(w[i + 7]), -db.z, -db.w);
          mul2(g[0], g[1], g[0], g[1], pp[0], pp[1]);
          mul2(g[2], g[3], g[2], g[3], pp[2], pp[3]);
          mul2(g[4], g[5], g[4], g[5], pp[4], pp[5]);
          mul2(g[6], g[7], g[6], g[7], pp[6], pp[7]);
          const uint4 v4 = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                                      pack_bf16x2(g[6], g[7]));
          dsk[4 * gg] = v4.x;
          dsk[4 * gg + 1] = v4.y;
          dsk[4 * gg + 2] = v4.z;
          dsk[4 * gg + 3] = v4.w;
          const uint32_t chunk = (uint32_t)(c0 / 8 + gg);
          if (FA_BOUNDS_OK(h * 16384 + r * 128 + (int)((chunk ^ sw) << 4) + 16 <= kBlock * kBlock * 2, p.status,
                           kSiteBwdDsSmem, r))
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ sw) << 4)) = v4;
        }
        // packed columns [c0/2, c0/2 + 16) of this warpgroup's dP^T region: their dP^T values
        // (columns < c0 + 32) have already been read
        __syncwarp();
        tmem_st16(tDP + c0 / 2, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&sh.ds_ready);
    }
    if (!ok) break;
    // ------------------------------------------------------------------ dK (h = 0) / dV (h = 1) epilogue
    if (!(ok = mbar_wait(&sh.acc_full, n & 1, abort_flag, p.status))) break;
    tc_fence_after();
    {
      const int key = jt * kBlock + r;
      const bool valid = key < p.N;
      const size_t orow = ((size_t)bh * p.N + (valid ? key : 0)) * D;
      const uint32_t t = tmem + (h == 0 ? C::kTmemDK : C::kTmemDV) + lane_off;
      const float mul = h == 0 ? p.scale : 1.f;
      __nv_bfloat16* out = h == 0 ? p.dk : p.dv;
      uint32_t bad = 0;  // NaN/Inf entries of this row, as stored
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t w[32];
        tmem_ld32(t + c0, w);
        tmem_ld_wait();
        reg_fence(w);
        uint4 pkd[4];
        uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float g0 = __uint_as_float(w[2 * i]) * mul, g1 = __uint_as_float(w[2 * i + 1]) * mul;
          pw[i] = pack_bf16x2(g0, g1);
          bad += nonfinite_bf16x2(pw[i]);
        }
        if (valid && FA_BOUNDS_OK(orow + c0 + 32 <= (size_t)p.BH * p.N * D, p.status, kSiteBwdKVRow, key)) {
          uint4* dst = reinterpret_cast<uint4*>(out + orow + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = pkd[i];
        }
      }
      // this row of dK / dV has been read: the next item's first dV product may overwrite it
      tc_fence_before();
      mbar_arrive(&sh.acc_empty);
      report_nonfinite(valid ? bad : 0u, p.status, h == 0 ? kOutDk : kOutDv);
    }
    g0 += n_it;
    }
  } else {
    // ------------------------------------------------------------------ dQ warpgroup
    // Each dQ tile leaves TMEM in one round trip (the whole row of D FP32 columns into
    // registers), so the columns go back to the MMA warp -- whose next dP^T product writes
    // them -- as early as possible.  The tile is then pushed into the FP32 accumulator one
    // 32-column group at a time: each group is written, one row per thread, into two
    // 128B-swizzled slots of a four-slot ring and handed to TMA reduce-adds issued by one
    // thread (rows past N are dropped by the hardware).  A group waits only for the group
    // two before it to have been read, so the TMA engine always has work while the next
    // group is written.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegDQ));
    const int lane_base = (warp % 4) * 32;
    const int r = lane_base + (threadIdx.x % 32);  // query row within the current query tile
    const bool leader = (r == 0);
    const uint32_t tDQ = tmem + C::kTmemDQ + ((uint32_t)lane_base << 16);
    const uint32_t sw = (uint32_t)(r & 7);
    int g_total = 0;  // 32-column groups pushed so far (slot pair = g_total % 2)
    int g0 = 0;       // query steps before the current item, over all items
    bool ok = true;
    for (int n = 0; ok && (C::kMultiItem || n == 0); ++n) {
    int jt, bh;
    if (!work_item(p, n, jt, bh)) break;
    const int i0 = p.causal ? jt : 0;
    const int n_it = p.n_tiles - i0;
    for (int it = 0; it < n_it; ++it) {
      if (!(ok = mbar_wait(&sh.dq_full, (g0 + it) & 1, abort_flag, p.status))) break;
      tc_fence_after();
      const int q0 = (i0 + it) * kBlock;
      uint32_t w[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32(tDQ + c0, *reinterpret_cast<uint32_t(*)[32]>(w + c0));
      tmem_ld_wait();
      reg_fence(w);
      tc_fence_before();
      mbar_arrive(&sh.dq_empty);
#pragma unroll
      for (int g = 0; g < D / 32; ++g, ++g_total) {
        const int pair = g_total & 1;  // slots 2*pair (rows 0-63) and 2*pair + 1 (rows 64-127)
        // the pair's previous group (two groups back) has been read
        if (leader) bulk_wait_read_but_one();
        named_barrier(1, kBlock);
        uint8_t* row = smem + C::kDQOff + (2 * pair + (r >> 6)) * C::kDQSlot + (r & 63) * 128;
        if (FA_BOUNDS_OK((2 * pair + (r >> 6)) * C::kDQSlot + (r & 63) * 128 + 128 <= 4 * C::kDQSlot, p.status,
                         kSiteBwdDqStage, r)) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(row + (((uint32_t)ch ^ sw) << 4)) = make_uint4(
                w[g * 32 + ch * 4], w[g * 32 + ch * 4 + 1], w[g * 32 + ch * 4 + 2], w[g * 32 + ch * 4 + 3]);
        }
        fence_proxy_async_smem();
        named_barrier(1, kBlock);
        if (leader && FA_BOUNDS_OK(g * 32 + 32 <= D && q0 < p.N_pad && bh < p.BH, p.status, kSiteBwdDqCoord, q0)) {
          tma_reduce_add_3d(&tmDQ, smem + C::kDQOff + (2 * pair) * C::kDQSlot, g * 32, q0, bh);
          tma_reduce_add_3d(&tmDQ, smem + C::kDQOff + (2 * pair + 1) * C::kDQSlot, g * 32, q0 + 64, bh);
          bulk_commit_group();
        }
      }
    }
    g0 += n_it;
    }
    // the accumulator must hold every reduction before the CTA retires
    if (leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bwd
}  // namespace fa

namespace {

// The backward's scratch, carved from one caller buffer: the FP32 dQ accumulator
// [BH, N, d], then delta and lse*log2(e) padded per head to N_pad = ceil(N/128)*128 rows,
// each region 256-byte aligned.
struct Scratch {
  float* dq_acc;
  float* delta;
  float* lse2;
};

size_t scratch_bytes(int B, int H, int N, int d) {
  const size_t bh = (size_t)B * H;
  const size_t n_pad = ((size_t)N + 127) / 128 * 128;
  return fa::round_up(bh * N * d * 4, 256) + 2 * fa::round_up(bh * n_pad * 4, 256);
}

Scratch carve_scratch(void* base, int B, int H, int N, int d) {
  const size_t bh = (size_t)B * H;
  const size_t n_pad = ((size_t)N + 127) / 128 * 128;
  char* p = static_cast<char*>(base);
  Scratch s;
  s.dq_acc = reinterpret_cast<float*>(p);
  p += fa::round_up(bh * N * d * 4, 256);
  s.delta = reinterpret_cast<float*>(p);
  p += fa::round_up(bh * n_pad * 4, 256);
  s.lse2 = reinterpret_cast<float*>(p);
  return s;
}

template <int D, bool kWalk>
int launch_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                const CUtensorMap& tdq, const fa::bwd::Params& p, cudaStream_t stream) {
  using namespace fa;
  using C = bwd::Cfg<D, kWalk>;
  auto kern = bwd::fa_bwd_main<D, kWalk>;
  // setmaxnreg.inc waits until the block's launch registers cover the new split: refuse to
  // launch a build whose launch allocation is smaller than the split needs
  constexpr int kSplit = 2 * 128 * bwd::kRegPdS + 128 * bwd::kRegDQ + 128 * bwd::kRegOther;
  static std::atomic<uint64_t> prepared{0};
  int rc = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, bwd::kThreads, kSplit,
                          "backward kernel", &prepared);
  if (rc) return rc;
  const long long items = (long long)p.n_tiles * p.BH;
  long long grid = items;
  if (kWalk) {
    const int sms = sm_count();
    if (sms > 0 && sms < grid) grid = sms;
#ifdef FA_TEST_HOOKS
    // item-walk test: any grid from 1 CTA (every item in one CTA) up to one CTA per item
    const char* grid_env = getenv("FA_TEST_BWD_GRID");
    if (grid_env && atoll(grid_env) > 0) grid = atoll(grid_env) < items ? atoll(grid_env) : items;
#endif
  }
  kern<<<(unsigned)grid, bwd::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, p);
  return check_cuda(cudaGetLastError(), "launch fa_bwd_main");
}

template <int D>
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
               void* dk, void* dv, float* delta_out, int B, int H, int N, int causal, float scale,
               const Scratch& sc, cudaStream_t stream, int stages, fa::DevStatus* status_word = nullptr) {
  using namespace fa;
  const long long rows = (long long)B * H * N;
  int rc;
  const int N_pad = (N + bwd::kBlock - 1) / bwd::kBlock * bwd::kBlock;
  if (stages & FA_BWD_PREPROCESS) {
    constexpr int rows_per_block = 8 * (32 / (D / 8));
    const long long rows_pad = (long long)B * H * N_pad;
    const long long grid = (rows_pad + rows_per_block - 1) / rows_per_block;
    bwd::fa_bwd_preprocess<D><<<(unsigned)grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, sc.delta, sc.lse2,
        delta_out, sc.dq_acc, rows_pad, N, N_pad);
    if ((rc = check_cuda(cudaGetLastError(), "launch fa_bwd_preprocess"))) return rc;
  }
  if (stages & FA_BWD_MAIN) {
  CUtensorMap tq, tk, tv, tdo;
  CUtensorMap tdq;
  if ((rc = make_tmap_bhnd(&tq, q, B * H, N, D, bwd::kBlock)) || (rc = make_tmap_bhnd(&tk, k, B * H, N, D, bwd::kBlock)) ||
      (rc = make_tmap_bhnd(&tv, v, B * H, N, D, bwd::kBlock)) || (rc = make_tmap_bhnd(&tdo, dO, B * H, N, D, bwd::kBlock)) ||
      (rc = make_tmap_f32_bhnd(&tdq, sc.dq_acc, B * H, N, D, 64)))
    return rc;
  bwd::Params p{};
  p.lse2 = sc.lse2;
  p.delta = sc.delta;
  p.dq_acc = sc.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.status = status_word ? status_word : device_status_word();
  if (!p.status) return set_error(FA_ERR_CUDA, "could not allocate the device status record");
  p.N = N;
  p.BH = B * H;
  p.N_pad = N_pad;
  p.n_tiles = N_pad / bwd::kBlock;
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
#ifdef FA_TEST_HOOKS
  const char* inject = getenv("FA_TEST_INJECT_STALL");
  p.inject_stall = (inject && inject[0] == '1') ? 1 : 0;
#endif
  // d = 64 with up to kItemWalkMaxTiles key tiles: one CTA per SM walking several items (the
  // next item's K/V load overlaps the current one; measured +7-8 % at 1024 and 2048 tokens,
  // +3 % at 4096).  Longer rows have few, long items; one CTA per item (placed by the
  // hardware as SMs free up) is 1-3 % faster there.  d = 128 has no room for a second K/V
  // buffer: one CTA per item.
  constexpr int kItemWalkMaxTiles = 32;
  if constexpr (D == 64) {
    if (p.n_tiles <= kItemWalkMaxTiles) rc = launch_main<D, true>(tq, tk, tv, tdo, tdq, p, stream);
    else rc = launch_main<D, false>(tq, tk, tv, tdo, tdq, p, stream);
  } else {
    rc = launch_main<D, false>(tq, tk, tv, tdo, tdq, p, stream);
  }
  if (rc) return rc;
  }
  if (!(stages & FA_BWD_DQ_CONVERT)) return FA_OK;
  const long long n8 = rows * D / 8;
  DevStatus* st_word = status_word ? status_word : device_status_word();
  if (!st_word) return set_error(FA_ERR_CUDA, "could not allocate the device status record");
  bwd::fa_bwd_dq_convert<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(sc.dq_acc, static_cast<__nv_bfloat16*>(dq),
                                                                           scale, n8, st_word);
  return check_cuda(cudaGetLastError(), "launch fa_bwd_dq_convert");
}

}  // namespace

extern "C" size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (fa::check_shape(B, H, N, d)) return 0;
  return scratch_bytes(B, H, N, d);
}

extern "C" int fa_bwd_staged(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dO, void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N,
                             int d, int causal, float scale, void* workspace, size_t workspace_bytes, void* stream,
                             int stages) {
  fa::NvtxRange nvtx_range("fa_bwd_staged");
  using namespace fa;
  clear_error();
  int rc;
  if (stages <= 0 || (stages & ~FA_BWD_ALL))
    return set_error(FA_ERR_INVALID_ARG, "stages must be a non-empty mask of FA_BWD_* bits (got %d)", stages);
  if ((rc = check_shape(B, H, N, d))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) || (rc = check_ptr(o, "o")) ||
      (rc = check_ptr(lse, "lse")) || (rc = check_ptr(dO, "dO")) || (rc = check_ptr(dq, "dq")) ||
      (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")))
    return rc;
  if (delta_out && (reinterpret_cast<uintptr_t>(delta_out) & 3))
    return set_error(FA_ERR_INVALID_ARG, "delta_out is not 4-byte aligned");
  if (!(scale > 0.f) || !isfinite(scale)) return set_error(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return set_error(FA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (workspace_bytes < need)
    return set_error(FA_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  const Scratch sc = carve_scratch(workspace, B, H, N, d);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_bwd<64>(q, k, v, o, lse, dO, dq, dk, dv, delta_out, B, H, N, causal ? 1 : 0, scale, sc, s,
                                  stages)
                 : launch_bwd<128>(q, k, v, o, lse, dO, dq, dk, dv, delta_out, B, H, N, causal ? 1 : 0, scale, sc, s,
                                   stages);
}

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                      void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N, int d, int causal,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  fa::NvtxRange nvtx_range("fa_bwd");
  return fa_bwd_staged(q, k, v, o, lse, dO, dq, dk, dv, delta_out, B, H, N, d, causal, scale, workspace,
                       workspace_bytes, stream, FA_BWD_ALL);
}

// ---------------------------------------------------------------------------------------------
// Backward without any device allocation.
//
// Some callers cannot call cudaMalloc: a plugin or custom operator running inside a host
// application that owns the device-memory budget and forbids allocations outside its own
// pool, or a latency-critical path where cudaMalloc/cudaFree would synchronise the device.
// fa_bwd_noalloc serves them: the backward's scratch (FP32 dQ accumulator and delta) lives in
// a fixed file-scope device array, so the call itself allocates nothing.  The array's size is
// fixed at FA_NOALLOC_SCRATCH_BYTES; every GPU that loads this library holds it until exit.
namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

// Scratch shared by every fa_bwd_noalloc call on a device, plus that entry point's own
// device status record (the library's allocated record is not used here; it is read with
// fa_bwd_noalloc_status).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) fa::DevStatus g_noalloc_status;

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
fa::DevStatus* g_noalloc_status_ptr[kNoAllocMaxDevices] = {};

// Device address of the static scratch for the current device.  In host code the array's
// name is only a host-side stand-in, so the address must come from cudaGetSymbolAddress,
// once per device, with that device current.
int noalloc_scratch(void** scratch, fa::DevStatus** status) {
  int dev = 0;
  int rc = fa::check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fa::set_error(FA_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kNoAllocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    void* s = nullptr;
    if ((rc = fa::check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)"))) return rc;
    if ((rc = fa::check_cuda(cudaGetSymbolAddress(&s, g_noalloc_status), "cudaGetSymbolAddress(status)"))) return rc;
    g_noalloc_ptr[dev] = p;
    g_noalloc_status_ptr[dev] = static_cast<fa::DevStatus*>(s);
  }
  *scratch = g_noalloc_ptr[dev];
  *status = g_noalloc_status_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, float* delta_out, int B, int H, int N,
                              int d, int causal, float scale, void* stream) {
  fa::NvtxRange nvtx_range("fa_bwd_noalloc");
  using namespace fa;
  clear_error();
  int rc;
  if ((rc = check_shape(B, H, N, d))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) || (rc = check_ptr(o, "o")) ||
      (rc = check_ptr(lse, "lse")) || (rc = check_ptr(dO, "dO")) || (rc = check_ptr(dq, "dq")) ||
      (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")))
    return rc;
  if (delta_out && (reinterpret_cast<uintptr_t>(delta_out) & 3))
    return set_error(FA_ERR_INVALID_ARG, "delta_out is not 4-byte aligned");
  if (!(scale > 0.f) || !isfinite(scale)) return set_error(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need > kNoAllocScratchBytes)
    return set_error(FA_ERR_INVALID_ARG,
                     "problem needs %zu bytes of backward scratch; fa_bwd_noalloc holds at most %zu "
                     "(use fa_bwd with a caller-allocated workspace)",
                     need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  DevStatus* status = nullptr;
  if ((rc = noalloc_scratch(&scratch, &status))) return rc;
  const Scratch sc = carve_scratch(scratch, B, H, N, d);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_bwd<64>(q, k, v, o, lse, dO, dq, dk, dv, delta_out, B, H, N, causal ? 1 : 0, scale, sc, s,
                                  FA_BWD_ALL, status)
                 : launch_bwd<128>(q, k, v, o, lse, dO, dq, dk, dv, delta_out, B, H, N, causal ? 1 : 0, scale, sc, s,
                                   FA_BWD_ALL, status);
}

extern "C" int fa_bwd_noalloc_status(void* stream, fa_device_report* out) {
  fa::NvtxRange nvtx_range("fa_bwd_noalloc_status");
  fa::clear_error();
  void* scratch = nullptr;
  fa::DevStatus* status = nullptr;
  int rc = noalloc_scratch(&scratch, &status);
  if (rc) return rc;
  return fa::read_and_clear_status(status, stream, out);
}
