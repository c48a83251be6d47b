// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA tile
// loads, tcgen05 MMA into tensor memory (TMEM), TMEM loads/stores and the
// shared-memory / instruction descriptors the MMA consumes.
//
// Written from the PTX ISA description of these instructions (tcgen05 family,
// cp.async.bulk.tensor, mbarrier).  Nothing here is specific to attention.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fa {

// ----------------------------------------------------------------- status record
// Device-side errors are OR-ed into the flags of a status record that the host reads back
// (its layout is fa_device_report of the public header).
enum : uint32_t {
  kDevOk = 0,
  kDevTimeout = 1u << 0,   // a bounded wait on an mbarrier ran out
  kDevBounds = 1u << 1,    // a device-side index or layout check failed
  kDevNonFinite = 1u << 2, // an output value was NaN or Inf
};

// Which output a non-finite count belongs to (index into DevStatus::nonfinite).
enum : int { kOutO = 0, kOutLse = 1, kOutDq = 2, kOutDk = 3, kOutDv = 4, kNumOuts = 5 };

struct DevStatus {
  uint32_t flags;                          // kDev* bits
  uint32_t bounds_site;                    // first failed index check: its site id (0 = none)
  long long bounds_value;                  // ... and the index it saw
  unsigned long long nonfinite[kNumOuts];  // entries of each output that held NaN or Inf
  unsigned long long reserved;
};
static_assert(sizeof(DevStatus) == 64, "status record layout");

// Count `bad` non-finite entries of output `which`: the warp sums its lanes' counts and one
// lane adds them to the record.  All 32 lanes of the warp must call it.
__device__ __forceinline__ void report_nonfinite(uint32_t bad, DevStatus* status, int which) {
  const uint32_t total = __reduce_add_sync(0xffffffffu, bad);
  if (total != 0 && (threadIdx.x % 32) == 0) {
    atomicAdd(&status->nonfinite[which], (unsigned long long)total);
    atomicOr(&status->flags, kDevNonFinite);
  }
}

// Number of NaN/Inf halves of a packed BF16 pair (exponent field all ones).
__device__ __forceinline__ uint32_t nonfinite_bf16x2(uint32_t w) {
  const uint32_t e = w & 0x7F807F80u;
  return ((e & 0xFFFFu) == 0x7F80u ? 1u : 0u) + ((e >> 16) == 0x7F80u ? 1u : 0u);
}

// Site ids of the device-side index checks (fa_device_report.bounds_site).  The alignment
// check is always compiled; the others only in builds with FA_DEBUG_BOUNDS, where the
// computed global, shared-memory, tensor-memory and TMA indices are checked before use (the
// fixed tensor-memory plans are checked at compile time).
enum : uint32_t {
  kSiteSmemAlign = 1,      // backward: dynamic shared memory not 1024-byte aligned
  kSiteFwdSmemSize = 10,   // forward: the tile layout does not fit the dynamic shared memory
  kSiteFwdQRow = 11,       // forward: a Q tile's first row is not below N
  kSiteFwdKVRow = 12,      // forward: a K/V block's first row is not below N
  kSiteFwdTmemS = 13,      // forward: an S / P~ buffer runs past the 512 TMEM columns
  kSiteFwdORow = 14,       // forward: an O row write runs past the output
  kSiteFwdLseRow = 15,     // forward: an LSE / statistics index runs past [B*H*N]
  kSiteFwdVDesc = 16,      // forward: a V operand address leaves its ring stage
  kSiteBwdSmemSize = 20,   // backward: the layout does not fit the dynamic shared memory
  kSiteBwdQRow = 21,       // backward: a Q / dO tile row or its lse/delta slice is out of range
  kSiteBwdDsSmem = 22,     // backward: a dS^T row store leaves the dS^T tile
  kSiteBwdDqStage = 23,    // backward: a dQ staging row leaves the staging ring
  kSiteBwdDqCoord = 24,    // backward: a dQ reduce-add box starts outside the accumulator
  kSiteBwdKVRow = 25,      // backward: a dK / dV row write runs past the output
};

// Record a failed index check: the flag, and the site and index of the first one seen.
__device__ __forceinline__ void report_bounds(DevStatus* status, uint32_t site, long long value) {
  if (atomicCAS(&status->bounds_site, 0u, site) == 0u) status->bounds_value = value;
  atomicOr(&status->flags, kDevBounds);
}

// FA_BOUNDS_OK(cond, status, site, value): in FA_DEBUG_BOUNDS builds, true when cond holds;
// otherwise it records the violation (never traps) and is false, so the caller skips the
// access.  In other builds it is the constant true and the check compiles away.
#ifdef FA_DEBUG_BOUNDS
#define FA_BOUNDS_OK(cond, status, site, value) \
  ((cond) ? true : (::fa::report_bounds((status), (site), (long long)(value)), false))
#else
#define FA_BOUNDS_OK(cond, status, site, value) true
#endif

// Bytes of dynamic shared memory this CTA was launched with.
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
  return n;
}

// Three-input minimum (sm_100+).
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// A wait gives up after this many nanoseconds of %globaltimer.
#ifndef FA_WAIT_TIMEOUT_NS
#define FA_WAIT_TIMEOUT_NS 2000000000ull
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n .reg .b32 r;\n"
      " elect.sync r|p, 0xffffffff;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// when the CTA-wide abort flag is raised (by this or another warp) or when the
// wait exceeds FA_WAIT_TIMEOUT_NS; in the latter case it raises the abort flag
// and records kDevTimeout in the global status record.  Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          DevStatus* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > FA_WAIT_TIMEOUT_NS) {
      *abort_flag = 1u;
      atomicOr(&status->flags, kDevTimeout);
      return false;
    }
  }
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled as
// transaction bytes on `bar`.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory box into global memory (FP32 add).  Rows past
// the tensor's extent are dropped by the hardware.  Tracked by the bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until at most one committed bulk group is still reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_but_one() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Barrier over a subset of the CTA's warps (id 1..15; `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMEM
// Allocation is warp-collective; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// D(tmem) = A(smem) * B(smem)^T (+ D when accumulate != 0); kind::f16, BF16 in, FP32 accumulate.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) = A(tmem) * B(smem)^T (+ D); A is M x K with row i in lane i, two BF16 per column.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two forms for kind::f8f6f4 (A and B both E4M3 here); K = 32 per instruction.
// A from TMEM holds four E4M3 values per 32-bit column (K element k in byte k % 4).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: D FP32, A and B E4M3 (format code 0), dense; the
// field positions are those of kind::f16 below.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: D FP32, A and B BF16, dense.
//   bits 4-5 D format (1 = F32), 7-9 A format (1 = BF16), 10-12 B format (1 = BF16),
//   bit 15 A MN-major, bit 16 B MN-major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major: rows of 128 B (64 BF16 along K), 8-row atoms SBO bytes apart; LBO unused.
// MN-major: 128 B along M/N, K rows 128 B apart inside an atom; LBO = bytes between
// 64-element M/N blocks, SBO = bytes between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// The same for a 64-byte swizzle (layout 4): rows of 64 B in 8-row atoms of 512 B, used
// when a tile row is 64 bytes (E4M3 with d = 64).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)4u << 61;
  return d;
}

// ----------------------------------------------------------------- TMEM <-> registers
// 32x32b shape: warp (w % 4) reaches lanes 32*(w%4) .. +31; thread t gets lane base+t,
// .xN gives N consecutive 32-bit columns.
#define FA_R8(o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), \
                 "=r"(r[o + 4]), "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7])
#define FA_W8(o) "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), \
                 "r"(r[o + 4]), "r"(r[o + 5]), "r"(r[o + 6]), "r"(r[o + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr));
}

// The same load with a max reduction (sm_103a): mx = the largest of the thread's 32 FP32
// values (NaN ignored, like max.f32).  Like r, mx is valid only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), "=f"(mx)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Values loaded by tcgen05.ld are only valid after tcgen05.wait::ld; routing the
// registers through an empty volatile asm after the wait keeps every use after it.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}
template <int N>
__device__ __forceinline__ void reg_fence(float (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(r[i]));
}

#undef FA_R8
#undef FA_W8

// ----------------------------------------------------------------- math helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1.0f if a == b else 0.0f.  Summed in FP32 pairs (add2) this counts equalities exactly (any
// count up to 2^24), in about 1.5 instructions per entry; an all-ones integer mask
// (set.eq.u32.f32) summed with integer adds measured about 2.5.
__device__ __forceinline__ float eq_one(float a, float b) {
  float m;
  asm("set.eq.f32.f32 %0, %1, %2;" : "=f"(m) : "f"(a), "f"(b));
  return m;
}

// Three-input maximum (sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed FP32 pair arithmetic (one instruction for two lanes of work, sm_100+):
// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1), (a0 + b0, a1 + b1), (a0 * b0, a1 * b1).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                     float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Pack two FP32 into BF16x2 with round-to-nearest-even; `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four FP32 to E4M3 (round to nearest even, saturating to +-448; NaN stays NaN), packed so
// that p0 lands in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}"
      : "=r"(r)
      : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
  return r;
}

}  // namespace fa
