// Dynamic per-tensor FP8 (E4M3) scaling of a BF16 tensor.
//
// ijyty.com/news/896914 §6.1: the stabilised shift carries over to FP8 when it is paired
// with dynamic scaling factors.  The scale is the tensor's largest magnitude mapped onto
// the largest finite E4M3 value: descale = amax(|x|) / 448, x8 = E4M3(x / descale).
// Pure bandwidth work: one read of x for amax, one read of x and one write of x8.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fa_host.h"
#include "sm103.cuh"

namespace fa {
namespace quant {

constexpr int kThreads = 256;
constexpr float kE4M3Max = 448.f;

// |x| of a BF16 as the bits of the equal FP32; non-negative FP32 bits order like unsigned
// integers (NaN above Inf), so an unsigned max is the float max.
__device__ __forceinline__ uint32_t abs_bits_lo(uint32_t w) { return (w & 0x7FFFu) << 16; }
__device__ __forceinline__ uint32_t abs_bits_hi(uint32_t w) { return w & 0x7FFF0000u; }

__global__ void __launch_bounds__(kThreads) amax_kernel(const __nv_bfloat16* __restrict__ x, size_t n,
                                                         uint32_t* __restrict__ amax_bits) {
  const size_t tid = (size_t)blockIdx.x * kThreads + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * kThreads;
  uint32_t m = 0;
  const size_t n8 = n / 8;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  for (size_t i = tid; i < n8; i += stride) {
    const uint4 u = x4[i];
    m = max(m, max(max(abs_bits_lo(u.x), abs_bits_hi(u.x)), max(abs_bits_lo(u.y), abs_bits_hi(u.y))));
    m = max(m, max(max(abs_bits_lo(u.z), abs_bits_hi(u.z)), max(abs_bits_lo(u.w), abs_bits_hi(u.w))));
  }
  const uint16_t* x16 = reinterpret_cast<const uint16_t*>(x);
  for (size_t i = n8 * 8 + tid; i < n; i += stride) m = max(m, abs_bits_lo(x16[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t part[kThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kThreads / 32; ++w) b = max(b, part[w]);
    atomicMax(amax_bits, b);
  }
}

__device__ __forceinline__ float descale_of(uint32_t amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax == 0.f ? 1.f : __fdiv_rn(amax, kE4M3Max);
}

__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float ds) {
  const float a = __fdiv_rn(__uint_as_float(w0 << 16), ds), b = __fdiv_rn(__uint_as_float(w0 & 0xFFFF0000u), ds);
  const float c = __fdiv_rn(__uint_as_float(w1 << 16), ds), d = __fdiv_rn(__uint_as_float(w1 & 0xFFFF0000u), ds);
  return pack_e4m3x4(a, b, c, d);
}

// x8 = E4M3(x / descale), 16 elements per thread step (two 16-byte loads, one 16-byte store).
__global__ void __launch_bounds__(kThreads) quantize_kernel(const __nv_bfloat16* __restrict__ x, size_t n,
                                                             uint8_t* __restrict__ x8,
                                                             const uint32_t* __restrict__ amax_bits) {
  const float ds = descale_of(*amax_bits);
  const size_t tid = (size_t)blockIdx.x * kThreads + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * kThreads;
  const size_t n16 = n / 16;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  uint4* o4 = reinterpret_cast<uint4*>(x8);
  for (size_t i = tid; i < n16; i += stride) {
    const uint4 u = x4[2 * i], v = x4[2 * i + 1];
    o4[i] = make_uint4(quant4(u.x, u.y, ds), quant4(u.z, u.w, ds), quant4(v.x, v.y, ds), quant4(v.z, v.w, ds));
  }
  const uint16_t* x16 = reinterpret_cast<const uint16_t*>(x);
  for (size_t i = n16 * 16 + tid; i < n; i += stride) {
    const float y = __fdiv_rn(__uint_as_float((uint32_t)x16[i] << 16), ds);
    x8[i] = (uint8_t)(pack_e4m3x4(y, 0.f, 0.f, 0.f) & 0xFFu);
  }
}

// The amax scratch becomes the descale once every block of quantize_kernel has read it.
__global__ void finalize_kernel(float* descale) {
  const uint32_t bits = __float_as_uint(*descale);
  *descale = descale_of(bits);
}

}  // namespace quant
}  // namespace fa

extern "C" int fa_quantize_fp8(const void* x, size_t n, void* x8, float* descale, void* stream) {
  fa::NvtxRange nvtx_range("fa_quantize_fp8");
  using namespace fa;
  clear_error();
  int rc;
  if ((rc = check_ptr(x, "x")) || (rc = check_ptr(x8, "x8"))) return rc;
  if (!descale) return set_error(FA_ERR_INVALID_ARG, "descale is NULL");
  if (reinterpret_cast<uintptr_t>(descale) & 3) return set_error(FA_ERR_INVALID_ARG, "descale is not 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(descale);
  if ((rc = check_cuda(cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), s), "cudaMemsetAsync(descale)"))) return rc;
  if (n == 0) {
    quant::finalize_kernel<<<1, 1, 0, s>>>(descale);
    return check_cuda(cudaGetLastError(), "launch fa_quantize_fp8 finalize");
  }
  const int sms = sm_count();
  const size_t want = (n / 16 + quant::kThreads - 1) / quant::kThreads + 1;
  const unsigned grid = (unsigned)(want < (size_t)sms * 8 ? want : (size_t)sms * 8);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  quant::amax_kernel<<<grid, quant::kThreads, 0, s>>>(xb, n, amax_bits);
  if ((rc = check_cuda(cudaGetLastError(), "launch fa_quantize_fp8 amax"))) return rc;
  quant::quantize_kernel<<<grid, quant::kThreads, 0, s>>>(xb, n, static_cast<uint8_t*>(x8), amax_bits);
  if ((rc = check_cuda(cudaGetLastError(), "launch fa_quantize_fp8 quantize"))) return rc;
  quant::finalize_kernel<<<1, 1, 0, s>>>(descale);
  return check_cuda(cudaGetLastError(), "launch fa_quantize_fp8 finalize");
}
