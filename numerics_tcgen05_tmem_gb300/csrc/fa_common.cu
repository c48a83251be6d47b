// Host-side common code: thread-local error messages, the per-device status
// record, tensor-map encoding through the driver entry point, fa_device_status.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fa_host.h"
#include "sm103.cuh"

namespace fa {

static thread_local char g_last_error[512] = "";

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_last_error[0] = '\0'; }

int check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FA_OK;
  return set_error(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevStatus* g_status[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
}  // namespace

DevStatus* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status[dev]) {
    DevStatus* p = nullptr;
    if (cudaMalloc(&p, sizeof(DevStatus)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(DevStatus)) != cudaSuccess) return nullptr;
    g_status[dev] = p;
  }
  return g_status[dev];
}

static_assert(sizeof(DevStatus) == sizeof(fa_device_report), "device record and public report differ");

int read_and_clear_status(void* dev_rec, void* stream, fa_device_report* out) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = check_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (rc) return rc;
  DevStatus v;
  rc = check_cuda(cudaMemcpy(&v, dev_rec, sizeof(v), cudaMemcpyDeviceToHost), "read status record");
  if (rc) return rc;
  if (out) memcpy(out, &v, sizeof(v));
  if (v.flags) {
    rc = check_cuda(cudaMemset(dev_rec, 0, sizeof(DevStatus)), "clear status record");
    if (rc) return rc;
  }
  if (v.flags & kDevTimeout) return set_error(FA_ERR_TIMEOUT, "a kernel's bounded wait timed out");
  if (v.flags & kDevBounds)
    return set_error(FA_ERR_DEVICE_BOUNDS, "a device-side index check failed (site %u, index %lld)", v.bounds_site,
                     v.bounds_value);
  if (v.flags & kDevNonFinite)
    return set_error(FA_WARN_NONFINITE,
                     "outputs held NaN or Inf (entries: O %llu, LSE %llu, dQ %llu, dK %llu, dV %llu)",
                     v.nonfinite[kOutO], v.nonfinite[kOutLse], v.nonfinite[kOutDq], v.nonfinite[kOutDk],
                     v.nonfinite[kOutDv]);
  return FA_OK;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 148;
  }
  return g_sms[dev];
}

int prepare_kernel(const void* kern, int smem_bytes, int threads, int split, const char* name,
                   std::atomic<uint64_t>* done) {
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done->load(std::memory_order_acquire) & bit)) return FA_OK;
  if ((rc = check_cuda(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes),
                       "cudaFuncSetAttribute")))
    return rc;
  cudaFuncAttributes attr;
  if ((rc = check_cuda(cudaFuncGetAttributes(&attr, kern), "cudaFuncGetAttributes"))) return rc;
  if (attr.numRegs * threads < split)
    return set_error(FA_ERR_CUDA, "%s built with %d registers/thread; its register split needs %d", name,
                     attr.numRegs, (split + threads - 1) / threads);
  if (bit) done->fetch_or(bit, std::memory_order_acq_rel);
  return FA_OK;
}

static int encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base, int BH, int N,
                     int d, int box_cols, int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return set_error(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)N * d * elem_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FA_OK;
}

int make_tmap_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, BH, N, d, 64, box_rows);
}

int make_tmap_u8_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  // one swizzle atom per row: 128-byte rows (d = 128) or 64-byte rows (d = 64)
  if (d >= 128) return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, BH, N, d, 128, box_rows);
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, BH, N, d, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
}

int make_tmap_f32_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, BH, N, d, 32, box_rows);
}

int check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return set_error(FA_ERR_INVALID_ARG, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if ((long long)B * H * N >= (1ll << 31))
    return set_error(FA_ERR_INVALID_ARG, "B*H*N must be < 2^31");
  if (d != 64 && d != 128) return set_error(FA_ERR_UNSUPPORTED, "head dim d=%d not supported (64 or 128)", d);
  return FA_OK;
}

int check_ptr(const void* p, const char* name) {
  if (!p) return set_error(FA_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) & 15) return set_error(FA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return FA_OK;
}

}  // namespace fa

extern "C" int fa_device_report_read(void* stream, fa_device_report* out) {
  fa::NvtxRange nvtx_range("fa_device_report_read");
  fa::clear_error();
  if (!out) return fa::set_error(FA_ERR_INVALID_ARG, "out is NULL");
  fa::DevStatus* w = fa::device_status_word();
  if (!w) return fa::set_error(FA_ERR_CUDA, "status record unavailable");
  return fa::read_and_clear_status(w, stream, out);
}

extern "C" int fa_device_status(void* stream) {
  fa::NvtxRange nvtx_range("fa_device_status");
  fa::clear_error();
  fa::DevStatus* w = fa::device_status_word();
  if (!w) return fa::set_error(FA_ERR_CUDA, "status record unavailable");
  return fa::read_and_clear_status(w, stream, nullptr);
}

extern "C" const char* fa_last_error(void) { return fa::g_last_error; }

extern "C" const char* fa_version(void) { return "numerics_tcgen05_tmem_gb300 0.1 (sm_103a)"; }
