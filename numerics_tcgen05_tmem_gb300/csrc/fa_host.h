// Host-side helpers shared by the entry points: error reporting, the per-device
// status record, tensor-map encoding and argument checks.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fa.h"

namespace fa {

// An NVTX range around one entry point's host work (argument checks, tensor maps, launches),
// so a profiler's timeline shows each ABI call; without a profiler attached it costs a call
// into a no-op stub.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Record `msg` as this thread's last error and return `code`.
int set_error(int code, const char* fmt, ...);
void clear_error();

// Returns FA_ERR_CUDA (with the CUDA message recorded) if e != cudaSuccess.
int check_cuda(cudaError_t e, const char* what);

struct DevStatus;

// The current device's status record (allocated and zeroed on first use); nullptr on failure.
DevStatus* device_status_word();

// Synchronise `stream`, copy the status record at `dev_rec` (a device address) into `out`,
// clear it on the device when anything was set, and map its flags to an fa_status code
// (FA_ERR_TIMEOUT, FA_ERR_DEVICE_BOUNDS, FA_WARN_NONFINITE in that order of precedence).
// Allocates nothing.
int read_and_clear_status(void* dev_rec, void* stream, fa_device_report* out);

// Encode a 3-D BF16 tensor map over a contiguous [BH, N, d] tensor with a
// 128-byte swizzle and a (64 x box_rows x 1) box; out-of-range rows read as zero.
int make_tmap_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// The same for a 1-byte (E4M3) tensor: one swizzle atom per box row -- a (128 x box_rows x 1)
// box with a 128-byte swizzle for d = 128, a (64 x box_rows x 1) box with a 64-byte swizzle
// for d = 64.
int make_tmap_u8_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// Encode a 3-D FP32 tensor map over a contiguous [BH, N, d] tensor with a 128-byte swizzle
// and a (32 x box_rows x 1) box (for TMA reductions into an FP32 accumulator).
int make_tmap_f32_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows);

// Common argument checks for [B,H,N,d] problems.
int check_shape(int B, int H, int N, int d);
int check_ptr(const void* p, const char* name);

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int sm_count();

// Once per kernel and device: raise the kernel's dynamic shared memory limit to smem_bytes and
// check that its launch register allocation (registers per thread x threads) covers the
// setmaxnreg split of `split` registers -- setmaxnreg.inc would otherwise wait forever.  `done`
// is the kernel's own bit mask of devices already prepared (a static of the caller); later
// calls on a prepared device cost one cudaGetDevice and an atomic load.
int prepare_kernel(const void* kern, int smem_bytes, int threads, int split, const char* name,
                   std::atomic<uint64_t>* done);

}  // namespace fa
