// Host-side helpers shared by the entry points: error reporting, the per-device
// status word, tensor-map encoding and argument checks.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

// Record `msg` as this thread's last error and return `code`.
int set_error(int code, const char* fmt, ...);
void clear_error();

// Returns FA_ERR_CUDA (with the CUDA message recorded) if e != cudaSuccess.
int check_cuda(cudaError_t e, const char* what);

// The current device's status word (allocated on first use); nullptr on failure.
uint32_t* device_status_word();

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

}  // namespace fa
