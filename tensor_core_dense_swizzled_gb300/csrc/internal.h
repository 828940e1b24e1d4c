// internal.h -- host helpers shared between the C-ABI translation units
// (defined in api.cpp).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "hgemm.h"

namespace hg {

// 2-D (batch 1) tiled, 128-byte-swizzled map over a row-major fp16/bf16
// array of `rows` x `cols` with leading dimension `ld` (elements).
hgemm_status_t encode_map_3d(CUtensorMap *map, const void *base, int bf16, int64_t cols,
                             int64_t rows, int64_t ld, uint32_t box_cols, uint32_t box_rows);

// 3-D tiled, 128-byte-swizzled map over a row-major 16-bit array of `batch`
// matrices of `rows` x `cols` (leading dimension `ld`, batch stride
// `stride`, elements), zero fill outside.
hgemm_status_t encode_map_batched(CUtensorMap *map, const void *base, int bf16, int64_t cols,
                                  int64_t rows, int64_t batch, int64_t ld, int64_t stride,
                                  uint32_t box_cols, uint32_t box_rows);

// The skinny path's split-K choice (units per wave >= 90% when possible).
int pick_split(int64_t work_tiles, int num_kb, int num_sms);

// The skinny path's default number of 64-column blocks per work unit.
int pick_skinny_nb(int64_t N, int64_t batch, int num_sms);

// Records `msg` as the calling thread's hgemm_last_error_detail() and returns s.
hgemm_status_t set_error_detail(hgemm_status_t s, const char *msg);

// The status a nonzero device error word stands for (a watchdog timeout:
// HGEMM_ERR_TIMEOUT; a failed debug invariant check: HGEMM_ERR_INTERNAL),
// with the word decoded into hgemm_last_error_detail(); HGEMM_OK for 0.
hgemm_status_t status_from_error_word(int32_t word);

// HGEMM_OK when `ptr` points into device (or managed) memory that `device`
// can read with TMA; HGEMM_ERR_INVALID_ARG naming `what` otherwise (host
// memory, another device's memory, or an address CUDA does not know), so
// that a wrong pointer is refused on the host instead of faulting the GPU.
hgemm_status_t check_device_pointer(const void *ptr, int device, const char *what);

}  // namespace hg
