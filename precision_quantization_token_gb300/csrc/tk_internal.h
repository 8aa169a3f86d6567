// Host-side helpers shared by the library's translation units (internal:
// not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tk_cast.h"

namespace tk_internal {

// Records the CUDA error's text for tk_last_cuda_error (per host thread)
// and returns TK_ERR_CUDA.
tk_status cuda_fail(cudaError_t err);

// The current device's SM count (cached per device), after raising the
// dynamic shared-memory limit of kernel `fn` to smem_bytes on that device
// (done once per kernel and device).
cudaError_t prepare_kernel(const void* fn, int smem_bytes, int* sms);

// Reads, and with `clear` zeroes, the fault word of the per-block and
// per-channel kernels (OR-ed into tk_get_device_fault's answer).
tk_status tile_fault(unsigned int* fault, int clear);

// Records `what` as the last error text and returns TK_ERR_CUDA (for
// driver-side failures that have no cudaError_t).
tk_status fail_message(const char* what);

const char* last_cuda_error();

// Dequantization of per-block (128 x 128) codes on the per-token
// dequantization pipeline; the caller has validated the arguments.
tk_status block_dequant(const void* codes, int64_t ld_codes, const void* scales,
                        int64_t ld_scales, int64_t M, int64_t K, int fmt, int mode, void* y,
                        int64_t ld_y, int out_dtype, void* stream);

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace tk_internal
