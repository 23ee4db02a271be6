// Helpers shared by the entry points of the library (defined in api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/attn_bwd.h"

namespace attn {

// Record a failure reason for attn_last_error() and return `st`.
attn_status_t api_fail(attn_status_t st, const char* fmt, ...);
// Clear the reason and return ATTN_OK.
attn_status_t api_ok();

// Address of the device error word of the current device (null without a device).
uint32_t* device_error_word();

// cuTensorMapEncodeTiled through the driver entry point; 128-byte swizzle,
// zero fill for out-of-range elements.  strides: rank-1 byte strides.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box);

// Timing hook of attn_set_timing_events: begin a call with `kernels` kernels
// (records event 0), record the next event after each kernel, end the call.
void timing_mark_begin(int kernels, cudaStream_t s);
void timing_mark(cudaStream_t s);
void timing_mark_end();

}  // namespace attn
