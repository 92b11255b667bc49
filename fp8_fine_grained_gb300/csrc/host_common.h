// Host-side helpers shared by the library's translation units: per-device
// status word, SM count, wait limit and argument checks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8fg.h"

namespace fp8fg {

// Device address of the current device's status word (a __device__ int in
// capi.cu), or nullptr when CUDA is unavailable.
int *status_word_ptr();

// Number of SMs of the current device (cached per device), 0 on error.
int sm_count();

// Wait limit of the device-side bounded waits, in nanoseconds.
uint64_t wait_limit_ns();

// One-shot test hook consumed by the next GEMM launch on the current device.
bool take_skip_first_load();

// Schedule of the grouped GEMM with rows in expert order: the skinny-tile
// row threshold (0: off) and a skinny tile's SM time relative to a full
// tile, in percent.
int grouped_skinny_rows();
int grouped_skinny_cost_pct();

// Current device is a Blackwell sm_103 part (cached per device).
bool device_supported();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8FG_OK : FP8FG_ECUDA;
}

}  // namespace fp8fg
