// dsa_host.h -- host-side helpers shared by the C-ABI entry points.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Records a message for dsa_last_error_message() and returns `st`.
dsa_status_t fail(dsa_status_t st, const char* fmt, ...);
// Clears the calling thread's message (successful call).
dsa_status_t ok();
// DSA_OK if the current device is an sm_103 part; caches per device.
dsa_status_t check_device();
// Checks a CUDA runtime result; on error records it and returns DSA_ERR_CUDA.
dsa_status_t cuda_check(cudaError_t e, const char* what);
// 2D bf16 tensor map over [rows, cols] (cols contiguous, row pitch = pitch_elems)
// with box {box_cols, box_rows} and 128-byte swizzle.
dsa_status_t make_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows);
// Validates the workspace (non-null, 256-aligned, >= need bytes).
dsa_status_t check_workspace(const void* ws, size_t bytes, size_t need, const char* who);
// Zeroes the device error word at the start of the workspace.
dsa_status_t clear_error_word(void* ws, cudaStream_t stream);
// Cycle limit of the kernels' bounded waits (dsa_set_wait_limit_cycles; default 2^31).
long long wait_limit_cycles();
// Sets the kernel's dynamic shared-memory limit to `bytes` once per (kernel, device),
// on the current device; thread-safe.
dsa_status_t configure_kernel_smem(const void* func, int bytes, const char* what);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kErrorWordBytes = 256;  // error word + padding keeps the rest 256-aligned

}  // namespace dsa
