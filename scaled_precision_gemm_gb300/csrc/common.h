// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "spg.h"

namespace spg {

// Device address of the library's error word on the current device (the
// word every bounded in-kernel wait writes on time-out).  nullptr on failure.
unsigned int* device_error_word();

// Bound of every in-kernel wait, in nanoseconds.
uint64_t wait_timeout_ns();

// Test hook set by spg_debug_inject_stall (one-CTA GEMM kernels only).
bool debug_stall_enabled();

// Call number tagging the arrival counters of a K-split launch (never 0).
uint32_t next_split_epoch();

// Streaming multiprocessors of the current device (queried once per device).
int num_sms();

// Shared-memory bytes each CTA of a cluster K split receives (one-CTA tiles
// bn columns wide, epilogue chunks of cw columns, split_k pieces): per chunk
// it finishes (chunk i goes to the CTA of rank i mod split_k), per 32-column
// sub-block, source piece and TMEM lane quarter one 4 KB block.
__host__ __device__ constexpr int cluster_recv_bytes(int bn, int cw, int split_k) {
  return ((bn / cw) + split_k - 1) / split_k * (cw / 32) * split_k * 4 * 4096;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Map a CUDA error to a status; with SPG_DEBUG set in the environment the
// error string is printed to stderr.
spg_status cuda_status(cudaError_t e, const char* where);

// Map the last launch error to a status.
inline spg_status launch_status() { return cuda_status(cudaGetLastError(), "launch"); }

}  // namespace spg
