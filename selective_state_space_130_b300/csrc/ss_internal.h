// Internal host/device interface between the C ABI (ss_api.cu) and the
// kernels (ss_scan_fwd.cu, ss_state_update.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ss_scan.h"

namespace ssk {

constexpr int kDState = 16;

// Parameters of one scan launch (device pointers, sizes, flags).
struct ScanParams {
  const void* u;
  const void* delta_raw;
  const void* z;            // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;           // may be null
  const float* delta_bias;  // may be null
  const float* h0;          // may be null
  void* y;
  float* h_last;            // may be null
  // chunk carries (workspace), used when nchunks > 1
  uint32_t* ws_header;      // [0] ticket counter, [1] fault word; then per-tile flags
  float* ws_carry;          // per (tile, channel): P[16], S_local[16], S_incl[16]
  unsigned int* fault;      // fault word (workspace header or the library's own)
  int64_t batch, seqlen, dim;
  int64_t chunk_len;        // timesteps per chunk (multiple of the tile length)
  int nchunks;              // chunks per sequence (1 = no split along L)
  int ncblk;                // channel blocks per batch element
};

// Parameters of one decode step.
struct StepParams {
  float* h;
  const void* u;
  const void* delta_raw;
  const void* z;
  const void* B;
  const void* C;
  const float* A;
  const float* D;
  const float* delta_bias;
  void* y;
  int64_t batch, dim;
};

// Launch plan for a scan problem.
struct ScanPlan {
  int sg;             // threads per channel (1, 2 or 4); each owns 16/sg states
  int cblk;           // channels per thread block
  int nchunks;        // chunks per sequence
  int64_t chunk_len;  // timesteps per chunk
  size_t workspace;   // bytes of workspace needed
};

ScanPlan plan_scan(int64_t batch, int64_t seqlen, int64_t dim);

// Launchers; return cudaSuccess or the launch error.
cudaError_t launch_scan_fwd(const ScanParams& p, const ScanPlan& plan, ss_dtype in_dtype, ss_dtype out_dtype,
                            bool use_tma, cudaStream_t stream);
cudaError_t launch_state_update(const StepParams& p, ss_dtype in_dtype, ss_dtype out_dtype, cudaStream_t stream);

// The library's own fault word (device symbol), used when no workspace is given.
unsigned int* device_fault_word();

}  // namespace ssk
