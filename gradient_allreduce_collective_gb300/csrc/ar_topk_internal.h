// ar_topk_internal.h — launch interface of the Top-K sparsification kernels
// and of the sparse-to-dense scatter used by the sparse allreduce.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "ar_internal.h"

namespace gar {

// Radix-select state, kept on the device between the passes. The key of a
// value is the bit pattern of its magnitude (sign bit cleared), which orders
// like the magnitude for every non-NaN binary32 value.
//   prefix/mask: the key bits fixed so far (after the last pass: the key T of
//                the k-th largest magnitude)
//   need:        how many keys equal to the prefix still have to be kept
//   gt:          keys strictly above the prefix (all kept)
struct TopkState {
  uint32_t prefix;
  uint32_t mask;
  uint32_t need;
  uint32_t gt;
};

// Scatter of every rank's (index, value) pairs into its zeroed dense buffer;
// work is cut into tiles of kThreads pairs, tile_start[r] is rank r's first.
struct ScatterArgs {
  const uint32_t* idx[kMaxRanks];
  const float* val[kMaxRanks];
  float* dst[kMaxRanks];
  uint64_t nnz[kMaxRanks];
  uint32_t tile_start[kMaxRanks + 1];
  uint64_t count;  // pairs with an index >= count are dropped
  int nranks;
};

// Workspace bytes for launch_topk over `count` values (a multiple of 256).
size_t topk_workspace_bytes(uint64_t count);
// a = grad + residual into residual; (idx, val) = the k largest |a| in index
// order (ties: lower index first); residual = a with those entries zeroed.
cudaError_t launch_topk(const float* grad, float* residual, uint64_t count, uint64_t k, uint32_t* idx, float* val,
                        void* ws, cudaStream_t stream);
cudaError_t launch_sparse_scatter(const ScatterArgs& a, cudaStream_t stream);

}  // namespace gar
