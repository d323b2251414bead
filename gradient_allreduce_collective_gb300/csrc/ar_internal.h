// ar_internal.h — launch interface between the host planner (ar_api.cpp) and
// the sm_103a kernels. Every per-launch argument block is passed by value in
// kernel parameter space (read through the constant cache with
// __grid_constant__), so a call needs no device allocation and no copy.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace gar {

constexpr int kMaxRanks = 64;
constexpr int kThreads = 256;

enum Dt { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_I32 = 3 };
enum Op { OP_SUM = 0, OP_AVG = 1, OP_MIN = 2, OP_MAX = 3 };

// How a reduction kernel orders the fold and where it stores.
enum Mode {
  MODE_RS = 0,          // ring order, store chunk c only to its owner dst[c]
  MODE_FUSED_RING = 1,  // ring order, store every element to all N outputs
  MODE_FUSED_TREE = 2,  // recursive-halving order, store to all N outputs
};

// Reduction over N ranks of `count` elements each. Chunk c covers elements
// [c*L, min((c+1)*L, count)).
//   MODE_RS:     element i of chunk c goes to dst[c] + (i - c*L).
//   MODE_FUSED_*: element i goes to dst[r] + i for every r.
struct ReduceArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t count;
  uint64_t L;
  int nranks;
  int vec;  // 1: all pointers 16-byte aligned and L a multiple of the vector width
};

// All-gather copy in units of `unit` bytes. Output q, unit i (chunk c = i / Lu)
// comes from src[c] + (i - c*Lu). Destinations whose bit c is set in skip_mask
// already hold chunk c (the owner, or an in-place slot) and are not written.
struct GatherArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t units;      // units per output buffer
  uint64_t Lu;         // chunk length in units
  uint64_t skip_mask;  // bit c: skip dst[c] for chunk c
  uint64_t tail_bytes; // bytes after units*unit still to copy (byte-wise)
  uint64_t Lb;         // chunk length in bytes (for the byte tail)
  int nranks;
};

// Batched memcpy of up to kMaxCopyItems ranges, cut into kCopyTile-byte tiles;
// tile_start[k] is the first tile of item k, tile_start[nitems] the total.
constexpr int kMaxCopyItems = 256;
constexpr uint32_t kCopyTile = 16384;
struct CopyItem {
  const void* src;
  void* dst;
  uint64_t bytes;
};
struct MultiCopyArgs {
  CopyItem item[kMaxCopyItems];
  uint32_t tile_start[kMaxCopyItems + 1];
  int nitems;
};

// FP8 block quantisation of N ranks: rank r's `count` inputs -> q[r] (bytes)
// and s[r] (one float per 128-element block).
constexpr int kFp8Block = 128;
struct Fp8QuantArgs {
  const void* src[kMaxRanks];
  uint8_t* q[kMaxRanks];
  float* s[kMaxRanks];
  uint64_t count;
  uint64_t first_block;  // blocks [first_block, ceil(count/128)) of every rank
  int nranks;
};

// Dequantise + reduce + store, same modes as ReduceArgs, with q/s per rank.
struct Fp8ReduceArgs {
  const uint8_t* q[kMaxRanks];
  const float* s[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t count;
  uint64_t L;
  int nranks;
  int vec;
};

// Bucket allreduce straight from the gradient tensors: tensor t of rank r is
// src[r * nt + t] (counts[t] elements) at element offset[t] of the bucket
// layout, whose chunk length is L; results go to dst[r * nt + t]. Work is cut
// into tiles of kThreads items (16-byte vectors, or elements on the
// element-wise path); tile_start[t] is tensor t's first tile.
constexpr int kBucketPtrs = 1024;
constexpr int kBucketTensors = 128;
struct BucketArgs {
  const void* src[kBucketPtrs];
  void* dst[kBucketPtrs];
  uint64_t count[kBucketTensors];
  uint64_t offset[kBucketTensors];
  uint32_t tile_start[kBucketTensors + 1];
  uint64_t L;
  int nt;
  int nranks;
  int vec;
};

// FP8 allreduce with the quantisation fused into the reduction (no wire
// buffer). The vector kernel takes every full 128-element block except those
// listed for the element-wise kernel; the element-wise kernel takes the
// listed blocks and blocks [first_block, nblocks).
constexpr int kFusedList = 160;
struct Fp8FusedArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t count;
  uint64_t L;
  uint64_t list[kFusedList];  // element-wise kernel: listed blocks first
  uint64_t first_block;       // then blocks [first_block, nblocks)
  int nlist;
  int nranks;
};

// FP8 re-quantised on every ring hop: one warp per 128-element block counted
// from its chunk's start; nbc = blocks per full chunk.
struct Fp8HopArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t count;
  uint64_t L;
  uint64_t nbc;
  int nranks;
};

// One step of a stepwise ring or recursive-halving reduce-scatter: for each
// task t, dst[t][i] = a[t][i] (+) b[t][i] for i < len[t], finished (AVG
// divide, canonical NaN) when `finish` is set. Tasks never overlap.
struct StepArgs {
  const void* a[kMaxRanks];
  const void* b[kMaxRanks];
  void* dst[kMaxRanks];
  uint64_t len[kMaxRanks];
  uint32_t tile_start[kMaxRanks + 1];  // tiles of kThreads items per task
  int ntasks;
  int nranks;  // divisor for AVG
  int finish;
  int vec;     // all pointers 16-byte aligned: items are 16-byte vectors
};

// Number of SMs of the calling thread's current device
// (cudaDevAttrMultiProcessorCount), read once per device and cached; sizes
// the resident grids, so that they follow the part (152 SMs on a GB300, fewer
// on a partition of one).
cudaError_t sm_count(int* out);

// Launchers: enqueue on `stream`, return the launch status.
cudaError_t launch_reduce(int dtype, int op, int mode, const ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_gather(int unit_bytes, const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_multicopy(const MultiCopyArgs& a, cudaStream_t stream);
cudaError_t launch_step_combine(int dtype, int op, const StepArgs& a, cudaStream_t stream);
// bf16/fp16 with binary32 partials: a32/b32 — operand a/b is a partial word
// (else a 16-bit input); a.finish — the result is the finished 16-bit value
// (else a partial word). Items are 4 elements.
cudaError_t launch_step_combine16(int dtype, int op, bool a32, bool b32, const StepArgs& a, cudaStream_t stream);
cudaError_t launch_bucket_reduce(int dtype, int op, int mode, const BucketArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_quant(int in_dtype, bool vec, const Fp8QuantArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_reduce(int out_dtype, int op, int mode, const Fp8ReduceArgs& a, cudaStream_t stream);
cudaError_t launch_fp8_hop(int in_dtype, int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t stream);
// vec: run the vector kernel over the full blocks; then the element-wise
// kernel over the listed blocks and [first_block, nblocks) (if any).
cudaError_t launch_fp8_fused(int in_dtype, int out_dtype, int op, int mode, bool vec, const Fp8FusedArgs& a,
                             cudaStream_t stream);

// Grid for the streaming kernels: one work item per thread. Measured on
// GB300, short-lived blocks that each move one item per thread keep more
// loads in flight across the whole kernel (and leave no partial last round of
// a persistent grid) than a grid of resident blocks looping over the data:
// the fused 8 x 25 MiB allreduce runs at the speed of a plain device copy of
// the same bytes this way. The kernels keep their grid-stride loops for
// counts beyond the largest grid.
inline unsigned grid_for(uint64_t items) {
  uint64_t need = (items + kThreads - 1) / kThreads;
  if (need > 0x7FFFFFFFull) need = 0x7FFFFFFFull;
  return (unsigned)(need > 0 ? need : 1);
}

#ifdef __CUDACC__
// First statement of a kernel launched by launch_pdl: wait until the previous
// grid in the stream has completed and its writes are visible (a no-op after
// an ordinary launch), then let the next grid be placed on the SMs this
// grid's last wave frees, so that it starts as soon as this one completes.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" :::);
}
#endif

// Launch with programmatic stream serialization: the grid may be placed on
// the SMs while the previous grid in the stream finishes. The kernel must
// call pdl_begin() before it touches memory that an earlier kernel writes or
// reads; stream order and results stay as for <<<...>>>.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace gar
