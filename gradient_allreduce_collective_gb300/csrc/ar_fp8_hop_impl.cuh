// ar_fp8_hop_impl.cuh — FP8 re-quantised on every hop of the ring (sm_103a).
//
// A ring that compresses its traffic sends each partial sum in FP8 ("AllReduce
// （オールリデュース）" glossary, §NCCLにおけるAllReduce: FP8 AllReduce; "All-
// Reduce・All-Gather・All-to-All とは？" vasteelab, §data typeと圧縮: reducing
// partial results at low precision changes the numerical error). Chunk c
// starts at rank c+1; at every hop the running partial of each 128-element
// block (counted from the chunk's start) is quantised (s = amax/448, E4M3
// nearest even, saturating), dequantised, and the next rank's value is added
// in binary32; the finished chunk is quantised once more for the all-gather
// and every rank stores the same dequantised values in the output type.
//
// One warp per block: lane l holds elements l, l+32, l+64, l+96; the block
// amax of each hop is a warp-wide xor reduction; the ranks' values are loaded
// in batches of eight ranks before they are folded.
#pragma once

#include <cstdint>

#include "ar_fp8_common.cuh"

namespace gar {

// quantise-dequantise a warp's 128-element block held 4 values per lane
__device__ __forceinline__ void qdq_block(float (&p)[4]) {
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(p[k]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 448.0f);
  const float x[4] = {p[0], p[1], p[2], p[3]};
  qdq_lane<4>(x, amax, s, p);
}

template <int DT> __device__ __forceinline__ float load_elem(const void* base, uint64_t e) {
  if constexpr (Fmt<DT>::bytes == 4) return to_f32<DT>(*(static_cast<const uint32_t*>(base) + e));
  else return to_f32<DT>(*(static_cast<const uint16_t*>(base) + e));
}

template <int IDT, int ODT, int OP, int MAXN>
__global__ void __launch_bounds__(kThreads) k_fp8_hop(const __grid_constant__ Fp8HopArgs A) {
  const int N = A.nranks;
  const int lane = threadIdx.x & 31;
  const uint64_t tasks = (uint64_t)N * A.nbc;
  const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  for (uint64_t t = warp0; t < tasks; t += nwarps) {  // warp-uniform
    const int c = (int)(t / A.nbc);
    const uint64_t j = t - (uint64_t)c * A.nbc;
    const uint64_t clo = (uint64_t)c * A.L;
    const uint64_t chi = (clo + A.L < A.count) ? clo + A.L : A.count;
    const uint64_t lo = clo + j * kFp8Block;
    if (clo >= A.count || lo >= chi) continue;
    const uint64_t hi = (lo + kFp8Block < chi) ? lo + kFp8Block : chi;
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) valid[k] = lo + lane + 32 * k < hi;
    const int s0 = (c + 1 == N) ? 0 : c + 1;
    float p[4];
#pragma unroll
    for (int b0 = 0; b0 < MAXN; b0 += 8) {
      if (b0 >= N) break;
      float x[8][4];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (b0 + m < N) {
          int r = s0 + b0 + m;
          r = (r >= N) ? r - N : r;
#pragma unroll
          for (int k = 0; k < 4; ++k) x[m][k] = valid[k] ? load_elem<IDT>(A.src[r], lo + lane + 32 * k) : 0.0f;
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (b0 + m < N) {
          if (b0 + m == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) p[k] = x[m][k];
          } else {
            qdq_block(p);  // the partial goes over the wire in FP8
#pragma unroll
            for (int k = 0; k < 4; ++k) p[k] = __fadd_rn(p[k], x[m][k]);
          }
        }
      }
    }
    if constexpr (OP == OP_AVG) {
#pragma unroll
      for (int k = 0; k < 4; ++k) p[k] = __fdiv_rn(p[k], (float)N);
    }
    qdq_block(p);  // the finished chunk, as the all-gather sends it
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (!valid[k]) continue;
      const uint32_t bits = from_f32<ODT>(p[k]);
      const uint64_t e = lo + lane + 32 * k;
      for (int r = 0; r < N; ++r) {
        if constexpr (Fmt<ODT>::bytes == 4) *(static_cast<uint32_t*>(A.dst[r]) + e) = bits;
        else *(static_cast<uint16_t*>(A.dst[r]) + e) = (uint16_t)bits;
      }
    }
  }
}

template <int IDT, int ODT, int OP>
cudaError_t launch_hop_op(const Fp8HopArgs& a, cudaStream_t s) {
  const uint64_t tasks = (uint64_t)a.nranks * a.nbc;
  if (tasks == 0) return cudaSuccess;
  const unsigned grid = grid_for(tasks * 32);
  if (a.nranks <= 8) k_fp8_hop<IDT, ODT, OP, 8><<<grid, kThreads, 0, s>>>(a);
  else if (a.nranks <= 16) k_fp8_hop<IDT, ODT, OP, 16><<<grid, kThreads, 0, s>>>(a);
  else k_fp8_hop<IDT, ODT, OP, kMaxRanks><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int IDT, int ODT> cudaError_t launch_hop_io(int op, const Fp8HopArgs& a, cudaStream_t s) {
  if (op == OP_SUM) return launch_hop_op<IDT, ODT, OP_SUM>(a, s);
  if (op == OP_AVG) return launch_hop_op<IDT, ODT, OP_AVG>(a, s);
  return cudaErrorInvalidValue;
}

template <int IDT> cudaError_t launch_hop_in(int out_dtype, int op, const Fp8HopArgs& a, cudaStream_t s) {
  switch (out_dtype) {
    case DT_F32: return launch_hop_io<IDT, DT_F32>(op, a, s);
    case DT_F16: return launch_hop_io<IDT, DT_F16>(op, a, s);
    case DT_BF16: return launch_hop_io<IDT, DT_BF16>(op, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gar
